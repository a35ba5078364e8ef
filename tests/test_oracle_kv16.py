"""Pins for the oracle's uncompressed (fp16) KV cache, the setting the pages
compare the 4-bit cache against ("FlexGen 完全拆解", results for input length
512: FlexGen with and without 4-bit compression).

The checks use facts outside the oracle's own arithmetic: an fp64 softmax
(scipy) over the stored rows; the 4-bit path on a cache whose rows are
exactly representable reduces to the same sums (the fp16 cache holding the
dequantised rows gives the 4-bit oracle's output bit for bit); the stores
are plain copies of the projection's rows; padding is a shift of slots."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle.model import DECODE, PREFILL, layer_step

H16 = 2.0 ** -11


def f16(a):
    return np.asarray(a, dtype=np.float16)


def _qkv(rng, B, H, d):
    return f16(rng.standard_normal((B, 3 * H * d)))


def _filled16(rng, B, H, d, cap, L):
    c = oracle.KVCache16(B, H, d, cap)
    c.k[:, :, :L] = f16(rng.standard_normal((B, H, L, d)))
    c.v[:, :, :L] = f16(rng.standard_normal((B, H, L, d)))
    return c


@pytest.mark.parametrize("B,H,d,L", [(1, 1, 64, 1), (2, 2, 64, 9), (1, 3, 128, 40)])
def test_decode_f16_against_scipy_softmax(B, H, d, L):
    rng = np.random.default_rng(L * 7 + d)
    c = _filled16(rng, B, H, d, L + 1, L - 1)
    qkv = _qkv(rng, B, H, d)
    out = oracle.decode_attn_f16(qkv, c, L - 1, append=True).astype(np.float64)
    h1 = H * d
    for b in range(B):
        for h in range(H):
            # the append stored the projection's k and v rows as they are
            assert np.array_equal(c.k[b, h, L - 1], qkv[b, h1 + h * d:h1 + (h + 1) * d])
            assert np.array_equal(c.v[b, h, L - 1], qkv[b, 2 * h1 + h * d:2 * h1 + (h + 1) * d])
            q = qkv[b, h * d:(h + 1) * d].astype(np.float64)
            k = c.k[b, h, :L].astype(np.float64)
            v = c.v[b, h, :L].astype(np.float64)
            ref = softmax(k @ q / np.sqrt(d)) @ v
            o = out[b, h * d:(h + 1) * d]
            assert np.all(np.abs(o - ref) <= np.maximum(np.abs(ref), 2.0 ** -14) * H16 + 2e-5)


def test_f16_cache_of_dequantised_rows_equals_4bit_path():
    rng = np.random.default_rng(61)
    B, H, d, L = 2, 2, 128, 33
    c4 = oracle.KVCache(B, H, d, L)
    c16 = oracle.KVCache16(B, H, d, L)
    for b in range(B):
        for h in range(H):
            kc, km = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            vc, vm = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            c4.k_codes[b, h], c4.k_meta[b, h], c4.v_codes[b, h], c4.v_meta[b, h] = kc, km, vc, vm
            c16.k[b, h] = oracle.dequant_g4(kc, km)
            c16.v[b, h] = oracle.dequant_g4(vc, vm)
    qkv = _qkv(rng, B, H, d)
    pad = np.array([0, 11], np.int32)
    a = oracle.decode_attn_g4(qkv, c4, L - 1, append=False, pad=pad)
    b = oracle.decode_attn_f16(qkv, c16, L - 1, append=False, pad=pad)
    assert np.array_equal(a, b)


def test_prefill_store_copies_rows():
    rng = np.random.default_rng(62)
    B, s, H, d = 2, 5, 3, 64
    qkv = f16(rng.standard_normal((B * s, 3 * H * d)))
    c = oracle.KVCache16(B, H, d, s + 2)
    oracle.kv_store_prefill_f16(qkv, B, s, c)
    x = qkv.reshape(B, s, 3, H, d)
    assert np.array_equal(c.k[:, :, :s], x[:, :, 1].transpose(0, 2, 1, 3))
    assert np.array_equal(c.v[:, :, :s], x[:, :, 2].transpose(0, 2, 1, 3))
    assert not c.k[:, :, s:].any() and not c.v[:, :, s:].any()


def test_padded_equals_shifted():
    rng = np.random.default_rng(63)
    B, H, d, L, p0 = 1, 2, 64, 14, 5
    c = _filled16(rng, B, H, d, L, L - 1)
    qkv = _qkv(rng, B, H, d)
    a = oracle.decode_attn_f16(qkv, c, L - 1, append=True, pad=np.array([p0], np.int32))
    c2 = oracle.KVCache16(B, H, d, L)
    c2.k[:, :, :L - p0], c2.v[:, :, :L - p0] = c.k[:, :, p0:L], c.v[:, :, p0:L]
    b = oracle.decode_attn_f16(qkv, c2, L - 1 - p0, append=False)
    assert np.array_equal(a, b)


def test_layer_step_with_f16_cache_views():
    """A decode layer over a block's fp16 cache equals the same layer over
    each batch's view of it (the per-batch order of the block schedule)."""
    rng = np.random.default_rng(64)
    h1, H, h2, B, s = 128, 2, 256, 4, 6
    w = {"w_qkv": f16(rng.standard_normal((3 * h1, h1)) * 0.05),
         "w_out": f16(rng.standard_normal((h1, h1)) * 0.05),
         "w_fc1": f16(rng.standard_normal((h2, h1)) * 0.05),
         "w_fc2": f16(rng.standard_normal((h1, h2)) * 0.05)}
    for n, m in (("b_qkv", 3 * h1), ("b_out", h1), ("b_fc1", h2), ("b_fc2", h1)):
        w[n] = f16(rng.standard_normal(m) * 0.1)
    for n in ("ln1", "ln2"):
        w[n + "_g"] = f16(1 + 0.1 * rng.standard_normal(h1))
        w[n + "_b"] = f16(0.1 * rng.standard_normal(h1))
    L = oracle.quantize_layer(w, h1, H, h2)
    x = f16(rng.standard_normal((B * s, h1)))
    x1 = f16(rng.standard_normal((B, h1)))
    ca, cb = oracle.KVCache16(B, H, h1 // H, s + 1), oracle.KVCache16(B, H, h1 // H, s + 1)
    layer_step(L, x, ca, PREFILL, B, s)
    layer_step(L, x, cb, PREFILL, B, s)
    ya = layer_step(L, x1, ca, DECODE, B, 1, pos=s)
    yb = np.concatenate([layer_step(L, x1[i:i + 2], cb.view(i, i + 2), DECODE, 2, 1, pos=s)
                         for i in (0, 2)])
    assert np.array_equal(ya, yb)
    assert np.array_equal(ca.k, cb.k) and np.array_equal(ca.v, cb.v)
    # the prompt's rows are stored as the QKV projection made them (not quantised)
    a = oracle.layernorm(x, L.ln1_g, L.ln1_b, L.eps)
    qkv = oracle.linear_g4(a, *L.qkv, bias=L.b_qkv)
    assert np.array_equal(ca.k[:, :, :s], qkv.reshape(B, s, 3, H, -1)[:, :, 1].transpose(0, 2, 1, 3))
