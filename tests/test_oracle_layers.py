"""Pins for the oracle's linear layers, LayerNorm and attention.

Each check uses facts that do not reuse the oracle's arithmetic: fp64 matmul
within the fp32-accumulation error bound, exact permutation matrices, the
LayerNorm closed form, scipy's softmax on tiny shapes, and special cases of
attention (equal keys give the mean of V; one row gives that row; causality;
independence of key order).  The dataflow follows "FlexGen 完全拆解"
(prefill K = XW_K, V = XW_V, Q = XW_Q; decode appends one K/V row and attends
over s+t rows) and the pages' rule that stored 4-bit tensors are dequantised
to FP16 before use.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle

U = 2.0 ** -24           # fp32 unit roundoff
H16 = 2.0 ** -11         # fp16 unit roundoff


def f16(a):
    return np.asarray(a, dtype=np.float16)


def half_ulp(x):
    return np.maximum(np.abs(x), 2.0 ** -14) * H16


# ------------------------------------------------------------------ linear

@pytest.mark.parametrize("M,K,N", [(1, 64, 1), (5, 192, 70), (17, 320, 33)])
def test_linear_against_fp64(M, K, N):
    rng = np.random.default_rng(M * 1000 + K)
    x = f16(rng.standard_normal((M, K)))
    w = f16(rng.standard_normal((N, K)) * 0.05)
    b = f16(rng.standard_normal(N) * 0.1)
    r = f16(rng.standard_normal((M, N)))
    for act in (0, 1):
        y = oracle.linear_f16(x, w, bias=b, residual=r, act=act).astype(np.float64)
        prod = x.astype(np.float64) @ w.astype(np.float64).T
        pre = prod + b.astype(np.float64)
        if act:
            pre = np.maximum(pre, 0)
        ref = pre + r.astype(np.float64)
        absdot = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
        bound = (K + 2) * U * (absdot + np.abs(b.astype(np.float64)) + np.abs(r.astype(np.float64))) \
            + half_ulp(ref) * (1 + 1e-6)
        assert np.all(np.abs(y - ref) <= bound)


def test_linear_order_bias_relu_residual():
    """ReLU applies to acc + bias, before the residual is added."""
    x = f16([[1.0, 0.0]])
    w = f16([[-2.0, 0.0], [3.0, 0.0]])
    b = f16([0.5, -1.0])
    r = f16([[10.0, 20.0]])
    y = oracle.linear_f16(x, w, bias=b, residual=r, act=1)
    assert y.tolist() == [[10.0, 22.0]]     # relu(-1.5)=0 -> 10 ; relu(2.0)=2 -> 22


def test_linear_g4_permutation_is_exact():
    """A permutation matrix survives 4-bit group quantisation exactly (each
    group is all zeros, or zeros and a single 1 with scale 1/15), so
    Y = X W^T picks columns of X: Y[m][n] = X[m][perm[n]]."""
    rng = np.random.default_rng(7)
    K = N = 256
    perm = rng.permutation(K)
    w = np.zeros((N, K), np.float16)
    w[np.arange(N), perm] = 1.0
    codes, meta = oracle.quantize_g4(w)
    assert np.array_equal(oracle.dequant_g4(codes, meta), w)
    x = f16(rng.standard_normal((9, K)))
    y = oracle.linear_g4(x, codes, meta)
    assert np.array_equal(y, x[:, perm])


def test_linear_g4_is_dequant_then_linear():
    rng = np.random.default_rng(8)
    x = f16(rng.standard_normal((7, 128)))
    w = f16(rng.standard_normal((40, 128)) * 0.02)
    codes, meta = oracle.quantize_g4(w)
    wh = oracle.dequant_g4(codes, meta)
    a = oracle.linear_g4(x, codes, meta)
    ref = x.astype(np.float64) @ wh.astype(np.float64).T
    bound = 130 * U * (np.abs(x.astype(np.float64)) @ np.abs(wh.astype(np.float64)).T) + half_ulp(ref)
    assert np.all(np.abs(a.astype(np.float64) - ref) <= bound)


def test_linear_f32out_against_fp64():
    rng = np.random.default_rng(9)
    x = f16(rng.standard_normal((6, 256)))
    w = f16(rng.standard_normal((50, 256)) * 0.02)
    y = oracle.linear_f16_f32out(x, w).astype(np.float64)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    bound = 258 * U * (np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T)
    assert np.all(np.abs(y - ref) <= bound)


# ------------------------------------------------------------------ LayerNorm

def test_layernorm_closed_form():
    rng = np.random.default_rng(10)
    x = f16(rng.standard_normal((13, 768)) * 3 + 1)
    g = f16(1 + rng.standard_normal(768) * 0.1)
    b = f16(rng.standard_normal(768) * 0.1)
    y = oracle.layernorm(x, g, b, 1e-5).astype(np.float64)
    xd = x.astype(np.float64)
    mu = xd.mean(-1, keepdims=True)
    var = ((xd - mu) ** 2).mean(-1, keepdims=True)
    ref = (xd - mu) / np.sqrt(var + 1e-5) * g.astype(np.float64) + b.astype(np.float64)
    assert np.all(np.abs(y - ref) <= half_ulp(ref) + 1e-4 * (1 + np.abs(ref)))


def test_layernorm_unit_moments():
    rng = np.random.default_rng(11)
    x = f16(rng.standard_normal((8, 2048)) * 5 - 2)
    y = oracle.layernorm(x, np.ones(2048), np.zeros(2048)).astype(np.float64)
    assert np.all(np.abs(y.mean(-1)) < 2e-3)
    assert np.all(np.abs(y.var(-1) - 1) < 2e-3)


def test_embed_sum():
    rng = np.random.default_rng(12)
    et = f16(rng.standard_normal((50, 64)))
    ep = f16(rng.standard_normal((10, 64)))
    ids = np.array([3, 49, 0], np.int32)
    pos = np.array([0, 9, 5], np.int32)
    y = oracle.embed(ids, pos, et, ep)
    ref = et[ids].astype(np.float32) + ep[pos].astype(np.float32)
    assert np.array_equal(y, ref.astype(np.float16))


# ------------------------------------------------------------------ attention

def _qkv(rng, B, T, H, d, scale=1.0):
    return f16(rng.standard_normal((B * T, 3 * H * d)) * scale)


def _prefill_ref(qkv, B, s, H, d):
    h1 = H * d
    q = qkv[:, :h1].astype(np.float64).reshape(B, s, H, d)
    k = qkv[:, h1:2 * h1].astype(np.float64).reshape(B, s, H, d)
    v = qkv[:, 2 * h1:].astype(np.float64).reshape(B, s, H, d)
    sc = np.einsum("bihc,bjhc->bhij", q, k) / np.sqrt(d)
    mask = np.tril(np.ones((s, s), bool))
    sc = np.where(mask, sc, -np.inf)
    p = softmax(sc, axis=-1)
    o = np.einsum("bhij,bjhc->bihc", p, v)
    return o.reshape(B * s, h1)


@pytest.mark.parametrize("B,s,H,d", [(1, 1, 1, 64), (2, 7, 2, 64), (1, 9, 1, 128)])
def test_prefill_attn_against_scipy_softmax(B, s, H, d):
    rng = np.random.default_rng(s * 10 + d)
    qkv = _qkv(rng, B, s, H, d)
    out = oracle.prefill_attn(qkv, B, s, H, d).astype(np.float64)
    ref = _prefill_ref(qkv, B, s, H, d)
    assert np.all(np.abs(out - ref) <= half_ulp(ref) + 1e-5 * (1 + np.abs(ref)))


def test_prefill_equal_keys_gives_running_mean():
    rng = np.random.default_rng(13)
    B, s, H, d = 1, 6, 1, 64
    qkv = _qkv(rng, B, s, H, d)
    qkv[:, H * d:2 * H * d] = qkv[0, H * d:2 * H * d]          # every key equal
    out = oracle.prefill_attn(qkv, B, s, H, d).astype(np.float64)
    v = qkv[:, 2 * H * d:].astype(np.float64)
    ref = np.cumsum(v, 0) / np.arange(1, s + 1)[:, None]
    assert np.all(np.abs(out - ref) <= half_ulp(ref) + 1e-6 * (1 + np.abs(ref)))


def test_prefill_is_causal():
    rng = np.random.default_rng(14)
    B, s, H, d = 1, 8, 2, 64
    qkv = _qkv(rng, B, s, H, d)
    a = oracle.prefill_attn(qkv, B, s, H, d)
    qkv2 = qkv.copy()
    qkv2[5:] = f16(rng.standard_normal(qkv2[5:].shape))
    b = oracle.prefill_attn(qkv2, B, s, H, d)
    assert np.array_equal(a[:5], b[:5])
    assert not np.array_equal(a[5:], b[5:])


def _filled_cache(rng, B, H, d, cap, L):
    c = oracle.KVCache(B, H, d, cap)
    for b in range(B):
        for h in range(H):
            kc, km = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            vc, vm = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            c.k_codes[b, h, :L], c.k_meta[b, h, :L] = kc, km
            c.v_codes[b, h, :L], c.v_meta[b, h, :L] = vc, vm
    return c


def _decode_ref(qkv, c, pos):
    """fp64 softmax over the dequantised cache rows 0..pos."""
    B, H, d = c.B, c.H, c.d
    h1 = H * d
    out = np.zeros((B, h1))
    for b in range(B):
        for h in range(H):
            q = qkv[b, h * d:(h + 1) * d].astype(np.float64)
            k = oracle.dequant_g4(c.k_codes[b, h, :pos + 1], c.k_meta[b, h, :pos + 1]).astype(np.float64)
            v = oracle.dequant_g4(c.v_codes[b, h, :pos + 1], c.v_meta[b, h, :pos + 1]).astype(np.float64)
            p = softmax(k @ q / np.sqrt(d))
            out[b, h * d:(h + 1) * d] = p @ v
    return out


@pytest.mark.parametrize("B,H,d,L", [(1, 1, 64, 1), (2, 2, 64, 8), (1, 2, 128, 5)])
def test_decode_attn_against_scipy_softmax(B, H, d, L):
    rng = np.random.default_rng(L * 100 + d)
    cap = L + 3
    c = _filled_cache(rng, B, H, d, cap, L - 1)
    qkv = _qkv(rng, B, 1, H, d)
    out = oracle.decode_attn_g4(qkv, c, L - 1, append=True).astype(np.float64)
    # append stored exactly the oracle quantisation of the new k and v rows
    h1 = H * d
    for b in range(B):
        for h in range(H):
            kc, km = oracle.quantize_g4(qkv[b:b + 1, h1 + h * d:h1 + (h + 1) * d])
            assert np.array_equal(c.k_codes[b, h, L - 1], kc[0])
            assert np.array_equal(c.k_meta[b, h, L - 1], km[0])
            vc, vm = oracle.quantize_g4(qkv[b:b + 1, 2 * h1 + h * d:2 * h1 + (h + 1) * d])
            assert np.array_equal(c.v_codes[b, h, L - 1], vc[0])
    ref = _decode_ref(qkv, c, L - 1)
    assert np.all(np.abs(out - ref) <= half_ulp(ref) + 1e-5 * (1 + np.abs(ref)))


def test_decode_single_row_returns_dequantised_v():
    rng = np.random.default_rng(15)
    B, H, d = 2, 3, 64
    c = oracle.KVCache(B, H, d, 4)
    qkv = _qkv(rng, B, 1, H, d)
    out = oracle.decode_attn_g4(qkv, c, 0, append=True)
    h1 = H * d
    for b in range(B):
        for h in range(H):
            vh = oracle.dequant_g4(c.v_codes[b, h, :1], c.v_meta[b, h, :1])
            assert np.array_equal(out[b, h * d:(h + 1) * d], vh[0])


def test_decode_equal_keys_gives_mean_of_v():
    rng = np.random.default_rng(16)
    B, H, d, L = 1, 1, 64, 12
    c = _filled_cache(rng, B, H, d, L, L)
    c.k_codes[:] = c.k_codes[:, :, :1]
    c.k_meta[:] = c.k_meta[:, :, :1]
    qkv = _qkv(rng, B, 1, H, d)
    out = oracle.decode_attn_g4(qkv, c, L - 1, append=False).astype(np.float64)
    v = oracle.dequant_g4(c.v_codes[0, 0], c.v_meta[0, 0]).astype(np.float64)
    ref = v.mean(0)
    assert np.all(np.abs(out[0] - ref) <= half_ulp(ref) + 1e-6)


def test_decode_key_order_invariance():
    rng = np.random.default_rng(17)
    B, H, d, L = 1, 2, 64, 16
    c = _filled_cache(rng, B, H, d, L, L)
    qkv = _qkv(rng, B, 1, H, d)
    a = oracle.decode_attn_g4(qkv, c, L - 1, append=False).astype(np.float64)
    perm = rng.permutation(L)
    for arr in (c.k_codes, c.v_codes, c.k_meta, c.v_meta):
        arr[:] = arr[:, :, perm]
    b = oracle.decode_attn_g4(qkv, c, L - 1, append=False).astype(np.float64)
    assert np.all(np.abs(a - b) <= 2 * half_ulp(a) + 1e-6)


def test_prefill_store_matches_row_quantisation():
    rng = np.random.default_rng(18)
    B, s, H, d = 2, 5, 2, 128
    qkv = _qkv(rng, B, s, H, d)
    c = oracle.KVCache(B, H, d, s + 2)
    oracle.kv_store_prefill(qkv, B, s, c)
    h1 = H * d
    for b in range(B):
        for t in range(s):
            for h in range(H):
                row = qkv[b * s + t]
                kc, km = oracle.quantize_g4(row[None, h1 + h * d:h1 + (h + 1) * d])
                vc, vm = oracle.quantize_g4(row[None, 2 * h1 + h * d:2 * h1 + (h + 1) * d])
                assert np.array_equal(c.k_codes[b, h, t], kc[0])
                assert np.array_equal(c.v_codes[b, h, t], vc[0])
                assert np.array_equal(c.k_meta[b, h, t], km[0])
                assert np.array_equal(c.v_meta[b, h, t], vm[0])


# ------------------------------------------------------------------ left padding

def _prefill_ref_padded(qkv, B, s, H, d, pad):
    """fp64 softmax with the causal mask and keys before pad[b] masked; rows
    in padding slots are zero."""
    h1 = H * d
    q = qkv[:, :h1].astype(np.float64).reshape(B, s, H, d)
    k = qkv[:, h1:2 * h1].astype(np.float64).reshape(B, s, H, d)
    v = qkv[:, 2 * h1:].astype(np.float64).reshape(B, s, H, d)
    o = np.zeros((B, s, H, d))
    for b in range(B):
        p0 = pad[b]
        sc = np.einsum("ihc,jhc->hij", q[b, p0:], k[b, p0:]) / np.sqrt(d)
        n = s - p0
        sc = np.where(np.tril(np.ones((n, n), bool)), sc, -np.inf)
        o[b, p0:] = np.einsum("hij,jhc->ihc", softmax(sc, axis=-1), v[b, p0:])
    return o.reshape(B * s, h1)


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_padded_against_scipy_softmax(d):
    rng = np.random.default_rng(31 + d)
    B, s, H = 3, 9, 2
    pad = np.array([0, 4, 8], np.int32)
    qkv = _qkv(rng, B, s, H, d)
    out = oracle.prefill_attn(qkv, B, s, H, d, pad=pad).astype(np.float64)
    ref = _prefill_ref_padded(qkv, B, s, H, d, pad)
    assert np.all(np.abs(out - ref) <= half_ulp(ref) + 1e-5 * (1 + np.abs(ref)))
    rows = out.reshape(B, s, -1)
    assert not np.any(rows[1, :4]) and not np.any(rows[2, :8])


def test_prefill_padded_equals_unpadded():
    """Padding never reaches a real token: the rows of a padded prompt equal,
    bit for bit, the same prompt run alone at its own length, whatever the
    padding slots hold."""
    rng = np.random.default_rng(33)
    B, s, H, d = 2, 11, 2, 64
    pad = np.array([5, 0], np.int32)
    qkv = _qkv(rng, B, s, H, d)
    qkv[:5] = f16(1e3 * rng.standard_normal((5, qkv.shape[1])))   # junk in padding slots
    out = oracle.prefill_attn(qkv, B, s, H, d, pad=pad)
    alone = oracle.prefill_attn(qkv[5:s], 1, s - 5, H, d)
    assert np.array_equal(out[5:s], alone)
    assert np.array_equal(out[s:], oracle.prefill_attn(qkv[s:], 1, s, H, d))


def test_decode_padded_against_scipy_softmax():
    rng = np.random.default_rng(34)
    B, H, d, L = 3, 2, 128, 10
    pad = np.array([0, 3, 9], np.int32)
    c = _filled_cache(rng, B, H, d, L + 1, L - 1)
    qkv = _qkv(rng, B, 1, H, d)
    out = oracle.decode_attn_g4(qkv, c, L - 1, append=True, pad=pad).astype(np.float64)
    for b in range(B):
        sub = oracle.KVCache(1, H, d, L)
        p0 = pad[b]
        n = L - p0
        sub.k_codes[0, :, :n], sub.k_meta[0, :, :n] = c.k_codes[b, :, p0:L], c.k_meta[b, :, p0:L]
        sub.v_codes[0, :, :n], sub.v_meta[0, :, :n] = c.v_codes[b, :, p0:L], c.v_meta[b, :, p0:L]
        ref = _decode_ref(qkv[b:b + 1], sub, n - 1)
        assert np.all(np.abs(out[b] - ref[0]) <= half_ulp(ref[0]) + 1e-5 * (1 + np.abs(ref[0])))


def test_decode_padded_equals_unpadded():
    """Attending slots pad..pos equals, bit for bit, attending the same rows
    moved to slots 0..pos-pad."""
    rng = np.random.default_rng(35)
    B, H, d, L, p0 = 1, 2, 64, 13, 6
    c = _filled_cache(rng, B, H, d, L, L - 1)
    qkv = _qkv(rng, B, 1, H, d)
    a = oracle.decode_attn_g4(qkv, c, L - 1, append=True, pad=np.array([p0], np.int32))
    c2 = oracle.KVCache(B, H, d, L)
    for src, dst in ((c.k_codes, c2.k_codes), (c.k_meta, c2.k_meta),
                     (c.v_codes, c2.v_codes), (c.v_meta, c2.v_meta)):
        dst[:, :, :L - p0] = src[:, :, p0:L]
    b = oracle.decode_attn_g4(qkv, c2, L - 1 - p0, append=False)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ greedy choice

def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(36)
    x = rng.standard_normal((7, 1001)).astype(np.float32)
    assert np.array_equal(oracle.argmax(x), np.argmax(x, axis=1))
    # rounded to few values: many ties, the lowest index wins
    y = np.round(rng.standard_normal((9, 333)), 0).astype(np.float32)
    assert np.array_equal(oracle.argmax(y), np.argmax(y, axis=1))


def test_argmax_ties_pick_lowest_index():
    x = np.zeros((3, 10), np.float32)
    x[0, [2, 7]] = 5.0
    x[1, :] = -1.0
    x[2, [9]] = 1.0
    x[2, [4]] = 1.0
    assert list(oracle.argmax(x)) == [2, 0, 4]
