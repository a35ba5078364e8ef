"""Left-padded prompts and greedy generation on the GPU, through the C ABI,
against the oracle.

Padding (prompts of different lengths in one block, left-padded to the
common length): decode attention over slots pad[b]..pos, prefill attention
over the real part of each sequence with zero rows in padding slots,
positions counted from the first real slot.  Greedy: fg_argmax picks the
lowest index among equal maxima; the generated tokens feed the next step on
the device.  Several greedy continuations are correct when logits nearly
tie, so the model-level test feeds the GPU's own tokens to the oracle
(teacher-forced) and checks that every GPU choice is a maximum of the
oracle's logits within the logits tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, Model, quantize_layer
from oracle.model import OracleModel, generate, positions_of
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, rel_l2, to_np

pytestmark = pytest.mark.gpu


def _fill_cache(B, H, d, cap, L, seed):
    """Cache slots 0..L-1 from N(0,1) fp16 rows, quantised by the oracle
    (the same bytes go to both sides)."""
    g = synth.generator(seed)
    rows = synth.normal_f16((2, B * H * L, d), 1.0, g).numpy()
    oc = oracle.KVCache(B, H, d, cap)
    kc, km = oracle.quantize_g4(rows[0])
    vc, vm = oracle.quantize_g4(rows[1])
    oc.k_codes[:, :, :L] = kc.reshape(B, H, L, -1)
    oc.k_meta[:, :, :L] = km.reshape(B, H, L, -1, 2)
    oc.v_codes[:, :, :L] = vc.reshape(B, H, L, -1)
    oc.v_meta[:, :, :L] = vm.reshape(B, H, L, -1, 2)
    gc = fg.KV4(*(torch.from_numpy(a.copy()).to(DEV) for a in
                  (oc.k_codes, oc.v_codes, oc.k_meta, oc.v_meta)), B, H, d, cap)
    return oc, gc


def _vmax(oc, L):
    m = oc.v_meta[:, :, :L, :, 0]
    s = oc.v_meta[:, :, :L, :, 1]
    return float(np.max(np.abs(m) + 15 * np.abs(s)))


def _ulp16(y):
    return np.maximum(np.abs(y), 2.0 ** -14) * 2.0 ** -10


# ------------------------------------------------------------------ decode attention

@pytest.mark.parametrize("d,L", [(64, 40), (128, 65), (128, 513), (128, 2048)])
def test_decode_attn_padded_matches_oracle(d, L):
    """pad in {0, 1, a chunk boundary, a ragged middle, L-1 (only the new
    token is real)}; the fused append is unaffected by the padding."""
    B, H = 5, 2
    oc, gc = _fill_cache(B, H, d, L + 1, L - 1, 50 + L + d)
    pad = np.array([0, 1, min(128, L - 1), (L * 5) // 7, L - 1], np.int32)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(L))
    out = fg.fg_decode_attn_g4(qkv.to(DEV), gc, L - 1, fuse_append=True,
                               pad=torch.from_numpy(pad).to(DEV))
    fg.fg_check()
    ref = oracle.decode_attn_g4(qkv.numpy(), oc, L - 1, append=True, pad=pad).astype(np.float64)
    for a, b in ((gc.k_codes, oc.k_codes), (gc.v_codes, oc.v_codes),
                 (gc.k_meta, oc.k_meta), (gc.v_meta, oc.v_meta)):
        assert np.array_equal(to_np(a), b)
    got = to_np(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 4e-3 * _vmax(oc, L) + _ulp16(ref))
    assert rel_l2(got, ref) < 2e-3


@pytest.mark.parametrize("d", [64, 128])
def test_decode_attn_padded_equals_shifted_cache(d):
    """Attending slots p0..pos equals, bit for bit, attending the same rows
    moved to slots 0..pos-p0 (the kernels' key chunks start at p0)."""
    B, H, L = 3, 2, 300
    pad = np.array([0, 77, 130], np.int32)
    _, gc = _fill_cache(B, H, d, L, L, 60 + d)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(61)).to(DEV)
    a = fg.fg_decode_attn_g4(qkv, gc, L - 1, fuse_append=False, pad=torch.from_numpy(pad).to(DEV))
    for b in range(B):
        p0 = int(pad[b])
        sub = fg.KV4.empty(1, H, d, L, DEV)
        for name in ("k_codes", "v_codes", "k_meta", "v_meta"):
            getattr(sub, name)[0, :, :L - p0] = getattr(gc, name)[b, :, p0:]
        one = fg.fg_decode_attn_g4(qkv[b:b + 1].contiguous(), sub, L - 1 - p0, fuse_append=False)
        torch.cuda.synchronize()
        assert torch.equal(a[b:b + 1], one), b
    fg.fg_check()


# ------------------------------------------------------------------ prefill attention

@pytest.mark.parametrize("d", [64, 128])
def test_prefill_attn_padded_matches_oracle(d):
    """s = 150 (three query blocks, a ragged last one) with pad in {0, 1, 63,
    64, 100, 149}: real rows against the oracle, padding rows exactly zero,
    the stored K/V of every slot bit-exact."""
    B, s, H = 6, 150, 2
    pad = np.array([0, 1, 63, 64, 100, 149], np.int32)
    h1 = H * d
    qkv = synth.normal_f16((B * s, 3 * h1), 1.0, synth.generator(70 + d))
    gc = fg.KV4.empty(B, H, d, s + 1, DEV)
    out = fg.fg_prefill_attn(qkv.to(DEV), B, s, H, d, cache=gc, pad=torch.from_numpy(pad).to(DEV))
    fg.fg_check()
    ref = oracle.prefill_attn(qkv.numpy(), B, s, H, d, pad=pad).astype(np.float64)
    oc = oracle.KVCache(B, H, d, s + 1)
    oracle.kv_store_prefill(qkv.numpy(), B, s, oc)
    for a, b in ((gc.k_codes, oc.k_codes), (gc.v_codes, oc.v_codes),
                 (gc.k_meta, oc.k_meta), (gc.v_meta, oc.v_meta)):
        assert np.array_equal(to_np(a), b)
    got = to_np(out).astype(np.float64).reshape(B, s, h1)
    ref = ref.reshape(B, s, h1)
    vmax = float(np.abs(qkv.numpy()[:, 2 * h1:]).max())
    for b in range(B):
        assert not np.any(got[b, :pad[b]])
    assert np.all(np.abs(got - ref) <= 4e-3 * vmax + _ulp16(ref))
    assert rel_l2(got, ref) < 2e-3


def test_prefill_attn_padded_equals_unpadded():
    """The real rows of a padded sequence equal, bit for bit, the same rows
    run as an unpadded sequence of their own length."""
    B, s, H, d = 3, 200, 2, 128
    pad = np.array([0, 37, 136], np.int32)
    h1 = H * d
    qkv = synth.normal_f16((B * s, 3 * h1), 1.0, synth.generator(80)).to(DEV)
    out = fg.fg_prefill_attn(qkv, B, s, H, d, pad=torch.from_numpy(pad).to(DEV))
    for b in range(B):
        p0 = int(pad[b])
        one = fg.fg_prefill_attn(qkv[b * s + p0:(b + 1) * s].contiguous(), 1, s - p0, H, d)
        torch.cuda.synchronize()
        assert torch.equal(out[b * s + p0:(b + 1) * s], one), b
    fg.fg_check()


# ------------------------------------------------------------------ embedding and argmax

def test_embed_padded_positions_match_oracle():
    V, P, h1, B, s = 500, 40, 256, 4, 30
    g = synth.generator(90)
    et, ep = synth.embeddings(V, P, h1, g)
    ids = synth.token_ids((B, s), V, g)
    pad = np.array([0, 3, 29, 12], np.int32)
    y = fg.fg_embed(ids.reshape(-1).to(DEV), s, 0, et.to(DEV), ep.to(DEV),
                    pad=torch.from_numpy(pad).to(DEV))
    pos = np.concatenate([positions_of(np.arange(s), p) for p in pad])
    ref = oracle.embed(ids.numpy().reshape(-1), pos, et.numpy(), ep.numpy())
    assert np.array_equal(to_np(y), ref)
    # a decode step: one token per sequence at slot s + 2
    yd = fg.fg_embed(ids[:, 0].contiguous().to(DEV), 1, s + 2, et.to(DEV), ep.to(DEV),
                     pad=torch.from_numpy(pad).to(DEV))
    refd = oracle.embed(ids.numpy()[:, 0], (s + 2 - pad).astype(np.int32), et.numpy(), ep.numpy())
    assert np.array_equal(to_np(yd), refd)
    fg.fg_check()


@pytest.mark.parametrize("B,V", [(144, 50272), (3, 1000), (2, 1), (5, 2049)])
def test_argmax_matches_oracle(B, V):
    """Bit-exact index per row, with ties planted: a duplicate of the
    maximum after it and before it (the lowest index must win)."""
    g = synth.generator(B + V)
    x = torch.randn((B, V), generator=g, dtype=torch.float32)
    if V > 10:
        top = x.argmax(1)
        for b in range(B):
            j = int(top[b])
            if b % 3 == 0:
                x[b, (j + V // 2) % V] = x[b, j]          # a tie elsewhere
            elif b % 3 == 1:
                x[b, :] = torch.round(x[b, :])            # many ties
    got = fg.fg_argmax(x.to(DEV))
    fg.fg_check()
    assert np.array_equal(to_np(got), oracle.argmax(x.numpy()))


# ------------------------------------------------------------------ model level

def _small_model(h1, H, h2, V, P, n_layers, seed):
    g = synth.generator(seed)
    ws = []
    for _ in range(n_layers):
        w = synth.layer_weights(h1, h2, g)
        w.update(synth.random_affine_params(h1, h2, g))
        ws.append(w)
    et, ep = synth.embeddings(V, P, h1, g)
    lnf_g = (1 + synth.normal_f16((h1,), 0.1, g).float()).half()
    lnf_b = synth.normal_f16((h1,), 0.1, g)
    return ws, et, ep, lnf_g, lnf_b, g


def _gpu_model(ws, et, ep, lnf_g, lnf_b, h1, H, h2, gbs, k, cap):
    layers = [quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2) for w in ws]
    return Model(LayerStack(layers, gbs, k, cap, DEV), et.to(DEV), ep.to(DEV), lnf_g.to(DEV),
                 lnf_b.to(DEV))


def test_padded_prompts_bitwise_equal_alone():
    """2 layers (h1 512, 4 heads of 128), block gbs 2 x k 2 of prompts padded
    to 300 (real lengths 300, 280, 260, 293: every launch of the block and of
    a prompt alone stays in the same GEMM summation regime), 3 teacher-forced
    decode steps: each sequence's logits in the block, under the block and
    zig-zag orders, equal bit for bit those of the prompt run alone."""
    h1, H, h2, V, gbs, k, s, D = 512, 4, 1024, 800, 2, 2, 300, 3
    ws, et, ep, lnf_g, lnf_b, g = _small_model(h1, H, h2, V, s + D + 1, 2, 100)
    pad = torch.tensor([0, 20, 40, 7], dtype=torch.int32)
    prompt = synth.token_ids((gbs * k, s), V, g)
    dec = synth.token_ids((D, gbs * k), V, g)
    outs = {}
    for order in ("block", "zigzag"):
        m = _gpu_model(ws, et, ep, lnf_g, lnf_b, h1, H, h2, gbs, k, s + D + 1)
        outs[order] = [t.clone() for t in m.generate(prompt.to(DEV), dec.to(DEV), order=order,
                                                      pad=pad.to(DEV))]
        del m
    fg.fg_check()
    for a, b in zip(outs["block"], outs["zigzag"]):
        assert torch.equal(a, b)
    for b in range(gbs * k):
        p0 = int(pad[b])
        m1 = _gpu_model(ws, et, ep, lnf_g, lnf_b, h1, H, h2, 1, 1, s + D + 1)
        one = m1.generate(prompt[b:b + 1, p0:].contiguous().to(DEV),
                          dec[:, b:b + 1].contiguous().to(DEV), order="block")
        fg.fg_check()
        for t, (a, o) in enumerate(zip(outs["block"], one)):
            assert torch.equal(a[b:b + 1], o), (b, t)
        del m1


@pytest.mark.parametrize("d", [64, 128])
def test_greedy_generation_padded_matches_oracle(d):
    """2 layers (h1 512, heads of d), vocab 1000, gbs 3 x k 2, prompts padded
    to 40 with a seeded length mix, 6 greedy tokens under the zig-zag order:
    every GPU token is fg_argmax of the GPU's logits (bit-exact), the oracle
    teacher-forced with the GPU's tokens gives logits within max-abs
    1e-2 * max|ref| of the GPU's, and every GPU choice is a maximum of the
    oracle's logits within twice that tolerance."""
    h1, h2, V, gbs, k, s, n = 512, 1024, 1000, 3, 2, 40, 6
    H = h1 // d
    ws, et, ep, lnf_g, lnf_b, g = _small_model(h1, H, h2, V, s + n + 1, 2, 110 + d)
    pad = synth.pad_counts(gbs * k, s, g, min_len=4)
    pad[0] = 0
    prompt = synth.token_ids((gbs * k, s), V, g)
    m = _gpu_model(ws, et, ep, lnf_g, lnf_b, h1, H, h2, gbs, k, s + n + 1)
    toks, logits = m.generate_greedy(prompt.to(DEV), n, order="zigzag", pad=pad.to(DEV),
                                     keep_logits=True)
    fg.fg_check()
    toks = to_np(toks).T                      # [bls][n]
    got = [to_np(t) for t in logits]
    for t in range(n):
        assert np.array_equal(toks[:, t], oracle.argmax(got[t]))
    om = OracleModel([oracle_layer({nm: x.numpy() for nm, x in w.items()}, h1, H, h2) for w in ws],
                     et.numpy(), ep.numpy(), lnf_g.numpy(), lnf_b.numpy())
    ref = generate(om, prompt.numpy(), toks[:, :n - 1], gbs, k, order="zigzag", pad=pad.numpy())
    for t in range(n):
        tol = 1e-2 * np.max(np.abs(ref[t]))
        assert np.max(np.abs(got[t] - ref[t])) <= tol, t
        chosen = ref[t][np.arange(gbs * k), toks[:, t]]
        assert np.all(chosen >= ref[t].max(1) - 2 * tol), t
