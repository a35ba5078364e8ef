"""Parity at the workloads' full sizes, in the launch configurations the
benchmark times, on outputs the oracle can compute one by one (sampled
sequences, rows or weight rows), plus properties that hold at any size.

Inputs are the seeded synthetic tensors; the oracle quantises its own copy of
every fp16 input (bit-identical to the GPU's by the quantiser tests) and
never reads a CUDA-path output.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, quantize_layer
from oracle.model import DECODE, layer_step
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, gemm_bound, rel_l2, to_np, ulp16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _kv_rows(B, H, L, d, g, dev):
    """N(0,1) fp16 K and V rows for slots 0..L-1 of every (sequence, head)."""
    return (synth.normal_f16((B, H, L, d), 1.0, g, dev),
            synth.normal_f16((B, H, L, d), 1.0, g, dev))


def _gpu_cache(k, v, cap):
    B, H, L, d = k.shape
    c = fg.KV4.empty(B, H, d, cap, DEV)
    kq = fg.fg_quantize_g4(k.reshape(-1, d))
    vq = fg.fg_quantize_g4(v.reshape(-1, d))
    c.k_codes[:, :, :L] = kq.codes.view(B, H, L, d // 2)
    c.k_meta[:, :, :L] = kq.meta.view(B, H, L, d // 64, 2)
    c.v_codes[:, :, :L] = vq.codes.view(B, H, L, d // 2)
    c.v_meta[:, :, :L] = vq.meta.view(B, H, L, d // 64, 2)
    return c


def _oracle_cache(k, v, seqs, cap):
    """Oracle cache of the sampled sequences, quantised by the oracle from the
    same fp16 rows."""
    k = to_np(k[seqs])
    v = to_np(v[seqs])
    B, H, L, d = k.shape
    c = oracle.KVCache(B, H, d, cap)
    kc, km = oracle.quantize_g4(k.reshape(-1, d))
    vc, vm = oracle.quantize_g4(v.reshape(-1, d))
    c.k_codes[:, :, :L] = kc.reshape(B, H, L, -1)
    c.k_meta[:, :, :L] = km.reshape(B, H, L, -1, 2)
    c.v_codes[:, :, :L] = vc.reshape(B, H, L, -1)
    c.v_meta[:, :, :L] = vm.reshape(B, H, L, -1, 2)
    return c


def test_opt30b_decode_layer_bls144_sampled():
    """OPT-30B-shaped decoder layer, decode step at context 513 for the whole
    block (gbs 48 x k 3 = 144 sequences, one weight-stationary launch per
    projection, as benchmarked); 2 sampled sequences through the oracle."""
    wl = synth.OPT30B
    g = synth.generator(30, DEV)
    w = synth.layer_weights(wl.h1, wl.h2, g, DEV)
    w.update(synth.random_affine_params(wl.h1, wl.h2, g, DEV))
    L = wl.s
    k, v = _kv_rows(wl.bls, wl.H, L, wl.d, g, DEV)
    stack = LayerStack([quantize_layer(w, wl.h1, wl.H, wl.h2)], wl.gbs, wl.k, L + 1, DEV)
    stack.caches[0] = _gpu_cache(k, v, L + 1)
    x = synth.normal_f16((wl.bls, wl.h1), 1.0, g, DEV)
    y = stack.run(x, fg.FG_PHASE_DECODE, 1, L, fg.FG_ORDER_BLOCK)
    fg.fg_check()
    seqs = [0, 143]
    ol = oracle_layer({n: to_np(t) for n, t in w.items()}, wl.h1, wl.H, wl.h2)
    oc = _oracle_cache(k, v, seqs, L + 1)
    ref = layer_step(ol, to_np(x[seqs]), oc, DECODE, len(seqs), 1, pos=L)
    assert rel_l2(to_np(y[seqs]), ref) <= 5e-3
    # The appended K/V rows are the oracle's quantisation of the layer's own
    # k and v (bit-exact).  That row is recomputed through the same kernels
    # (rows do not depend on the other rows; M <= 256 as in the block), since
    # fp32 summation order may round a few k/v elements to the neighbouring
    # fp16 value, which can move a 4-bit code.
    L0 = stack.layers[0]
    a = fg.fg_layernorm(x[seqs], L0.ln1_g, L0.ln1_b)
    qkv = to_np(fg.fg_dequant_gemm_g4(a, L0.qkv, bias=L0.b_qkv))
    h1 = wl.h1
    for part, (codes, meta) in ((1, (stack.caches[0].k_codes, stack.caches[0].k_meta)),
                                (2, (stack.caches[0].v_codes, stack.caches[0].v_meta))):
        oc_codes, oc_meta = oracle.quantize_g4(qkv[:, part * h1:(part + 1) * h1].reshape(-1, wl.d))
        assert np.array_equal(to_np(codes[seqs, :, L]).reshape(oc_codes.shape), oc_codes)
        assert np.array_equal(to_np(meta[seqs, :, L]).reshape(oc_meta.shape), oc_meta)


@pytest.mark.parametrize("L,kv", [(1024, "g4"), (512, "f16"), (1024, "f16")])
def test_opt30b_decode_layer_bls144_context_and_cache_variants(L, kv):
    """The benchmark's other OPT-30B configurations at full size: the decode
    layer for the whole block of 144 sequences at context L + 1 (prompts of
    1024 tokens, the pages' second padded length) and over the uncompressed
    fp16 cache; 2 sampled sequences through the oracle (rel-L2 <= 5e-3).  The
    fp16 cache's appended rows equal the layer's own k and v (recomputed
    through the same kernels) bit for bit."""
    wl = synth.OPT30B
    g = synth.generator(31 + L, DEV)
    w = synth.layer_weights(wl.h1, wl.h2, g, DEV)
    w.update(synth.random_affine_params(wl.h1, wl.h2, g, DEV))
    k, v = _kv_rows(wl.bls, wl.H, L, wl.d, g, DEV)
    stack = LayerStack([quantize_layer(w, wl.h1, wl.H, wl.h2)], wl.gbs, wl.k, L + 1, DEV, kv=kv)
    if kv == "f16":
        c = fg.KV16.empty(wl.bls, wl.H, wl.d, L + 1, DEV)
        c.k[:, :, :L] = k
        c.v[:, :, :L] = v
        stack.caches[0] = c
    else:
        stack.caches[0] = _gpu_cache(k, v, L + 1)
    x = synth.normal_f16((wl.bls, wl.h1), 1.0, g, DEV)
    y = stack.run(x, fg.FG_PHASE_DECODE, 1, L, fg.FG_ORDER_BLOCK)
    fg.fg_check()
    seqs = [0, 143]
    ol = oracle_layer({n: to_np(t) for n, t in w.items()}, wl.h1, wl.H, wl.h2)
    if kv == "f16":
        oc = oracle.KVCache16(len(seqs), wl.H, wl.d, L + 1)
        oc.k[:, :, :L] = to_np(k[seqs])
        oc.v[:, :, :L] = to_np(v[seqs])
    else:
        oc = _oracle_cache(k, v, seqs, L + 1)
    ref = layer_step(ol, to_np(x[seqs]), oc, DECODE, len(seqs), 1, pos=L)
    assert rel_l2(to_np(y[seqs]), ref) <= 5e-3
    if kv == "f16":
        L0 = stack.layers[0]
        a = fg.fg_layernorm(x[seqs], L0.ln1_g, L0.ln1_b)
        qkv = fg.fg_dequant_gemm_g4(a, L0.qkv, bias=L0.b_qkv)
        h1 = wl.h1
        c = stack.caches[0]
        assert torch.equal(c.k[seqs, :, L].reshape(len(seqs), h1), qkv[:, h1:2 * h1])
        assert torch.equal(c.v[seqs, :, L].reshape(len(seqs), h1), qkv[:, 2 * h1:])


@pytest.mark.parametrize("bls", synth.SWEEP_GEMM_BLS)
@pytest.mark.parametrize("proj", ["qkv", "out", "fc1", "fc2"])
def test_opt175b_dequant_gemm_sampled(bls, proj):
    """OPT-175B-shaped projections at bls in {32, 144, 256, 512}: every row
    of Y on a 256-feature slice of W compared with the oracle."""
    h1, h2 = synth.OPT175B_H1, synth.OPT175B_H2
    N, K = {"qkv": (3 * h1, h1), "out": (h1, h1), "fc1": (h2, h1), "fc2": (h1, h2)}[proj]
    g = synth.generator(bls + N, DEV)
    w = synth.normal_f16((N, K), 0.02, g, DEV)
    x = synth.normal_f16((bls, K), 1.0, g, DEV)
    b = synth.normal_f16((N,), 0.1, g, DEV)
    q = fg.fg_quantize_g4(w)
    y = fg.fg_dequant_gemm_g4(x, q, bias=b, act=1 if proj == "fc1" else 0)
    fg.fg_check()
    n0 = (N // 2) // 128 * 128 + 64          # a slice that straddles two 128-row tiles
    sl = slice(n0, n0 + 256)
    codes, meta = oracle.quantize_g4(to_np(w[sl]))
    ref = oracle.linear_g4(to_np(x), codes, meta, bias=to_np(b[sl]),
                           act=1 if proj == "fc1" else 0).astype(np.float64)
    got = to_np(y[:, sl]).astype(np.float64)
    bound = gemm_bound(to_np(x), codes, meta) + ulp16(ref)
    assert np.all(np.abs(got - ref) <= bound)
    assert rel_l2(got, ref) < 2e-3


@pytest.mark.parametrize("ctx", synth.SWEEP_ATTN_CTX)
def test_opt175b_decode_attention_sampled(ctx):
    """OPT-175B decode attention at bls 144, 96 heads of 128, context in
    {512, 1024, 2048} (fused append at slot ctx-1): 4 sequences x all heads
    through the oracle, appended rows bit-exact."""
    B, H, d = synth.SWEEP_ATTN_BLS, synth.OPT175B_H, synth.OPT175B_H1 // synth.OPT175B_H
    g = synth.generator(ctx, DEV)
    k, v = _kv_rows(B, H, ctx - 1, d, g, DEV)
    cache = _gpu_cache(k, v, ctx)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, g, DEV)
    out = fg.fg_decode_attn_g4(qkv, cache, ctx - 1, fuse_append=True)
    fg.fg_check()
    seqs = [0, 50, 101, 143]
    oc = _oracle_cache(k, v, seqs, ctx)
    ref = oracle.decode_attn_g4(to_np(qkv[seqs]), oc, ctx - 1, append=True).astype(np.float64)
    got = to_np(out[seqs]).astype(np.float64)
    vmax = float(np.max(np.abs(oc.v_meta[..., 0]) + 15 * np.abs(oc.v_meta[..., 1])))
    assert np.all(np.abs(got - ref) <= 4e-3 * vmax + ulp16(ref))
    assert rel_l2(got, ref) < 2e-3
    assert np.array_equal(to_np(cache.k_codes[seqs, :, ctx - 1]), oc.k_codes[:, :, ctx - 1])
    assert np.array_equal(to_np(cache.v_codes[seqs, :, ctx - 1]), oc.v_codes[:, :, ctx - 1])


def test_opt67b_block_orders_identical_full_block():
    """OPT-6.7B-shaped layers at the full block (gbs 32 x k 8 = 256, prompt
    512): whole-block launches, batch order and zig-zag order give
    bit-identical prefill and decode outputs."""
    wl = synth.OPT6_7B
    outs = []
    for order in (lambda t: fg.FG_ORDER_BLOCK, lambda t: fg.FG_ORDER_BATCHES,
                  lambda t: fg.FG_ORDER_BATCHES if t % 2 == 0 else fg.FG_ORDER_BATCHES_REV):
        g = synth.generator(67, DEV)
        w = synth.layer_weights(wl.h1, wl.h2, g, DEV)
        stack = LayerStack([quantize_layer(w, wl.h1, wl.H, wl.h2)], wl.gbs, wl.k, wl.s + 3, DEV)
        del w
        x = synth.normal_f16((wl.bls * wl.s, wl.h1), 1.0, g, DEV)
        ys = [stack.run(x, fg.FG_PHASE_PREFILL, wl.s, 0, order(0))[::97].clone()]
        for t in (1, 2):
            xt = synth.normal_f16((wl.bls, wl.h1), 1.0, g, DEV)
            ys.append(stack.run(xt, fg.FG_PHASE_DECODE, 1, wl.s + t - 1, order(t)).clone())
        fg.fg_check()
        outs.append(ys)
        del stack, x
        torch.cuda.empty_cache()
    for a, b, c in zip(*outs):
        assert torch.equal(a, b) and torch.equal(a, c)


def test_opt13b_sequence_independence_full_size():
    """OPT-1.3B-shaped model slice (4 layers, vocab 50272), gbs 16, prompt
    512, 3 decode steps: rows never mix -- sequence 5's logits are bit for
    bit the same when the other 15 prompts and decode tokens are replaced by
    different ones (same block size, so the same launch plan)."""
    from bit_group_quant_gb300.model import Model
    wl = synth.OPT1_3B
    g = synth.generator(13, DEV)
    layers = [quantize_layer(synth.layer_weights(wl.h1, wl.h2, g, DEV), wl.h1, wl.H, wl.h2)
              for _ in range(4)]
    et, ep = synth.embeddings(wl.vocab, wl.cap, wl.h1, g, DEV)
    ones = torch.ones(wl.h1, dtype=torch.float16, device=DEV)
    zeros = torch.zeros(wl.h1, dtype=torch.float16, device=DEV)
    prompt = synth.token_ids((wl.gbs, wl.s), wl.vocab, g, DEV)
    dec = synth.token_ids((3, wl.gbs), wl.vocab, g, DEV)
    other_p = synth.token_ids((wl.gbs, wl.s), wl.vocab, g, DEV)
    other_d = synth.token_ids((3, wl.gbs), wl.vocab, g, DEV)
    other_p[5], other_d[:, 5] = prompt[5], dec[:, 5]
    m = Model(LayerStack(layers, wl.gbs, 1, wl.cap, DEV), et, ep, ones, zeros)
    full = [t.clone() for t in m.generate(prompt, dec)]
    mixed = m.generate(other_p, other_d)
    fg.fg_check()
    for a, b in zip(full, mixed):
        assert torch.isfinite(a).all()
        assert torch.equal(a[5:6], b[5:6])
        assert not torch.equal(a[4:5], b[4:5])
