"""Oracle parity of the prefill as the benchmark runs it.

The prefill projects all s prompt tokens of every sequence of the block, then
attends causally over them and stores their K/V rows ("FlexGen 完全拆解",
section 从 Transformer 推理的数据流重新定义卸载).  In this library a projection
whose block has at least 8192 planned rows first dequantises the weights once
into fp16 in the workspace, then runs the fp16 tensor-core pipeline; these
tests compare that regime with the oracle element by element at small shapes
(a whole and a ragged last token tile, all three epilogues), then at the
OPT-30B block's full size (144 sequences x 512 tokens = 73,728 rows) on
sampled rows and features, a full prefill layer on sampled sequences, and the
prefill attention at the pages' two padded lengths, 512 and 1024.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, quantize_layer
from oracle.model import PREFILL, layer_step
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, gemm_bound, rel_l2, to_np, ulp16

pytestmark = pytest.mark.gpu

F16W_ROWS = 8192     # planned rows from which the weights are dequantised once


def _compare_gemm(x_np, w_np, b_np, r_np, act, got, rows=None, feats=None):
    """got: the GPU's Y restricted to (rows, feats); the oracle computes the
    same outputs from its own quantisation of the fp16 weights."""
    xs = x_np if rows is None else x_np[rows]
    ws = w_np if feats is None else w_np[feats]
    codes, meta = oracle.quantize_g4(ws)
    bs = None if b_np is None else (b_np if feats is None else b_np[feats])
    rs = None
    if r_np is not None:
        rs = r_np if rows is None else r_np[rows]
        rs = rs if feats is None else rs[:, feats]
    ref = oracle.linear_g4(xs, codes, meta, bias=bs, residual=rs, act=act).astype(np.float64)
    got = np.asarray(got, np.float64)
    bound = gemm_bound(xs, codes, meta) + ulp16(ref)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    assert rel_l2(got, ref) < 2e-3


@pytest.mark.parametrize("M", [F16W_ROWS, F16W_ROWS + 80])     # whole / ragged last tile
@pytest.mark.parametrize("N,K", [(512, 1024), (256, 2048)])
@pytest.mark.parametrize("act,use_bias,use_res", [(0, True, True), (1, True, False), (0, False, False)])
def test_fp16_weight_regime_matches_oracle(M, N, K, act, use_bias, use_res):
    # the workspace query plans the fp16 copy of the weights for this M
    assert fg.fg_dequant_gemm_workspace_bytes(M, N, K) >= N * K * 2
    assert fg.fg_dequant_gemm_workspace_bytes(F16W_ROWS - 1, N, K) < N * K * 2
    g = synth.generator(M + 7 * N + K + act)
    x = synth.normal_f16((M, K), 1.0, g)
    w = synth.normal_f16((N, K), 0.02, g)
    b = synth.normal_f16((N,), 0.1, g)
    r = synth.normal_f16((M, N), 1.0, g)
    q = fg.fg_quantize_g4(w.to(DEV))
    y = fg.fg_dequant_gemm_g4(x.to(DEV), q, bias=b.to(DEV) if use_bias else None,
                              residual=r.to(DEV) if use_res else None, act=act)
    fg.fg_check()
    _compare_gemm(x.numpy(), w.numpy(), b.numpy() if use_bias else None,
                  r.numpy() if use_res else None, act, to_np(y))


def test_fp16_weight_regime_rows_independent_of_M_bitwise():
    """Inside the prefill regime every row's result is independent of M and of
    the row's position: the rows of an 8192-row launch equal, bit for bit,
    the same rows inside a longer launch whose last 256-row tile is ragged."""
    N, K = 384, 1536
    g = synth.generator(5, DEV)
    w = synth.normal_f16((N, K), 0.02, g, DEV)
    x = synth.normal_f16((2 * F16W_ROWS + 80, K), 1.0, g, DEV)
    b = synth.normal_f16((N,), 0.1, g, DEV)
    q = fg.fg_quantize_g4(w)
    big = fg.fg_dequant_gemm_g4(x, q, bias=b, act=1)
    small = fg.fg_dequant_gemm_g4(x[F16W_ROWS + 80:].contiguous(), q, bias=b, act=1)
    fg.fg_check()
    assert torch.equal(big[F16W_ROWS + 80:], small)


def _sample_rows(M, tile=256):
    """Rows spread over every 256-row token tile, with both edges of the first
    and last tiles."""
    rows = set(range(0, M, 61)) | {0, 1, tile - 1, tile, M - tile, M - 2, M - 1}
    return np.array(sorted(r for r in rows if 0 <= r < M))


@pytest.mark.slow
@pytest.mark.parametrize("proj", ["qkv", "out", "fc1", "fc2"])
def test_opt30b_prefill_projection_full_size_sampled(proj):
    """One OPT-30B prefill projection at the benchmark's full size (144
    sequences x 512 tokens = 73,728 rows, weights dequantised once into fp16),
    with its epilogue as in the layer (out and fc2 add the residual, fc1
    applies ReLU): a 256-feature slice straddling two weight tiles, on rows
    sampled from every token tile."""
    wl = synth.OPT30B
    M = wl.bls * wl.s
    h1, h2 = wl.h1, wl.h2
    N, K = {"qkv": (3 * h1, h1), "out": (h1, h1), "fc1": (h2, h1), "fc2": (h1, h2)}[proj]
    act = 1 if proj == "fc1" else 0
    g = synth.generator(3000 + N + K, DEV)
    w = synth.normal_f16((N, K), 0.02, g, DEV)
    b = synth.normal_f16((N,), 0.1, g, DEV)
    x = synth.normal_f16((M, K), 1.0, g, DEV)
    r = synth.normal_f16((M, N), 1.0, g, DEV) if proj in ("out", "fc2") else None
    q = fg.fg_quantize_g4(w)
    assert fg.fg_dequant_gemm_workspace_bytes(M, N, K) >= N * K * 2
    y = fg.fg_dequant_gemm_g4(x, q, bias=b, residual=r, act=act)
    fg.fg_check()
    rows = _sample_rows(M)
    n0 = (N // 2) // 128 * 128 + 64
    feats = np.arange(n0, n0 + 256)
    ri = torch.from_numpy(rows).to(DEV)
    got = to_np(y[ri][:, n0:n0 + 256])
    x_s = to_np(x[ri])
    r_s = None if r is None else to_np(r[ri][:, n0:n0 + 256])
    del x, y, r
    torch.cuda.empty_cache()
    _compare_gemm(x_s, to_np(w[n0:n0 + 256]), to_np(b)[feats], r_s, act, got)


@pytest.mark.slow
def test_opt30b_prefill_layer_bls144_sampled():
    """The OPT-30B prefill layer for the whole block (48 x 3 = 144 sequences
    of 512 tokens, one weight-stationary launch per projection) with
    non-trivial biases and LayerNorm parameters: 2 sampled sequences through
    the oracle at relative L2 <= 5e-3, and their stored K/V rows (all 512
    slots, every head) bit-exact against the oracle's quantisation of the
    layer's own k and v."""
    wl = synth.OPT30B
    B, s, h1, H, d = wl.bls, wl.s, wl.h1, wl.H, wl.d
    g = synth.generator(3030, DEV)
    w = synth.layer_weights(h1, wl.h2, g, DEV)
    w.update(synth.random_affine_params(h1, wl.h2, g, DEV))
    stack = LayerStack([quantize_layer(w, h1, H, wl.h2)], wl.gbs, wl.k, s + 1, DEV)
    x = synth.normal_f16((B * s, h1), 1.0, g, DEV)
    y = stack.run(x, fg.FG_PHASE_PREFILL, s, 0, fg.FG_ORDER_BLOCK)
    fg.fg_check()
    seqs = [0, 143]
    cache = stack.caches[0]
    kc, km = to_np(cache.k_codes[seqs, :, :s]), to_np(cache.k_meta[seqs, :, :s])
    vc, vm = to_np(cache.v_codes[seqs, :, :s]), to_np(cache.v_meta[seqs, :, :s])
    got = to_np(y.view(B, s, h1)[seqs])
    xs = to_np(x.view(B, s, h1)[seqs]).reshape(-1, h1)
    # the layer's own q|k|v rows, through the same public kernels at the same
    # planned size (the whole block)
    L0 = stack.layers[0]
    a = fg.fg_layernorm(x, L0.ln1_g, L0.ln1_b)
    qkv = fg.fg_dequant_gemm_g4(a, L0.qkv, bias=L0.b_qkv).view(B, s, 3 * h1)
    own = to_np(qkv[seqs])
    del a, qkv, y, x, stack
    torch.cuda.empty_cache()
    for part, codes, meta in ((1, kc, km), (2, vc, vm)):
        rows = own[:, :, part * h1:(part + 1) * h1].reshape(len(seqs), s, H, d).transpose(0, 2, 1, 3)
        oc, om = oracle.quantize_g4(np.ascontiguousarray(rows).reshape(-1, d))
        assert np.array_equal(codes.reshape(oc.shape), oc)
        assert np.array_equal(meta.reshape(om.shape).view(np.uint32), om.view(np.uint32))
    ol = oracle_layer({n: to_np(t) for n, t in w.items()}, h1, H, wl.h2)
    oc = oracle.KVCache(len(seqs), H, d, s + 1)
    ref = layer_step(ol, xs, oc, PREFILL, len(seqs), s)
    assert rel_l2(got.reshape(-1, h1), ref) <= 5e-3


@pytest.mark.slow
@pytest.mark.parametrize("s,padded", [(512, False), (512, True), (1024, False)])
def test_prefill_attention_full_size_sampled(s, padded):
    """Prefill attention and K/V store at the OPT-30B block (144 sequences, 56
    heads of 128) for prompts of 512 and 1024 tokens (8 and 16 query blocks,
    heaviest first), dense and with a seeded mix of left-padding counts: 3
    sampled sequences through the oracle, their stored K/V bit-exact."""
    wl = synth.OPT30B
    B, H, d = wl.bls, wl.H, wl.d
    h1 = H * d
    g = synth.generator(4000 + s + padded, DEV)
    qkv = synth.normal_f16((B * s, 3 * h1), 1.0, g, DEV)
    pad = synth.pad_counts(B, s, g, device=DEV) if padded else None
    cache = fg.KV4.empty(B, H, d, s + 1, DEV)
    out = fg.fg_prefill_attn(qkv, B, s, H, d, cache=cache, pad=pad)
    fg.fg_check()
    seqs = [0, 71, 143]
    q_s = to_np(qkv.view(B, s, 3 * h1)[seqs]).reshape(-1, 3 * h1)
    pad_s = None if pad is None else to_np(pad)[seqs]
    ref = oracle.prefill_attn(q_s, len(seqs), s, H, d, pad=pad_s).astype(np.float64)
    got = to_np(out.view(B, s, h1)[seqs]).reshape(-1, h1).astype(np.float64)
    vmax = float(np.abs(q_s[:, 2 * h1:]).max())
    assert np.all(np.abs(got - ref) <= 4e-3 * vmax + ulp16(ref))
    assert rel_l2(got, ref) < 2e-3
    if pad_s is not None:
        for i, p in enumerate(pad_s):
            assert not np.any(got.reshape(len(seqs), s, h1)[i, :p])
    oc = oracle.KVCache(len(seqs), H, d, s + 1)
    oracle.kv_store_prefill(q_s, len(seqs), s, oc)
    for name in ("k_codes", "v_codes", "k_meta", "v_meta"):
        assert np.array_equal(to_np(getattr(cache, name)[seqs]), getattr(oc, name)), name
