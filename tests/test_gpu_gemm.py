"""tcgen05 dequant-GEMM and fp16 LM-head GEMM against the oracle, through the
C ABI; row results independent of M (bitwise)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, gemm_bound, rel_l2, to_np, ulp16

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed, wstd=0.02):
    g = synth.generator(seed)
    x = synth.normal_f16((M, K), 1.0, g)
    w = synth.normal_f16((N, K), wstd, g)
    b = synth.normal_f16((N,), 0.1, g)
    r = synth.normal_f16((M, N), 1.0, g)
    return x, w, b, r


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 64), (4, 2304, 768), (16, 768, 3072), (144, 512, 1024),
    (200, 384, 512), (300, 256, 640), (513, 128, 256), (4, 128, 8192),
    (512, 512, 1024), (768, 384, 512),   # 256-row tiles: 3-stage ring, 4- and 1-CTA clusters
    # decode regime, odd tile counts (1-CTA clusters): a partial last weight
    # tile and activation rows past M, read as zeros in the staged residual
    # tile; tiles split over two and three clusters (several later parts)
    (37, 1040, 512), (130, 2176, 1536),
])
@pytest.mark.parametrize("act,use_bias,use_res", [(0, True, True), (1, True, False), (0, False, False)])
def test_dequant_gemm_matches_oracle(M, N, K, act, use_bias, use_res):
    x, w, b, r = _case(M, N, K, M * 31 + N + K)
    q = fg.fg_quantize_g4(w.to(DEV))
    y = fg.fg_dequant_gemm_g4(x.to(DEV), q, bias=b.to(DEV) if use_bias else None,
                              residual=r.to(DEV) if use_res else None, act=act)
    fg.fg_check()
    codes, meta = oracle.quantize_g4(w.numpy())
    ref = oracle.linear_g4(x.numpy(), codes, meta, bias=b.numpy() if use_bias else None,
                           residual=r.numpy() if use_res else None, act=act)
    got = to_np(y).astype(np.float64)
    want = ref.astype(np.float64)
    bound = gemm_bound(x.numpy(), codes, meta) + ulp16(want)
    bad = np.abs(got - want) > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], want[bad][:5])
    assert rel_l2(got, want) < 2e-3


def test_dequant_gemm_rows_independent_of_M():
    """Bitwise: a block of 144 rows in one launch equals three launches of 48
    rows (the block schedule's fused and per-batch orders)."""
    N, K = 1024, 2048
    x, w, b, r = _case(144, N, K, 77)
    q = fg.fg_quantize_g4(w.to(DEV))
    xd, bd, rd = x.to(DEV), b.to(DEV), r.to(DEV)
    full = fg.fg_dequant_gemm_g4(xd, q, bias=bd, residual=rd, act=1)
    parts = [fg.fg_dequant_gemm_g4(xd[i:i + 48].contiguous(), q, bias=bd,
                                   residual=rd[i:i + 48].contiguous(), act=1)
             for i in range(0, 144, 48)]
    one = fg.fg_dequant_gemm_g4(xd[5:6].contiguous(), q, bias=bd, residual=rd[5:6].contiguous(), act=1)
    torch.cuda.synchronize()
    assert torch.equal(full, torch.cat(parts))
    assert torch.equal(full[5:6], one)


def test_dequant_gemm_permutation_exact():
    """A permutation weight survives 4-bit quantisation exactly; Y must pick
    columns of X exactly (catches transposed operands or swizzle errors)."""
    K = N = 1024
    perm = np.random.default_rng(3).permutation(K)
    w = np.zeros((N, K), np.float16)
    w[np.arange(N), perm] = 1.0
    x = synth.normal_f16((37, K), 1.0, synth.generator(4))
    q = fg.fg_quantize_g4(torch.from_numpy(w).to(DEV))
    y = fg.fg_dequant_gemm_g4(x.to(DEV), q)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(y), x.numpy()[:, perm])


@pytest.mark.parametrize("N,K", [(384, 512), (256, 1024)])
def test_dequant_gemm_identity_gives_dequantised_weights_exactly(N, K):
    """X = I: every output is one product 1 * w^[n][k], exact in fp32 and back
    in fp16, so Y^T must equal the oracle's dequantised weights bit for bit --
    a direct pin of the fused on-chip dequantisation (every code, group,
    swizzle position and K-walk offset) against the definition."""
    g = synth.generator(K + N)
    w = synth.normal_f16((N, K), 0.02, g)
    w[:, 64:128] = 0.0                       # a constant group (scale 0)
    w[:3, 128:192] = torch.linspace(-2.0, 2.0, 64, dtype=torch.float16)   # wide range
    q = fg.fg_quantize_g4(w.to(DEV))
    eye = torch.eye(K, dtype=torch.float16, device=DEV)
    y = fg.fg_dequant_gemm_g4(eye, q)
    torch.cuda.synchronize()
    codes, meta = oracle.quantize_g4(w.numpy())
    want = oracle.dequant_g4(codes, meta)
    # compared as values: a weight that rounds to -0 comes out of the sum of
    # products as +0
    assert np.array_equal(to_np(y).T.astype(np.float32), np.asarray(want).astype(np.float32))


def test_dequant_gemm_zero_rows():
    q = fg.fg_quantize_g4(synth.normal_f16((128, 128), 0.02, synth.generator(0)).to(DEV))
    y = fg.fg_dequant_gemm_g4(torch.empty((0, 128), dtype=torch.float16, device=DEV), q)
    assert y.shape == (0, 128)


@pytest.mark.parametrize("M,N,K", [(3, 50272 // 8, 768), (144, 1040, 2048)])
def test_lm_head_f32out(M, N, K):
    g = synth.generator(M + N)
    x = synth.normal_f16((M, K), 1.0, g)
    w = synth.normal_f16((N, K), 0.02, g)
    y = fg.fg_gemm_f16_f32out(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.linear_f16_f32out(x.numpy(), w.numpy()).astype(np.float64)
    dot_abs = np.abs(x.numpy().astype(np.float64)) @ np.abs(w.numpy().astype(np.float64)).T
    assert np.all(np.abs(to_np(y) - ref) <= K * 2.0 ** -23 * dot_abs + 1e-30)


def test_split_k_path_used_and_correct():
    """Few output tiles and long K take the K-split + fixed-order reduction."""
    N, K = 256, 8192
    assert fg.fg_dequant_gemm_workspace_bytes(8, N, K) > 0
    x, w, b, r = _case(8, N, K, 9)
    q = fg.fg_quantize_g4(w.to(DEV))
    y = fg.fg_dequant_gemm_g4(x.to(DEV), q, bias=b.to(DEV), residual=r.to(DEV), act=1)
    torch.cuda.synchronize()
    codes, meta = oracle.quantize_g4(w.numpy())
    ref = oracle.linear_g4(x.numpy(), codes, meta, bias=b.numpy(), residual=r.numpy(), act=1)
    bound = gemm_bound(x.numpy(), codes, meta) + ulp16(ref)
    assert np.all(np.abs(to_np(y).astype(np.float64) - ref.astype(np.float64)) <= bound)


@pytest.mark.parametrize("M,N,K", [(32, 12288, 49152), (144, 7168, 28672)])
def test_dequant_gemm_repeatable_long_k(M, N, K):
    """Long K walks (192 and 56 codes boxes per CTA, 4- and 2-CTA clusters):
    repeated launches give bit-identical results.  Every codes box slot is
    rewritten by TMA hundreds of times per CTA here, so a slot released
    before its reads are ordered shows up as run-to-run differences."""
    g = synth.generator(M + N, DEV)
    q = fg.fg_quantize_g4(synth.normal_f16((N, K), 0.02, g, DEV))
    x = synth.normal_f16((M, K), 1.0, g, DEV)
    ys = [fg.fg_dequant_gemm_g4(x, q) for _ in range(6)]
    fg.fg_check()
    for y in ys[1:]:
        assert torch.equal(ys[0], y)
