"""fg_dequant_gemm_g4_noalloc: the dequant-GEMM for callers that cannot
allocate device memory (a plugin inside a host program that owns the whole
device-memory budget, or a latency-critical loop where cudaMalloc would
synchronise the device).  It keeps its K-split scratch in a fixed array
inside libfg instead of a caller workspace.  Called through the C ABI, two
calls in a row, each checked against fg_dequant_gemm_g4 with a caller
workspace.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, gemm_bound, rel_l2, to_np, ulp16

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    g = synth.generator(seed)
    x = synth.normal_f16((M, K), 1.0, g).to(DEV)
    w = synth.normal_f16((N, K), 0.02, g).to(DEV)
    b = synth.normal_f16((N,), 0.1, g).to(DEV)
    r = synth.normal_f16((M, N), 1.0, g).to(DEV)
    return x, fg.fg_quantize_g4(w), b, r


def _noalloc_c(x, q, b, r, act, y):
    """Direct C-ABI call of the new entry point."""
    lib = fg.load()
    c = q.c()
    st = lib.fg_dequant_gemm_g4_noalloc(
        ctypes.c_void_p(x.data_ptr()), x.shape[0], ctypes.byref(c),
        ctypes.c_void_p(b.data_ptr()), None if r is None else ctypes.c_void_p(r.data_ptr()),
        act, ctypes.c_void_p(y.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _check_against_existing(x, q, b, r, act, exact=True):
    M, N = x.shape[0], q.rows
    assert fg.fg_dequant_gemm_workspace_bytes(M, N, q.cols) > 0   # a path that needs scratch
    y_new = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    assert _noalloc_c(x, q, b, r, act, y_new) == fg.FG_OK, fg.load().fg_last_error()
    y_old = fg.fg_dequant_gemm_g4(x, q, bias=b, residual=r, act=act)
    fg.fg_check()
    got, want = to_np(y_new).astype(np.float64), to_np(y_old).astype(np.float64)
    codes, meta = to_np(q.codes), to_np(q.meta)
    bound = gemm_bound(to_np(x), codes, meta) + ulp16(want)
    assert np.all(np.abs(got - want) <= bound)
    assert rel_l2(got, want) < 2e-3
    # the same kernel and plan run on both sides, so the results agree
    # exactly (at M >= 8192 the allocating call multiplies weights dequantised
    # once into its workspace, in another summation order: the bound above)
    if exact:
        assert torch.equal(y_new, y_old)


def test_noalloc_matches_existing_entry_point_twice():
    # first call: few output tiles, long K -> K split into fp32 partials
    _check_against_existing(*_inputs(8, 256, 8192, 1), act=1)
    # second call right after, other shape and inputs: the scratch keeps the
    # first call's partials, and none of them may leak into this result
    _check_against_existing(*_inputs(144, 512, 4096, 2), act=0)


def test_noalloc_split_k_across_ctas_twice():
    # 161..256 rows: one token tile with K split across CTAs, fp32 partials in
    # the built-in array, then summed in a fixed order by a second kernel
    assert fg.fg_dequant_gemm_workspace_bytes(200, 512, 4096) <= fg.NOALLOC_SCRATCH_BYTES
    _check_against_existing(*_inputs(200, 512, 4096, 3), act=1)
    _check_against_existing(*_inputs(232, 256, 2048, 4), act=0)


def test_noalloc_prefill_sized_block_uses_no_weight_copy():
    # M >= 8192: the allocating entry point dequantises the weights once into
    # its workspace; this call is offered no scratch for that and takes the
    # fused path, with the same result up to the fp32 summation order
    M, N, K = 8192 + 48, 256, 512
    assert fg.fg_dequant_gemm_workspace_bytes(M, N, K) == N * K * 2
    _check_against_existing(*_inputs(M, N, K, 5), act=0, exact=False)
    _check_against_existing(*_inputs(M, N, K, 6), act=1, exact=False)


def test_noalloc_rejects_scratch_beyond_its_maximum():
    limit = fg.NOALLOC_SCRATCH_BYTES
    shape = None
    for M, N, K in [(256, 3072, 4096), (256, 1536, 8192), (256, 768, 16384), (256, 2048, 65536)]:
        if fg.fg_dequant_gemm_workspace_bytes(M, N, K) > limit:
            shape = (M, N, K)
            break
    if shape is None:
        pytest.skip("no candidate shape needs more than the fixed scratch on this GPU")
    M, N, K = shape
    x = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    q = fg.Q4.empty(N, K, DEV)
    b = torch.zeros(N, dtype=torch.float16, device=DEV)
    y = torch.empty((M, N), dtype=torch.float16, device=DEV)
    assert _noalloc_c(x, q, b, None, 0, y) == fg.FG_ERR_WORKSPACE
    assert b"built-in scratch holds" in fg.load().fg_last_error()
