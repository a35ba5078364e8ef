"""Failure detection on the GPU without a GPU fault: a producer that never
arms a barrier (the drop-arrive test knob) makes the consumers' bounded waits
expire.  The launch must report FG_ERR_TIMEOUT through fg_check, a launch made
before the check must end without waiting again (its output is unspecified),
and the context must stay usable: the next launch after the check computes
the right result."""
import numpy as np
import pytest
import torch

import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, to_np

pytestmark = pytest.mark.gpu

WAIT_NS = 30_000_000   # 30 ms: every wait of the failing launch gives up quickly


@pytest.fixture
def short_waits():
    fg.fg_check()
    fg.fg_debug_set(fg.FG_KNOB_WAIT_NS, WAIT_NS)
    yield
    fg.fg_debug_set(fg.FG_KNOB_WAIT_NS, 0)
    fg.fg_debug_set(fg.FG_KNOB_DROP_ARRIVE, 0)
    try:
        fg.fg_check()
    except fg.FgError:
        pass


# M 16 with K a multiple of 256: the TMEM-operand kernel (also with a
# residual, whose tiles a TMA warp stages: its waits must end too); M 200:
# one token tile with K split across CTAs; M 300: whole tiles; M 8192: the
# weights dequantised once, then the CTA-pair GEMM
@pytest.mark.parametrize("M,N,K,res", [(16, 512, 1024, False), (16, 512, 1024, True),
                                       (200, 384, 512, False), (300, 256, 640, False),
                                       (8192, 384, 512, False)])
def test_dropped_arrive_reports_timeout_and_context_survives(short_waits, M, N, K, res):
    g = synth.generator(M + N + K, DEV)
    x = synth.normal_f16((M, K), 1.0, g, DEV)
    q = fg.fg_quantize_g4(synth.normal_f16((N, K), 0.02, g, DEV))
    r = synth.normal_f16((M, N), 1.0, g, DEV) if res else None
    good = fg.fg_dequant_gemm_g4(x, q, residual=r)
    fg.fg_check()
    ref = to_np(good).copy()

    fg.fg_debug_set(fg.FG_KNOB_DROP_ARRIVE, 1)
    bad = torch.zeros_like(good)
    fg.fg_dequant_gemm_g4(x, q, residual=r, Y=bad)   # box 0 never armed: waits expire
    fg.fg_dequant_gemm_g4(x, q, residual=r, Y=torch.empty_like(good))   # status set: skips its work
    with pytest.raises(fg.FgError) as e:
        fg.fg_check()
    assert e.value.status == fg.FG_ERR_TIMEOUT

    again = fg.fg_dequant_gemm_g4(x, q, residual=r)   # knob consumed, status cleared
    fg.fg_check()
    assert np.array_equal(to_np(again), ref)
