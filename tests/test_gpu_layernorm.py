"""LayerNorm through the C ABI against the oracle: y = (x - mean) /
sqrt(var + eps) * gamma + beta with mean and biased variance in fp32.  Both
sides compute the same formula; only the order of the fp32 sums differs, so
each output lies within the error bound of its sums from the fp64 value and
from the oracle's, and almost always equals the oracle's exactly.  Covers
single rows, the decode block (144 rows of 7168), ragged column counts, the
largest supported width, rows far from zero mean, and strided rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, to_np, ulp16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,offset", [
    (1, 64, 0.0), (3, 768, 0.0), (144, 7168, 0.0), (257, 2048, 3.0), (33, 12288, 0.0),
    (5, 16384, -2.0), (1000, 192, 0.5),
])
def test_layernorm_matches_oracle(rows, cols, offset):
    g = synth.generator(rows * 7 + cols)
    x = (synth.normal_f16((rows, cols), 1.0, g).float() + offset).half()
    gamma = (1 + synth.normal_f16((cols,), 0.1, g).float()).half()
    beta = synth.normal_f16((cols,), 0.1, g)
    y = fg.fg_layernorm(x.to(DEV), gamma.to(DEV), beta.to(DEV), 1e-5)
    fg.fg_check()
    ref = oracle.layernorm(x.numpy(), gamma.numpy(), beta.numpy(), 1e-5).astype(np.float64)
    got = to_np(y).astype(np.float64)
    # Error bounds from the two sides' fp32 sums (mean, then the squared
    # deviations): the oracle sums each row in sequence (error up to
    # cols * 2^-24 of the sum of |x|), the kernel per thread and then by a
    # tree (cols/256 + 13 additions deep).  The normalised value x^ moves by
    # that relative to the row's spread, and gamma carries it to y.
    x64 = x.numpy().astype(np.float64)
    mu = x64.mean(1, keepdims=True)
    sd = np.sqrt(x64.var(1, keepdims=True) + 1e-5)
    xn = (x64 - mu) / sd
    g64, b64 = gamma.numpy().astype(np.float64), beta.numpy().astype(np.float64)
    exact = xn * g64 + b64
    scale = np.abs(g64) * (np.abs(x64).mean(1, keepdims=True) / sd + np.abs(xn)) * 2.0 ** -23
    assert np.all(np.abs(got - exact) <= ulp16(exact) + (cols / 256 + 13) * scale + 1e-6)
    assert np.all(np.abs(got - ref) <= 2 * ulp16(ref) + (cols + cols / 256 + 13) * scale + 1e-6)
    assert np.mean(got == ref) > 0.95


def test_layernorm_strided_rows_equal_contiguous():
    rows, cols, ld = 37, 2048, 2048 + 192
    g = synth.generator(5)
    big = synth.normal_f16((rows, ld), 1.0, g).to(DEV)
    gamma = synth.normal_f16((cols,), 1.0, g).to(DEV)
    beta = synth.normal_f16((cols,), 1.0, g).to(DEV)
    a = fg.fg_layernorm(big, gamma, beta, 1e-5, rows=rows, x_ld=ld)
    b = fg.fg_layernorm(big[:, :cols].contiguous(), gamma, beta, 1e-5)
    fg.fg_check()
    assert torch.equal(a, b)
