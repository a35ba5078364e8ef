"""GPU quantiser, dequantiser and KV append against the oracle: bit-exact
codes, metadata and packed bytes (the quantiser's integer decisions are
taken in fp32 on both sides)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, to_np

pytestmark = pytest.mark.gpu


def _special_rows():
    rng = np.random.default_rng(0)
    rows = [
        rng.standard_normal(64 * 12) * 0.02,
        rng.standard_normal(64 * 12),
        np.repeat([0.0, 1.5, -3.25, 65504.0, -65504.0, 6e-8, 0.1, -0.0, 0.0, 2.0, -2.0, 5.0], 64),
        rng.uniform(-65504, 65504, 64 * 12),
        rng.uniform(-5, -1, 64 * 12),
        rng.standard_normal(64 * 12) * 1e-6,
    ]
    out = rng.standard_normal(64 * 12) * 0.1
    out[::64] = 40.0
    rows.append(out)
    z = np.zeros(64 * 12)
    z[1::7] = -0.0
    rows.append(z * -1.0)
    # exact ties of the rounding: values on (m + (k + 1/2) * scale)
    t = np.zeros(64 * 12)
    for g in range(12):
        o = (g % 3) * 16.0                  # min o, max o + 15, scale exactly 1
        grp = np.concatenate([[o, o + 15.0], o + (np.arange(62) % 15) + 0.5])
        t[g * 64:(g + 1) * 64] = grp
    rows.append(t)
    return np.stack(rows).astype(np.float16)


@pytest.mark.parametrize("rows,cols", [(1, 64), (3, 192), (17, 768), (129, 2048), (1000, 4096)])
def test_quantize_bit_exact(rows, cols):
    g = synth.generator(rows * 7 + cols)
    x = synth.normal_f16((rows, cols), 0.02, g)
    q = fg.fg_quantize_g4(x.to(DEV))
    torch.cuda.synchronize()
    codes, meta = oracle.quantize_g4(x.numpy())
    assert np.array_equal(to_np(q.codes), codes)
    assert np.array_equal(to_np(q.meta).view(np.uint32), meta.view(np.uint32))


def test_quantize_special_groups_bit_exact():
    x = _special_rows()
    q = fg.fg_quantize_g4(torch.from_numpy(x).to(DEV))
    codes, meta = oracle.quantize_g4(x)
    assert np.array_equal(to_np(q.codes), codes)
    assert np.array_equal(to_np(q.meta).view(np.uint32), meta.view(np.uint32))


def test_dequant_bit_exact():
    x = _special_rows()
    q = fg.fg_quantize_g4(torch.from_numpy(x).to(DEV))
    xh = fg.fg_dequant_g4(q)
    codes, meta = oracle.quantize_g4(x)
    ref = oracle.dequant_g4(codes, meta)
    assert np.array_equal(to_np(xh).view(np.uint16), ref.view(np.uint16))


def test_quantize_large_sampled():
    """Weight-load size (an OPT-30B fc1 matrix, 28672 x 7168): sampled rows
    compared with the oracle one by one."""
    g = synth.generator(5, DEV)
    x = synth.normal_f16((28672, 7168), 0.02, g, DEV)
    q = fg.fg_quantize_g4(x)
    torch.cuda.synchronize()
    rows = np.random.default_rng(1).choice(28672, 24, replace=False)
    rows = np.concatenate([rows, [0, 28671]])
    xs = to_np(x[torch.as_tensor(rows, device=DEV)])
    codes, meta = oracle.quantize_g4(xs)
    assert np.array_equal(to_np(q.codes[torch.as_tensor(rows, device=DEV)]), codes)
    assert np.array_equal(to_np(q.meta[torch.as_tensor(rows, device=DEV)]), meta)


@pytest.mark.parametrize("B,H,d", [(4, 12, 64), (3, 2, 128)])
def test_kv_append_bit_exact(B, H, d):
    g = synth.generator(B * H + d)
    h1 = H * d
    ld = 3 * h1 + 8                                  # a padded row stride
    qkv = synth.normal_f16((B, ld), 1.0, g)
    cap = 7
    cache = fg.KV4.empty(B, H, d, cap, DEV)
    fg.fg_kv_append_g4(qkv.to(DEV), cache, pos=5)
    torch.cuda.synchronize()
    qn = qkv.numpy()
    for b in range(B):
        for h in range(H):
            kc, km = oracle.quantize_g4(qn[b:b + 1, h1 + h * d:h1 + (h + 1) * d])
            vc, vm = oracle.quantize_g4(qn[b:b + 1, 2 * h1 + h * d:2 * h1 + (h + 1) * d])
            assert np.array_equal(to_np(cache.k_codes[b, h, 5]), kc[0])
            assert np.array_equal(to_np(cache.v_codes[b, h, 5]), vc[0])
            assert np.array_equal(to_np(cache.k_meta[b, h, 5]), km[0])
            assert np.array_equal(to_np(cache.v_meta[b, h, 5]), vm[0])
    # other slots untouched
    assert int(cache.k_codes[:, :, :5].sum()) == 0 and int(cache.v_meta[:, :, 6].abs().sum()) == 0


def _golden_pins():
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "rounding_pins.json")
    with open(path, encoding="utf-8") as f:
        return json.load(f)


def test_quantize_dequant_hit_the_golden_rounding_pins():
    """The hand-derived groups that separate rint from rounding half away,
    the IEEE quotient from a reciprocal product, and one fused multiply-add
    from a separate multiply and add: the kernels' codes and dequantised
    values equal the fixture's expected values directly (no oracle)."""
    pins = _golden_pins()
    names = ["ties_half_even", "quotient_tie", "quotient_near_tie"]
    x = np.zeros((16, 64), np.float16)      # the GEMM takes N in multiples of 16
    x[:4] = np.array([pins[n]["x"] for n in names] + [pins["fma_dequant"]["x"]], np.float16)
    q = fg.fg_quantize_g4(torch.from_numpy(x).to(DEV))
    deq = fg.fg_dequant_g4(q)
    # the fused GEMM dequantisation: X = I returns the dequantised weights
    eye = torch.eye(64, dtype=torch.float16, device=DEV)
    y = fg.fg_dequant_gemm_g4(eye, q)
    torch.cuda.synchronize()
    codes = to_np(q.codes)
    got = np.stack([codes & 0xF, codes >> 4], -1).reshape(16, 64)
    for i, n in enumerate(names):
        assert np.array_equal(got[i], np.array(pins[n]["codes"])), n
    p = pins["fma_dequant"]
    assert got[3, p["index"]] == p["code"]
    assert int(to_np(deq)[3, p["index"]].view(np.uint16)) == p["dequant_fp16_bits"]
    assert int(to_np(y)[p["index"], 3].view(np.uint16)) == p["dequant_fp16_bits"]
