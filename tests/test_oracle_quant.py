"""Pins for the oracle's binary16 conversion, 4-bit quantiser and dequantiser.

The quantiser follows the group-wise asymmetric min/max scheme of "FlexGen
完全拆解" (section "权重压缩与 KV Cache 压缩"): per group of 64 values,
q = round((x - min)/(max - min) * 15) and x^ = min + q/15 * (max - min); two
codes per byte ("bjbfmj.com/news/40234", section 6.3).  These tests check the
oracle against facts that do not reuse its arithmetic: numpy's binary16,
exact rationals, nearest-level brute force, reconstruction bounds and special
groups.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- binary16

def test_h2f_exhaustive_against_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle.h2f_array(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2h_against_numpy_rne():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(200_000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(50_000) * 1e-5).astype(np.float32),       # subnormals
        (rng.standard_normal(50_000) * 3e4).astype(np.float32),        # near overflow
        rng.integers(0, 1 << 32, 200_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    # exact halfway points between neighbouring fp16 values (ties to even)
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    parts.append(((lo + hi) / 2).astype(np.float32))
    parts.append(np.array([65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -25,
                           2.0 ** -24, 3 * 2.0 ** -26, 0.0, -0.0, np.inf, -np.inf],
                          np.float32))
    x = np.concatenate(parts)
    x = x[~np.isnan(x)]
    ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f2h_array(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


# ---------------------------------------------------------------- helpers

def unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def groups_f64(x):
    return x.astype(np.float64).reshape(x.shape[0], -1, 64)


# ---------------------------------------------------------------- worked group

def test_ramp_group_exact_rational():
    """x_i = i for i = 0..63: min 0, max 63, scale = 63/15 = 4.2 (fp32), and
    code_i = nearest integer to i*15/63 = 5i/21.  5i/21 is never within 1/42
    of a half-integer, so fp32 rounding cannot move it across a tie."""
    x = np.arange(64, dtype=np.float16)[None, :]
    codes, meta = oracle.quantize_g4(x)
    assert meta[0, 0, 0] == 0.0
    assert meta[0, 0, 1] == np.float32(63) / np.float32(15)
    want = []
    for i in range(64):
        f = Fraction(5 * i, 21)
        want.append(int(f + Fraction(1, 2)))    # floor(f + 1/2): no exact ties
    assert unpack(codes)[0].tolist() == want
    # nibble order: element 2j low nibble, element 2j+1 high nibble
    for j in range(32):
        assert codes[0, j] == want[2 * j] | (want[2 * j + 1] << 4)


def test_packing_fixture():
    """Hand-made group whose 64 codes are known without arithmetic: values
    0 and 15 only (min 0, max 15, scale 1), alternating in blocks."""
    pattern = [(i // 3) % 2 * 15 for i in range(64)]
    x = np.array(pattern, np.float16)[None, :]
    codes, meta = oracle.quantize_g4(x)
    assert meta[0, 0].tolist() == [0.0, 1.0]
    golden = open(__file__.replace("test_oracle_quant.py", "golden/pack_0_15_blocks3.txt")).read().split()
    assert [int(b, 16) for b in golden] == codes[0].tolist()


# ---------------------------------------------------------------- invariants

def _random_groups():
    rng = np.random.default_rng(1)
    g = [
        rng.standard_normal((64, 512)) * 0.02,                  # weight-like
        rng.standard_normal((64, 512)),                         # activation-like
        rng.uniform(-5, -1, (32, 512)),                         # negative only
        rng.standard_normal((32, 512)) * 1e-3 + 7.0,            # offset, narrow
    ]
    out = rng.standard_normal((32, 512)) * 0.1                  # one outlier per group
    out[:, ::64] = 40.0
    g.append(out)
    ext = rng.uniform(-65504, 65504, (8, 512))                  # full fp16 range
    ext[:, ::64] = 65504.0
    ext[:, 1::64] = -65504.0
    g.append(ext)
    g.append(rng.standard_normal((16, 512)) * 1e-6)              # subnormal fp16 values
    return [a.astype(np.float16) for a in g]


@pytest.mark.parametrize("idx", range(7))
def test_codes_are_nearest_level(idx):
    """Each code names the grid level m + c*scale (c in 0..15) nearest to x,
    judged in fp64 with the stored fp32 (m, scale); near-ties may go either
    way, by at most fp32 rounding of (x - m)/scale."""
    x = _random_groups()[idx]
    codes, meta = oracle.quantize_g4(x)
    q = unpack(codes).reshape(x.shape[0], -1, 64).astype(np.float64)
    xg = groups_f64(x)
    m = meta[..., 0].astype(np.float64)[..., None]
    s = meta[..., 1].astype(np.float64)[..., None]
    levels = m[..., None] + np.arange(16, dtype=np.float64) * s[..., None]
    dist = np.abs(xg[..., None] - levels)
    best = dist.min(-1)
    chosen = np.take_along_axis(dist, q.astype(np.int64)[..., None], -1)[..., 0]
    slack = s * 2.0 ** -20 + np.abs(xg) * 2.0 ** -22
    assert np.all(chosen <= best + slack)


@pytest.mark.parametrize("idx", range(7))
def test_min_max_codes_and_reconstruction_bound(idx):
    x = _random_groups()[idx]
    codes, meta = oracle.quantize_g4(x)
    q = unpack(codes).reshape(x.shape[0], -1, 64)
    xg = groups_f64(x)
    s = meta[..., 1].astype(np.float64)
    assert np.all(meta[..., 0] == xg.min(-1))                    # stored min is exact
    amin = xg.argmin(-1)
    amax = xg.argmax(-1)
    pos = s > 0
    assert np.all(np.take_along_axis(q, amin[..., None], -1)[..., 0] == 0)
    assert np.all(np.take_along_axis(q, amax[..., None], -1)[..., 0][pos] == 15)
    assert q.max() <= 15
    xh = groups_f64(oracle.dequant_g4(codes, meta))
    # |x - x^| <= scale/2, plus the fp16 rounding of x^ (half an ulp at |x^|)
    # and the fp32 rounding of scale.
    ulp16 = np.maximum(np.abs(xh), 2.0 ** -14) * 2.0 ** -11
    bound = s[..., None] / 2 * (1 + 2.0 ** -20) + ulp16
    assert np.all(np.abs(xg - xh) <= bound)


def test_signed_zero_min_is_order_independent():
    """min/max use the IEEE total order (-0 below +0): a group of zeros of
    both signs stores min = -0 and max = +0 wherever the -0 sits."""
    for where in (0, 17, 63):
        x = np.zeros((1, 64), np.float16)
        x[0, where] = np.float16(-0.0)
        codes, meta = oracle.quantize_g4(x)
        assert np.signbit(meta[0, 0, 0]) and meta[0, 0, 1] == 0.0
        assert np.all(codes == 0)


def test_monotone_codes():
    rng = np.random.default_rng(2)
    x = np.sort(rng.standard_normal((16, 64 * 8)).reshape(16, 8, 64), -1).reshape(16, -1)
    codes, _ = oracle.quantize_g4(x.astype(np.float16))
    q = unpack(codes).reshape(16, 8, 64)
    assert np.all(np.diff(q.astype(np.int64), axis=-1) >= 0)


def test_constant_groups_exact():
    vals = np.array([0.0, 1.0, -3.5, 65504.0, -65504.0, 2.0 ** -24, 0.1], np.float16)
    x = np.repeat(vals, 64)[None, :].astype(np.float16)
    codes, meta = oracle.quantize_g4(x)
    assert np.all(meta[..., 1] == 0.0)
    assert np.all(codes == 0)
    assert np.array_equal(oracle.dequant_g4(codes, meta).view(np.uint16), x.view(np.uint16))


def test_two_valued_groups():
    """Groups holding only two distinct values a < b: codes are 0 for a and
    15 for b; a reconstructs exactly, b within one fp16 ulp plus the fp32
    rounding of scale = (b - a)/15 carried through 15 * scale (relative to
    the range b - a, not to b)."""
    rng = np.random.default_rng(3)
    finite = np.arange(0, 0x7BFF, dtype=np.uint16).view(np.float16)
    allv = np.concatenate([finite, -finite])
    pairs = rng.choice(allv, size=(4000, 2))
    pairs = pairs[pairs[:, 0] != pairs[:, 1]]
    a = np.minimum(pairs[:, 0], pairs[:, 1])
    b = np.maximum(pairs[:, 0], pairs[:, 1])
    sel = rng.integers(0, 2, (a.size, 64)).astype(bool)
    sel[:, 0], sel[:, 1] = False, True
    x = np.where(sel, b[:, None], a[:, None]).astype(np.float16)
    codes, meta = oracle.quantize_g4(x)
    q = unpack(codes)
    assert np.array_equal(q, np.where(sel, 15, 0))
    xh = oracle.dequant_g4(codes, meta)
    assert np.array_equal(xh[:, 0].view(np.uint16), a.view(np.uint16))
    bh = xh[:, 1].astype(np.float64)
    b64, a64 = b.astype(np.float64), a.astype(np.float64)
    ulp = np.maximum(np.abs(b64), 2.0 ** -14) * 2.0 ** -10
    fp32_err = (b64 - a64) * 2.0 ** -21
    assert np.all(np.abs(bh - b64) <= ulp + fp32_err)
    # when the range is within one binade of b the fp32 part is negligible
    tight = (b64 - a64) <= np.abs(b64)
    assert np.all(np.abs(bh - b64)[tight] <= ulp[tight])


def test_agrees_with_pages_formula_away_from_ties():
    """The pages write q = round((x - min)/(max - min) * (2^b - 1)).  The
    oracle divides by the fp32 scale instead; the two agree except where
    the exact value sits within fp32 rounding of a half-integer."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((256, 64 * 4)) * 0.02).astype(np.float16)
    codes, _ = oracle.quantize_g4(x)
    q = unpack(codes).reshape(256, 4, 64)
    xg = groups_f64(x)
    mn = xg.min(-1, keepdims=True)
    mx = xg.max(-1, keepdims=True)
    t = (xg - mn) / (mx - mn) * 15.0
    near_tie = np.abs(t - np.floor(t) - 0.5) < 1e-5
    pages = np.floor(t + 0.5)
    assert np.all((q == pages) | near_tie)
    assert near_tie.mean() < 1e-3


def test_dequant_closed_form():
    """x^ = fp16(min + q*scale): within half an fp16 ulp of the exact value."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)).astype(np.float16)
    codes, meta = oracle.quantize_g4(x)
    xh = oracle.dequant_g4(codes, meta).astype(np.float64).reshape(64, 4, 64)
    q = unpack(codes).reshape(64, 4, 64).astype(np.float64)
    exact = meta[..., 0:1].astype(np.float64) + q * meta[..., 1:2].astype(np.float64)
    half_ulp = np.maximum(np.abs(exact), 2.0 ** -14) * 2.0 ** -11
    assert np.all(np.abs(xh - exact) <= half_ulp * (1 + 1e-6))
