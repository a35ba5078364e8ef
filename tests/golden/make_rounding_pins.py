"""Writes rounding_pins.json: groups that separate the quantiser's and the
dequantiser's fixed arithmetic from plausible near-misses.

The arithmetic being pinned is the group-wise 4-bit scheme of "FlexGen
完全拆解" (section 权重压缩与 KV Cache 压缩) in the fixed form this library
adopts: scale = (M - m) / 15 by IEEE fp32 division, code = clamp(rint((x -
m) / scale), 0, 15) with round-half-to-even, and the dequantised value
fp16(fma(code, scale, m)) with a single-rounding fused multiply-add.

Nothing here calls the oracle or the CUDA library.  Expected values come from
exact rational arithmetic (fractions.Fraction) and numpy's IEEE float32
division; the candidate groups were found by searching seeded random groups
with the same two tools.  Run from the repository root:
    python tests/golden/make_rounding_pins.py
"""
import json
import os
from fractions import Fraction

import numpy as np

F32 = np.float32


def f32_round(fr: Fraction) -> np.float32:
    """Round an exact rational to binary32 (nearest, ties to even) through
    binary64: valid when fr is exactly a binary64 value, which is checked."""
    d = float(fr)
    assert Fraction(d) == fr, "not exact in binary64"
    return F32(d)


def half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def ties_group():
    """min 0, max 30, so scale = 30/15 = 2 exactly; every odd integer x then
    has (x - 0)/2 = k + 1/2 exactly and rounds to the even neighbour."""
    odd = list(range(1, 30, 2))                    # 15 values, exact ties
    even = list(range(0, 31, 2))                   # 16 values, exact integers
    x = [0, 30] + odd + even
    x += [7, 9, 11, 13] * ((64 - len(x)) // 4)
    x += [0] * (64 - len(x))
    assert len(x) == 64
    codes = [half_even(Fraction(v, 2)) for v in x]
    return {"x": [float(v) for v in x], "codes": codes,
            "why": "scale is exactly 2, so every odd x sits exactly halfway between two "
                   "codes: rint (half to even) gives 0,2,2,4,4,...; rounding half away "
                   "from zero would give 1,2,3,4,5,..."}


def quotient_group(M: float, x: float):
    """{0, M, x, ...}: min 0, max M, scale = fl(M / 15).  The IEEE quotient
    x / scale and the product x * fl(1 / scale) round to different codes."""
    xs = [0.0, M, x] + [0.0, M] * 30 + [0.0]
    h = np.array(xs, np.float16)
    assert np.array_equal(h.astype(np.float64), np.array(xs)), "values must be fp16-exact"
    scale = F32(M) / F32(15)                        # IEEE division (numpy float32)
    q_ieee = F32(x) / scale
    q_recip = F32(x) * (F32(1) / scale)
    code = int(np.clip(np.rint(q_ieee), 0, 15))
    code_recip = int(np.clip(np.rint(q_recip), 0, 15))
    assert code != code_recip
    codes = [0, 15, code] + [0, 15] * 30 + [0]
    return {"x": xs, "codes": codes, "index": 2, "scale": float(scale),
            "ieee_quotient": float(q_ieee), "reciprocal_product": float(q_recip),
            "why": "IEEE quotient %r -> code %d; x * (1/scale) = %r -> code %d"
                   % (float(q_ieee), code, float(q_recip), code_recip)}


def fma_group():
    """A seeded N(0, 30) fp16 group in which one element's single-rounding
    fma(code, scale, min) and the separately rounded code*scale + min land on
    different fp16 values."""
    rng = np.random.default_rng(7)
    for _ in range(1000):
        x = (rng.standard_normal(64) * rng.choice([0.02, 1.0, 30.0])).astype(np.float16)
        v = x.astype(np.float32)
        mn, mx = v.min(), v.max()
        scale = F32(mx - mn) / F32(15)
        if scale == 0:
            continue
        q = np.clip(np.rint((v - mn) / scale), 0, 15)
        for i in range(64):
            exact = Fraction(int(q[i])) * Fraction(float(scale)) + Fraction(float(mn))
            try:
                fused = f32_round(exact)
            except AssertionError:
                continue
            split = F32(F32(F32(q[i]) * scale) + mn)
            a, b = np.float16(fused), np.float16(split)
            if a.view(np.uint16) != b.view(np.uint16):
                return {"x": [float(t) for t in x.astype(np.float64)], "index": i,
                        "code": int(q[i]), "min": float(mn), "scale": float(scale),
                        "dequant_fp16_bits": int(a.view(np.uint16)),
                        "split_fp16_bits": int(b.view(np.uint16)),
                        "why": "fp16(fma(%d, scale, min)) = %r; fp16(code*scale + min) with two "
                               "roundings = %r" % (int(q[i]), float(a), float(b))}
    raise RuntimeError("no group found")


def main():
    out = {
        "source": "FlexGen 完全拆解, section 权重压缩与 KV Cache 压缩 (q(x) and its inverse), "
                  "in this library's fixed arithmetic: IEEE fp32 divide, rint (half to even), "
                  "single-rounding fma then fp16",
        "ties_half_even": ties_group(),
        # an exact tie under IEEE division that the reciprocal pushes past the half
        "quotient_tie": quotient_group(1.0205078125, 0.30615234375),
        # no tie under IEEE division; the reciprocal product lands exactly on one
        "quotient_near_tie": quotient_group(1.0888671875, 0.54443359375),
        "fma_dequant": fma_group(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rounding_pins.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, ensure_ascii=False)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
