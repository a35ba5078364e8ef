"""Pins of the quantiser's rounding and division and of the dequantiser's
single-rounding multiply-add, against hand-derived groups.

The scheme is the group-wise 4-bit min/max quantisation of "FlexGen 完全拆解"
(section 权重压缩与 KV Cache 压缩), in this library's fixed arithmetic:
scale = (M - m)/15 by IEEE fp32 division, code = clamp(rint((x - m)/scale),
0, 15) with ties to even, dequantised value fp16(fma(code, scale, m)).

The groups in ``golden/rounding_pins.json`` (written by
``golden/make_rounding_pins.py`` from exact rationals and numpy's IEEE float32
division, never from the oracle) are chosen so that each plausible near-miss
-- rounding half away from zero, multiplying by the reciprocal of the scale,
or a separately rounded multiply then add -- gives a different result.  The
last test proves it: it plants each near-miss in a copy of the oracle's C
source and checks that a pin fails.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
PINS = json.load(open(os.path.join(HERE, "golden", "rounding_pins.json"), encoding="utf-8"))


def _unpack(codes):
    codes = np.asarray(codes)
    return np.stack([codes & 0xF, codes >> 4], -1).reshape(-1)


def _quantize_with(quantize, x):
    codes, meta = quantize(np.array([x], np.float16))
    return _unpack(codes[0]), meta


def _check_quant_pins(quantize):
    """Returns the names of the quantiser pins the function fails."""
    bad = []
    for name in ("ties_half_even", "quotient_tie", "quotient_near_tie"):
        pin = PINS[name]
        got, _ = _quantize_with(quantize, pin["x"])
        if not np.array_equal(got, np.array(pin["codes"])):
            bad.append(name)
    return bad


def _check_dequant_pin(quantize, dequant):
    pin = PINS["fma_dequant"]
    codes, meta = quantize(np.array([pin["x"]], np.float16))
    out = dequant(codes, meta)
    return int(out[0, pin["index"]].view(np.uint16)) == pin["dequant_fp16_bits"]


def test_ties_round_half_to_even():
    pin = PINS["ties_half_even"]
    got, meta = _quantize_with(oracle.quantize_g4, pin["x"])
    assert meta[0, 0, 0] == 0.0 and meta[0, 0, 1] == 2.0
    assert list(got[2:17]) == [0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14, 14]
    assert np.array_equal(got, np.array(pin["codes"]))


@pytest.mark.parametrize("name", ["quotient_tie", "quotient_near_tie"])
def test_code_uses_the_ieee_quotient(name):
    pin = PINS[name]
    got, meta = _quantize_with(oracle.quantize_g4, pin["x"])
    assert meta[0, 0, 1] == np.float32(pin["scale"])
    assert got[pin["index"]] == pin["codes"][pin["index"]]
    assert np.array_equal(got, np.array(pin["codes"]))


def test_dequant_is_one_fused_rounding():
    pin = PINS["fma_dequant"]
    codes, meta = oracle.quantize_g4(np.array([pin["x"]], np.float16))
    assert _unpack(codes[0])[pin["index"]] == pin["code"]
    assert meta[0, 0, 0] == np.float32(pin["min"]) and meta[0, 0, 1] == np.float32(pin["scale"])
    assert _check_dequant_pin(oracle.quantize_g4, oracle.dequant_g4)


# ------------------------------------------------------------ planted mistakes

_MUTANTS = {
    "round_half_away": ("float r = rintf(t);", "float r = roundf(t);"),
    "reciprocal_product": ("float t = (v[i] - mn) / scale;",
                           "float t = (v[i] - mn) * (1.0f / scale);"),
    "split_multiply_add": ("return or_f2h(fmaf((float)q, scale, mn));",
                           "return or_f2h((float)q * scale + mn);"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fg_oracle.c")).read()
    old, new = _MUTANTS[name]
    assert src.count(old) == 1, "the oracle no longer contains: " + old
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(old, new))
    lib = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", str(path), "-o", str(lib), "-lm"], check=True, capture_output=True)
    so = ctypes.CDLL(str(lib))
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    so.or_quantize_g4.argtypes = [P, I64, I64, P, P]
    so.or_dequant_g4.argtypes = [P, P, I64, I64, P]

    def quantize(x):
        x = np.ascontiguousarray(x, np.float16)
        rows, cols = x.shape
        codes = np.empty((rows, cols // 2), np.uint8)
        meta = np.empty((rows, cols // 64, 2), np.float32)
        so.or_quantize_g4(x.ctypes.data, rows, cols, codes.ctypes.data, meta.ctypes.data)
        return codes, meta

    def dequant(codes, meta):
        codes = np.ascontiguousarray(codes, np.uint8)
        meta = np.ascontiguousarray(meta, np.float32)
        out = np.empty((codes.shape[0], codes.shape[1] * 2), np.float16)
        so.or_dequant_g4(codes.ctypes.data, meta.ctypes.data, codes.shape[0],
                         codes.shape[1] * 2, out.ctypes.data)
        return out

    return quantize, dequant


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistakes_fail_a_pin(tmp_path, name):
    quantize, dequant = _build_mutant(tmp_path, name)
    failed = _check_quant_pins(quantize)
    fma_ok = _check_dequant_pin(quantize, dequant)
    if name == "split_multiply_add":
        assert not fma_ok and failed == []
    else:
        assert failed and fma_ok
