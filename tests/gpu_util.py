"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

DEV = "cuda:0"


def to_np(t):
    return t.detach().cpu().numpy()


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))


def unpack_codes(codes):
    codes = np.asarray(codes)
    return np.stack([codes & 0xF, codes >> 4], -1).reshape(*codes.shape[:-1], -1)


def gemm_bound(x, codes, meta, extra_abs=0.0):
    """Per-element bound |Y_gpu - Y_oracle| for the 4-bit linear layer.

    Both sides multiply by the same dequantised weights w^ = fp16(fma(q, s,
    m)) (the GPU's fused dequantisation is bit-exact with the oracle's), and
    fp16 x fp16 products are exact in fp32, so only the fp32 summation orders
    differ: at most K * 2^-23 of the absolute dot product sum |x| |w^| between
    the two (each side <= K/2 * 2^-23).  Callers add one fp16 ulp of Y for the
    final rounding."""
    q = unpack_codes(codes).astype(np.float64)
    N, K = q.shape
    m = np.repeat(meta[..., 0].astype(np.float64), 64, axis=1)
    s = np.repeat(meta[..., 1].astype(np.float64), 64, axis=1)
    wmag = np.abs(m + q * s) * (1.0 + 2.0 ** -10)   # >= |w^| (one fp16 rounding)
    xa = np.abs(x.astype(np.float64))
    return K * 2.0 ** -23 * (xa @ wmag.T) + extra_abs


def ulp16(y):
    y = np.abs(np.asarray(y, np.float64))
    return np.maximum(y, 2.0 ** -14) * 2.0 ** -10
