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
    """Per-element bound |Y_gpu - Y_oracle| for the 4-bit linear layer:
    the GPU dequantises with one fused fp16 multiply-add on fp16-rounded
    (min, scale), the oracle with one fp32 fused multiply-add rounded to fp16;
    each weight then differs by at most 2^-10 (|m| + q*s + |w^|).  Both
    accumulate fp16 x fp16 products in fp32 (orders differ: K * 2^-23 of the
    absolute dot product), then one fp16 rounding of Y (1 ulp between two
    roundings)."""
    q = unpack_codes(codes).astype(np.float64)
    N, K = q.shape
    m = np.repeat(np.abs(meta[..., 0].astype(np.float64)), 64, axis=1)
    s = np.repeat(np.abs(meta[..., 1].astype(np.float64)), 64, axis=1)
    wmag = m + q * s
    xa = np.abs(x.astype(np.float64))
    dot_abs = xa @ wmag.T
    return 2.0 ** -9 * dot_abs + K * 2.0 ** -23 * dot_abs + extra_abs


def ulp16(y):
    y = np.abs(np.asarray(y, np.float64))
    return np.maximum(y, 2.0 ** -14) * 2.0 ** -10
