"""CPU oracle for the 4-bit group-quantised OPT decoder hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the product library.  It
shares no code with the CUDA path; the C arithmetic lives in ``fg_oracle.c``
and is compiled here with gcc (``-O2 -ffp-contract=off``, no fast-math).

Arrays are numpy: fp16 tensors are passed as ``np.float16`` (bit patterns are
what the C side reads), codes as ``np.uint8``, metadata as ``np.float32``.

Parity status of each function (what pins it, in ``tests/test_oracle_*.py``):
  quantize_g4 / dequant_g4 .. pinned (nearest-level brute force, exact rational
                               worked group, reconstruction bound, constant and
                               two-valued groups, nibble order fixture; exact
                               ties -> even codes, IEEE quotient vs reciprocal
                               product, one fused multiply-add in dequant)
  linear_* .................. pinned (fp64 matmul within the fp32-accumulation
                               bound; permutation-matrix exactness)
  layernorm ................. pinned (fp64 closed form; zero-mean/unit-variance)
  prefill_attn / decode_attn  pinned (fp64 softmax via scipy on tiny shapes;
                               equal keys -> mean of V; one row -> v itself;
                               causality; key-order invariance)
  model / block orders ...... pinned only through the pieces above plus the
                               row-by-row == zig-zag identity: the pages print
                               no end-to-end output values (parity unpinned
                               beyond those properties).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 64


def build(force: bool = False) -> str:
    """Compile fg_oracle.c into oracle/_build/liboracle.so (OpenMP if gcc has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-lm"]
    tmp = _LIB + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base[:-1] + ["-fopenmp", "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I32 = ctypes.c_int32
            F = ctypes.c_float
            sig = {
                "or_h2f": ([ctypes.c_uint16], F),
                "or_h2f_array": ([P, P, I64], None),
                "or_f2h_array": ([P, P, I64], None),
                "or_f2h": ([F], ctypes.c_uint16),
                "or_num_threads": ([], ctypes.c_int),
                "or_set_num_threads": ([ctypes.c_int], None),
                "or_quantize_g4": ([P, I64, I64, P, P], None),
                "or_dequant_g4": ([P, P, I64, I64, P], None),
                "or_linear_f16": ([P, I64, I64, P, I64, P, P, ctypes.c_int, P], None),
                "or_linear_f16_f32out": ([P, I64, I64, P, I64, P], None),
                "or_linear_g4": ([P, I64, I64, P, P, I64, P, P, ctypes.c_int, P], None),
                "or_layernorm": ([P, I64, I64, P, P, F, P], None),
                "or_embed": ([P, P, I64, P, P, I64, P], None),
                "or_kv_store_prefill": ([P, I32, I32, P, P, P, P, I32, I32, I32], None),
                "or_prefill_attn": ([P, I32, I32, I32, I32, P, P], None),
                "or_decode_attn_g4": ([P, I64, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P], None),
                "or_decode_attn_topk_g4": ([P, I64, P, P, P, P, I32, I32, I32, I32, I32, I32, P,
                                            I32, P, P, P], None),
                "or_topk_count": ([I64, I32], I32),
                "or_kv_store_prefill_f16": ([P, I32, I32, P, P, I32, I32, I32], None),
                "or_decode_attn_f16": ([P, I64, P, P, I32, I32, I32, I32, I32, I32, P, P], None),
                "or_argmax": ([P, I64, I64, P], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return _load().or_num_threads()


def set_num_threads(n: int) -> None:
    _load().or_set_num_threads(int(n))


# --------------------------------------------------------------------------
# binary16 conversion (exposed so the tests can pin it against numpy)
# --------------------------------------------------------------------------

def h2f(bits: int) -> float:
    return _load().or_h2f(int(bits))


def f2h(x: float) -> int:
    return _load().or_f2h(float(x))


def h2f_array(bits):
    """uint16 bit patterns -> fp32 values."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().or_h2f_array(_p(bits), _p(out), bits.size)
    return out


def f2h_array(x):
    """fp32 values -> uint16 binary16 bit patterns (round to nearest even)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().or_f2h_array(_p(x), _p(out), x.size)
    return out


# --------------------------------------------------------------------------
# group-wise 4-bit quantisation
# --------------------------------------------------------------------------

def quantize_g4(x):
    """x: fp16 [rows][cols], cols % 64 == 0 -> (codes u8 [rows][cols/2],
    meta f32 [rows][cols/64][2] = (min, scale))."""
    x = _c(x, np.float16)
    rows, cols = x.shape
    assert cols % GROUP == 0
    assert np.all(np.isfinite(x)), "non-finite input is outside the contract"
    codes = np.empty((rows, cols // 2), np.uint8)
    meta = np.empty((rows, cols // GROUP, 2), np.float32)
    _load().or_quantize_g4(_p(x), rows, cols, _p(codes), _p(meta))
    return codes, meta


def dequant_g4(codes, meta, cols=None):
    codes = _c(codes, np.uint8)
    meta = _c(meta, np.float32)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2 if cols is None else cols
    out = np.empty((rows, cols), np.float16)
    _load().or_dequant_g4(_p(codes), _p(meta), rows, cols, _p(out))
    return out


# --------------------------------------------------------------------------
# linear layers, LayerNorm, embedding
# --------------------------------------------------------------------------

def linear_f16(x, w, bias=None, residual=None, act=0):
    x = _c(x, np.float16)
    w = _c(w, np.float16)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K
    b = None if bias is None else _c(bias, np.float16)
    r = None if residual is None else _c(residual, np.float16)
    y = np.empty((M, N), np.float16)
    _load().or_linear_f16(_p(x), M, K, _p(w), N, _p(b), _p(r), int(act), _p(y))
    return y


def linear_f16_f32out(x, w):
    x = _c(x, np.float16)
    w = _c(w, np.float16)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), np.float32)
    _load().or_linear_f16_f32out(_p(x), M, K, _p(w), N, _p(y))
    return y


def linear_g4(x, codes, meta, bias=None, residual=None, act=0):
    x = _c(x, np.float16)
    codes = _c(codes, np.uint8)
    meta = _c(meta, np.float32)
    M, K = x.shape
    N = codes.shape[0]
    assert codes.shape[1] * 2 == K
    b = None if bias is None else _c(bias, np.float16)
    r = None if residual is None else _c(residual, np.float16)
    y = np.empty((M, N), np.float16)
    _load().or_linear_g4(_p(x), M, K, _p(codes), _p(meta), N, _p(b), _p(r),
                         int(act), _p(y))
    return y


def layernorm(x, gamma, beta, eps=1e-5):
    x = _c(x, np.float16)
    rows, cols = x.shape
    y = np.empty_like(x)
    _load().or_layernorm(_p(x), rows, cols, _p(_c(gamma, np.float16)),
                         _p(_c(beta, np.float16)), float(eps), _p(y))
    return y


def embed(ids, pos, e_tok, e_pos):
    ids = _c(ids, np.int32).reshape(-1)
    pos = _c(pos, np.int32).reshape(-1)
    e_tok = _c(e_tok, np.float16)
    e_pos = _c(e_pos, np.float16)
    h1 = e_tok.shape[1]
    y = np.empty((ids.size, h1), np.float16)
    _load().or_embed(_p(ids), _p(pos), ids.size, _p(e_tok), _p(e_pos), h1, _p(y))
    return y


# --------------------------------------------------------------------------
# 4-bit KV cache and attention
# --------------------------------------------------------------------------

class KVCache:
    """One layer's 4-bit K and V cache: codes [B][H][cap][d/2] u8 and
    meta [B][H][cap][d/64][2] f32 for each of K and V."""

    def __init__(self, B, H, d, cap):
        self.B, self.H, self.d, self.cap = B, H, d, cap
        self.k_codes = np.zeros((B, H, cap, d // 2), np.uint8)
        self.v_codes = np.zeros((B, H, cap, d // 2), np.uint8)
        self.k_meta = np.zeros((B, H, cap, d // GROUP, 2), np.float32)
        self.v_meta = np.zeros((B, H, cap, d // GROUP, 2), np.float32)

    def view(self, b0, b1):
        """Sequences [b0, b1) as a cache sharing this one's storage."""
        v = KVCache.__new__(KVCache)
        v.B, v.H, v.d, v.cap = b1 - b0, self.H, self.d, self.cap
        v.k_codes = self.k_codes[b0:b1]
        v.v_codes = self.v_codes[b0:b1]
        v.k_meta = self.k_meta[b0:b1]
        v.v_meta = self.v_meta[b0:b1]
        return v

    def _ptrs(self):
        for a in (self.k_codes, self.v_codes, self.k_meta, self.v_meta):
            assert a.flags["C_CONTIGUOUS"]
        return (_p(self.k_codes), _p(self.v_codes), _p(self.k_meta),
                _p(self.v_meta))


def kv_store_prefill(qkv, B, s, cache: KVCache):
    qkv = _c(qkv, np.float16)
    assert qkv.shape == (B * s, 3 * cache.H * cache.d)
    kc, vc, km, vm = cache._ptrs()
    _load().or_kv_store_prefill(_p(qkv), B, s, kc, vc, km, vm, cache.H,
                                cache.d, cache.cap)


def _pad(pad, B):
    if pad is None:
        return None
    pad = _c(pad, np.int32).reshape(-1)
    assert pad.size == B
    return pad


def prefill_attn(qkv, B, s, H, d, pad=None):
    """pad: None or [B] left-padding counts (prompt b fills slots pad[b]..s-1)."""
    qkv = _c(qkv, np.float16)
    assert qkv.shape == (B * s, 3 * H * d)
    out = np.empty((B * s, H * d), np.float16)
    pad = _pad(pad, B)
    _load().or_prefill_attn(_p(qkv), B, s, H, d, None if pad is None else _p(pad), _p(out))
    return out


def decode_attn_g4(qkv, cache: KVCache, pos, append=True, pad=None):
    """qkv: [B][>=3*h1] fp16 (row stride = qkv.shape[1]); pad: None or [B]
    left-padding counts (sequence b attends slots pad[b]..pos)."""
    qkv = _c(qkv, np.float16)
    B = qkv.shape[0]
    assert B == cache.B and 0 <= pos < cache.cap
    out = np.empty((B, cache.H * cache.d), np.float16)
    kc, vc, km, vm = cache._ptrs()
    pad = _pad(pad, B)
    _load().or_decode_attn_g4(_p(qkv), qkv.shape[1], kc, vc, km, vm, cache.B,
                              cache.H, cache.d, cache.cap, int(pos),
                              1 if append else 0, None if pad is None else _p(pad), _p(out))
    return out


class KVCache16:
    """One layer's uncompressed K and V cache: fp16 [B][H][cap][d] each."""

    def __init__(self, B, H, d, cap):
        self.B, self.H, self.d, self.cap = B, H, d, cap
        self.k = np.zeros((B, H, cap, d), np.float16)
        self.v = np.zeros((B, H, cap, d), np.float16)

    def view(self, b0, b1):
        """Sequences [b0, b1) as a cache sharing this one's storage."""
        v = KVCache16.__new__(KVCache16)
        v.B, v.H, v.d, v.cap = b1 - b0, self.H, self.d, self.cap
        v.k, v.v = self.k[b0:b1], self.v[b0:b1]
        return v


def kv_store_prefill_f16(qkv, B, s, cache: KVCache16):
    qkv = _c(qkv, np.float16)
    assert qkv.shape == (B * s, 3 * cache.H * cache.d) and s <= cache.cap
    _load().or_kv_store_prefill_f16(_p(qkv), B, s, _p(cache.k), _p(cache.v), cache.H, cache.d,
                                    cache.cap)


def decode_attn_f16(qkv, cache: KVCache16, pos, append=True, pad=None):
    """Decode attention over the fp16 cache (rows read as stored); qkv
    [B][>=3*h1] fp16, pad None or [B]."""
    qkv = _c(qkv, np.float16)
    B = qkv.shape[0]
    assert B == cache.B and 0 <= pos < cache.cap
    out = np.empty((B, cache.H * cache.d), np.float16)
    pad = _pad(pad, B)
    _load().or_decode_attn_f16(_p(qkv), qkv.shape[1], _p(cache.k), _p(cache.v), cache.B, cache.H,
                               cache.d, cache.cap, int(pos), 1 if append else 0,
                               None if pad is None else _p(pad), _p(out))
    return out


def topk_count(n, keep_pct):
    """Rows kept out of n by top-K sparse attention at keep_pct percent."""
    return int(_load().or_topk_count(int(n), int(keep_pct)))


def decode_attn_topk_g4(qkv, cache: KVCache, pos, keep_pct, append=True, pad=None, sel=None):
    """Top-K sparse decode attention (full softmax, only the keep_pct percent
    highest-scoring rows' V summed).  sel: None, or [B][H][kmax] int32 kept
    slots to use instead of the oracle's own choice.  Returns (out, sel_used)
    with sel_used [B][H][kmax] (-1 past a sequence's own count)."""
    qkv = _c(qkv, np.float16)
    B = qkv.shape[0]
    assert B == cache.B and 0 <= pos < cache.cap and 1 <= keep_pct <= 100
    H = cache.H
    kmax = topk_count(pos + 1, keep_pct)
    out = np.empty((B, H * cache.d), np.float16)
    sel_out = np.empty((B, H, kmax), np.int32)
    if sel is not None:
        sel = _c(sel, np.int32)
        assert sel.shape == (B, H, kmax)
    kc, vc, km, vm = cache._ptrs()
    pad = _pad(pad, B)
    _load().or_decode_attn_topk_g4(_p(qkv), qkv.shape[1], kc, vc, km, vm, cache.B, H, cache.d,
                                   cache.cap, int(pos), 1 if append else 0,
                                   None if pad is None else _p(pad), int(keep_pct),
                                   None if sel is None else _p(sel), _p(sel_out), _p(out))
    return out, sel_out


def argmax(logits):
    """Greedy token per row of fp32 logits [B][V] (lowest index among ties)."""
    logits = _c(logits, np.float32)
    B, V = logits.shape
    out = np.empty(B, np.int32)
    _load().or_argmax(_p(logits), B, V, _p(out))
    return out


from .model import (OracleLayer, OracleModel, layer_step, quantize_layer,  # noqa: E402
                    size_m_kv, size_m_w, size_q4)
