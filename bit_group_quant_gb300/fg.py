"""ctypes binding of libfg (include/fg.h): the same names as the C ABI,
argument marshalling only.  Tensors are torch CUDA tensors (device memory and
streams come from torch); every step of the computation runs in libfg's CUDA
kernels.  There is no fallback: if libfg.so is missing or fails to load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libfg.so")

FG_OK, FG_ERR_NULL, FG_ERR_SHAPE, FG_ERR_ALIGN, FG_ERR_UNSUPPORTED, FG_ERR_CUDA, \
    FG_ERR_TIMEOUT, FG_ERR_WORKSPACE = range(8)
FG_ORDER_BLOCK, FG_ORDER_BATCHES, FG_ORDER_BATCHES_REV = 0, 1, 2
FG_PHASE_PREFILL, FG_PHASE_DECODE = 0, 1
FG_ACT_NONE, FG_ACT_RELU = 0, 1
FG_KNOB_DROP_ARRIVE, FG_KNOB_WAIT_NS = 1, 2

EXPORTS = (
    "fg_status_str", "fg_last_error", "fg_version", "fg_check", "fg_quantize_g4",
    "fg_dequant_g4", "fg_dequant_gemm_workspace_bytes", "fg_dequant_gemm_g4",
    "fg_gemm_f16_f32out", "fg_layernorm", "fg_embed", "fg_kv_append_g4",
    "fg_decode_attn_g4", "fg_prefill_attn", "fg_layer_workspace_bytes", "fg_layer_step",
    "fg_debug_set", "fg_trace_begin", "fg_trace_end", "fg_dequant_gemm_g4_noalloc",
    "fg_argmax", "fg_decode_attn_topk_g4", "fg_decode_attn_topk_workspace_bytes",
    "fg_topk_count", "fg_kv_store_f16",
    "fg_decode_attn_f16", "fg_layer_step_kv16",
)


class FgError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__("libfg status %d: %s" % (status, detail))
        self.status = status


class c_q4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class c_kv4(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_meta", ctypes.c_void_p), ("v_meta", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d", ctypes.c_int32),
                ("cap", ctypes.c_int32)]


class c_kv16(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("B", ctypes.c_int32),
                ("H", ctypes.c_int32), ("d", ctypes.c_int32), ("cap", ctypes.c_int32)]


class c_policy(ctypes.Structure):
    _fields_ = [("gbs", ctypes.c_int32), ("k", ctypes.c_int32), ("order", ctypes.c_int32),
                ("topk_pct", ctypes.c_int32)]


class c_layer(ctypes.Structure):
    _fields_ = [("qkv", c_q4), ("out", c_q4), ("fc1", c_q4), ("fc2", c_q4),
                ("b_qkv", ctypes.c_void_p), ("b_out", ctypes.c_void_p),
                ("b_fc1", ctypes.c_void_p), ("b_fc2", ctypes.c_void_p),
                ("ln1_g", ctypes.c_void_p), ("ln1_b", ctypes.c_void_p),
                ("ln2_g", ctypes.c_void_p), ("ln2_b", ctypes.c_void_p),
                ("h1", ctypes.c_int32), ("H", ctypes.c_int32), ("h2", ctypes.c_int32),
                ("ln_eps", ctypes.c_float)]


FG_TRACE_GEMM_PREFILL, FG_TRACE_GEMM_DECODE, FG_TRACE_ATTN_DECODE, FG_TRACE_ATTN_PREFILL, \
    FG_TRACE_OTHER = 1, 2, 4, 8, 16
TRACE_CLASSES = ("gemm_prefill", "gemm_decode", "attn_decode", "attn_prefill", "other")


class c_trace_stats(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * 5), ("ms", ctypes.c_double * 5),
                ("flops", ctypes.c_double * 5), ("bytes", ctypes.c_double * 5)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libfg.so and declare every export.  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError("libfg.so is not built (%s); run __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ, F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                              ctypes.c_float)
        st = ctypes.c_int
        sig = {
            "fg_status_str": ([st], ctypes.c_char_p),
            "fg_last_error": ([], ctypes.c_char_p),
            "fg_version": ([], I32),
            "fg_check": ([P], st),
            "fg_quantize_g4": ([P, I64, I64, ctypes.POINTER(c_q4), P], st),
            "fg_dequant_g4": ([ctypes.POINTER(c_q4), P, P], st),
            "fg_dequant_gemm_workspace_bytes": ([I64, I64, I64], SZ),
            "fg_dequant_gemm_g4": ([P, I64, ctypes.POINTER(c_q4), P, P, I32, P, P, SZ, P], st),
            "fg_gemm_f16_f32out": ([P, I64, P, I64, I64, P, P], st),
            "fg_dequant_gemm_g4_noalloc": ([P, I64, ctypes.POINTER(c_q4), P, P, I32, P, P], st),
            "fg_layernorm": ([P, I64, I64, I64, P, P, F, P, P], st),
            "fg_embed": ([P, I64, I32, I32, P, P, I64, P, I64, I32, P, P], st),
            "fg_argmax": ([P, I64, I64, P, P], st),
            "fg_kv_append_g4": ([P, I64, ctypes.POINTER(c_kv4), I32, P], st),
            "fg_decode_attn_g4": ([P, I64, ctypes.POINTER(c_kv4), I32, P, I32, P, P], st),
            "fg_decode_attn_topk_g4": ([P, I64, ctypes.POINTER(c_kv4), I32, P, I32, I32, P, P, P,
                                        SZ, P], st),
            "fg_decode_attn_topk_workspace_bytes": ([I32, I32, I32], SZ),
            "fg_topk_count": ([I32, I32], I32),
            "fg_kv_store_f16": ([P, I64, I32, ctypes.POINTER(c_kv16), I32, P], st),
            "fg_decode_attn_f16": ([P, I64, ctypes.POINTER(c_kv16), I32, P, I32, P, P], st),
            "fg_layer_step_kv16": ([ctypes.POINTER(c_layer), ctypes.POINTER(c_kv16), P, P, I32,
                                    I32, I32, P, c_policy, P, SZ, P], st),
            "fg_prefill_attn": ([P, I32, I32, I32, I32, P, ctypes.POINTER(c_kv4), P, P], st),
            "fg_layer_workspace_bytes": ([ctypes.POINTER(c_layer), I32, I32, I32, I32, c_policy],
                                         SZ),
            "fg_layer_step": ([ctypes.POINTER(c_layer), ctypes.POINTER(c_kv4), P, P, I32, I32,
                               I32, P, c_policy, P, SZ, P], st),
            "fg_debug_set": ([I32, I64], st),
            "fg_trace_begin": ([I32], st),
            "fg_trace_end": ([ctypes.POINTER(c_trace_stats)], st),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ok(status):
    if status != FG_OK:
        lib = load()
        raise FgError(status, lib.fg_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "libfg takes contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _pad(pad, n):
    """None, or a contiguous int32 CUDA tensor of n left-padding counts."""
    if pad is None:
        return None
    assert pad.dtype == torch.int32 and pad.numel() == n, "pad: int32 tensor of one count per sequence"
    return _ptr(pad)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------
# containers mirroring the C structs (they keep the torch tensors alive)
# ---------------------------------------------------------------------------

@dataclass
class Q4:
    """4-bit group-quantised [rows][cols]: codes u8 [rows][cols/2], meta f32
    [rows][cols/64][2] = (min, scale)."""
    codes: torch.Tensor
    meta: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows, cols, device="cuda"):
        return Q4(torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
                  torch.empty((rows, cols // 64, 2), dtype=torch.float32, device=device),
                  rows, cols)

    def c(self):
        return c_q4(_ptr(self.codes), _ptr(self.meta), self.rows, self.cols)

    @property
    def nbytes(self):
        return self.codes.numel() + self.meta.numel() * 4


@dataclass
class KV4:
    """One layer's 4-bit K/V cache: codes [B][H][cap][d/2], meta
    [B][H][cap][d/64][2] for each of K and V."""
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_meta: torch.Tensor
    v_meta: torch.Tensor
    B: int
    H: int
    d: int
    cap: int

    @staticmethod
    def empty(B, H, d, cap, device="cuda", zero=True):
        mk = torch.zeros if zero else torch.empty
        return KV4(mk((B, H, cap, d // 2), dtype=torch.uint8, device=device),
                   mk((B, H, cap, d // 2), dtype=torch.uint8, device=device),
                   mk((B, H, cap, d // 64, 2), dtype=torch.float32, device=device),
                   mk((B, H, cap, d // 64, 2), dtype=torch.float32, device=device),
                   B, H, d, cap)

    def c(self):
        return c_kv4(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_meta),
                     _ptr(self.v_meta), self.B, self.H, self.d, self.cap)

    @property
    def nbytes(self):
        return 2 * (self.k_codes.numel() + self.k_meta.numel() * 4)


@dataclass
class KV16:
    """One layer's uncompressed K/V cache: k, v fp16 [B][H][cap][d]."""
    k: torch.Tensor
    v: torch.Tensor
    B: int
    H: int
    d: int
    cap: int

    @staticmethod
    def empty(B, H, d, cap, device="cuda", zero=True):
        mk = torch.zeros if zero else torch.empty
        return KV16(mk((B, H, cap, d), dtype=torch.float16, device=device),
                    mk((B, H, cap, d), dtype=torch.float16, device=device), B, H, d, cap)

    def c(self):
        return c_kv16(_ptr(self.k), _ptr(self.v), self.B, self.H, self.d, self.cap)

    @property
    def nbytes(self):
        return 2 * self.k.numel() * 2


# ---------------------------------------------------------------------------
# calls (same names as the C ABI)
# ---------------------------------------------------------------------------

def fg_version():
    return load().fg_version()


def fg_check(stream=None):
    _ok(load().fg_check(_stream(stream)))


def fg_debug_set(knob, value):
    _ok(load().fg_debug_set(int(knob), int(value)))


def fg_trace_begin(timed_mask=0):
    _ok(load().fg_trace_begin(int(timed_mask)))


def fg_trace_end() -> dict:
    """Returns {class: {"launches", "ms", "flops", "bytes"}}."""
    st = c_trace_stats()
    _ok(load().fg_trace_end(ctypes.byref(st)))
    return {name: {"launches": int(st.launches[i]), "ms": float(st.ms[i]),
                   "flops": float(st.flops[i]), "bytes": float(st.bytes[i])}
            for i, name in enumerate(TRACE_CLASSES)}


def fg_quantize_g4(x, out: Q4 | None = None, stream=None) -> Q4:
    assert x.dtype == torch.float16 and x.dim() == 2
    rows, cols = x.shape
    if out is None:
        out = Q4.empty(rows, cols, device=x.device)
    q = out.c()
    _ok(load().fg_quantize_g4(_ptr(x), rows, cols, ctypes.byref(q), _stream(stream)))
    return out


def fg_dequant_g4(q: Q4, out=None, stream=None):
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=torch.float16, device=q.codes.device)
    c = q.c()
    _ok(load().fg_dequant_g4(ctypes.byref(c), _ptr(out), _stream(stream)))
    return out


def fg_dequant_gemm_workspace_bytes(M, N, K) -> int:
    return int(load().fg_dequant_gemm_workspace_bytes(int(M), int(N), int(K)))


def fg_dequant_gemm_g4(X, W: Q4, bias=None, residual=None, act=FG_ACT_NONE, Y=None,
                       workspace=None, stream=None):
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, W.rows), dtype=torch.float16, device=X.device)
    need = fg_dequant_gemm_workspace_bytes(M, W.rows, W.cols)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    c = W.c()
    _ok(load().fg_dequant_gemm_g4(_ptr(X), M, ctypes.byref(c), _ptr(bias), _ptr(residual),
                                  int(act), _ptr(Y), _ptr(workspace), ws_bytes,
                                  _stream(stream)))
    return Y


NOALLOC_SCRATCH_BYTES = 16 << 20


def fg_dequant_gemm_g4_noalloc(X, W: Q4, bias=None, residual=None, act=FG_ACT_NONE, Y=None,
                               stream=None):
    """fg_dequant_gemm_g4 without a workspace argument, for callers that must
    not allocate device memory (the K-split scratch is a fixed 16 MiB array
    inside libfg).  Y must be passed in by such callers; it is created here
    only for convenience when omitted."""
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, W.rows), dtype=torch.float16, device=X.device)
    c = W.c()
    _ok(load().fg_dequant_gemm_g4_noalloc(_ptr(X), M, ctypes.byref(c), _ptr(bias),
                                          _ptr(residual), int(act), _ptr(Y), _stream(stream)))
    return Y


def fg_gemm_f16_f32out(X, W, Y=None, stream=None):
    M, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _ok(load().fg_gemm_f16_f32out(_ptr(X), M, _ptr(W), N, K, _ptr(Y), _stream(stream)))
    return Y


def fg_layernorm(x, gamma, beta, eps=1e-5, y=None, stream=None, rows=None, x_ld=None):
    """x: [rows][cols] fp16, or any tensor whose row r starts at element
    r * x_ld of its storage (pass rows and x_ld for a strided view)."""
    cols = gamma.shape[0]
    if rows is None:
        rows = x.shape[0]
    if x_ld is None:
        x_ld = cols
    if y is None:
        y = torch.empty((rows, cols), dtype=torch.float16, device=x.device)
    assert x.is_cuda and y.is_contiguous()
    _ok(load().fg_layernorm(ctypes.c_void_p(x.data_ptr()), int(rows), int(cols), int(x_ld),
                            _ptr(gamma), _ptr(beta), float(eps), _ptr(y), _stream(stream)))
    return y


def fg_embed(ids, T, pos0, e_tok, e_pos, y=None, stream=None, pad=None):
    ntok = ids.numel()
    h1 = e_tok.shape[1]
    if y is None:
        y = torch.empty((ntok, h1), dtype=torch.float16, device=e_tok.device)
    _ok(load().fg_embed(_ptr(ids), ntok, int(T), int(pos0), _pad(pad, ntok // max(int(T), 1)),
                        _ptr(e_tok), e_tok.shape[0], _ptr(e_pos), e_pos.shape[0], h1, _ptr(y),
                        _stream(stream)))
    return y


def fg_argmax(logits, out=None, stream=None):
    """Greedy token per row of fp32 logits [B][V] (lowest index among ties)."""
    B, V = logits.shape
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    _ok(load().fg_argmax(_ptr(logits), B, V, _ptr(out), _stream(stream)))
    return out


def fg_kv_append_g4(qkv, cache: KV4, pos, stream=None):
    c = cache.c()
    _ok(load().fg_kv_append_g4(_ptr(qkv), qkv.shape[1], ctypes.byref(c), int(pos),
                               _stream(stream)))


def fg_decode_attn_g4(qkv, cache: KV4, pos, fuse_append=True, out=None, stream=None, pad=None):
    if out is None:
        out = torch.empty((qkv.shape[0], cache.H * cache.d), dtype=torch.float16,
                          device=qkv.device)
    c = cache.c()
    _ok(load().fg_decode_attn_g4(_ptr(qkv), qkv.shape[1], ctypes.byref(c), int(pos),
                                 _pad(pad, cache.B), 1 if fuse_append else 0, _ptr(out),
                                 _stream(stream)))
    return out


def fg_topk_count(n, keep_pct) -> int:
    return int(load().fg_topk_count(int(n), int(keep_pct)))


def fg_decode_attn_topk_workspace_bytes(B, H, pos) -> int:
    return int(load().fg_decode_attn_topk_workspace_bytes(int(B), int(H), int(pos)))


def fg_decode_attn_topk_g4(qkv, cache: KV4, pos, keep_pct, fuse_append=True, out=None,
                           sel_out=None, stream=None, pad=None, workspace=None):
    """sel_out: None, True (allocate [B][H][kmax] int32 and return it), or a
    device int32 tensor of that shape.  workspace: None (allocated here) or
    a uint8 device tensor of fg_decode_attn_topk_workspace_bytes.  Returns
    out, or (out, sel_out)."""
    if workspace is None:
        n = fg_decode_attn_topk_workspace_bytes(cache.B, cache.H, pos)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=qkv.device)
    if out is None:
        out = torch.empty((qkv.shape[0], cache.H * cache.d), dtype=torch.float16,
                          device=qkv.device)
    want = sel_out is not None
    if sel_out is True:
        kmax = fg_topk_count(pos + 1, keep_pct)
        sel_out = torch.empty((cache.B, cache.H, max(kmax, 0)), dtype=torch.int32,
                              device=qkv.device)
    c = cache.c()
    _ok(load().fg_decode_attn_topk_g4(_ptr(qkv), qkv.shape[1], ctypes.byref(c), int(pos),
                                      _pad(pad, cache.B), int(keep_pct), 1 if fuse_append else 0,
                                      _ptr(out), _ptr(sel_out) if want else None,
                                      _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream)))
    return (out, sel_out) if want else out


def fg_prefill_attn(qkv, B, s, H, d, cache: KV4 | None = None, out=None, stream=None, pad=None):
    if out is None:
        out = torch.empty((B * s, H * d), dtype=torch.float16, device=qkv.device)
    c = None if cache is None else ctypes.byref(cache.c())
    _ok(load().fg_prefill_attn(_ptr(qkv), int(B), int(s), int(H), int(d), _pad(pad, B), c,
                               _ptr(out), _stream(stream)))
    return out


def fg_layer_workspace_bytes(layer_c: c_layer, phase, bls, T, policy: c_policy, cap=0) -> int:
    """cap: the cache capacity (sizes top-K attention's scores; 0 otherwise)."""
    return int(load().fg_layer_workspace_bytes(ctypes.byref(layer_c), int(phase), int(bls),
                                               int(T), int(cap), policy))


def fg_kv_store_f16(qkv, T, cache: KV16, slot0=0, stream=None):
    _ok(load().fg_kv_store_f16(_ptr(qkv), qkv.shape[1], int(T), ctypes.byref(cache.c()),
                               int(slot0), _stream(stream)))


def fg_decode_attn_f16(qkv, cache: KV16, pos, fuse_append=True, out=None, stream=None, pad=None):
    if out is None:
        out = torch.empty((qkv.shape[0], cache.H * cache.d), dtype=torch.float16,
                          device=qkv.device)
    c = cache.c()
    _ok(load().fg_decode_attn_f16(_ptr(qkv), qkv.shape[1], ctypes.byref(c), int(pos),
                                  _pad(pad, cache.B), 1 if fuse_append else 0, _ptr(out),
                                  _stream(stream)))
    return out


def fg_layer_step(layer_c: c_layer, cache, x_in, x_out, phase, T, pos,
                  policy: c_policy, workspace, stream=None, pad=None):
    """cache: KV4 (4-bit) or KV16 (fp16): fg_layer_step or fg_layer_step_kv16."""
    c = cache.c()
    fn = load().fg_layer_step_kv16 if isinstance(cache, KV16) else load().fg_layer_step
    _ok(fn(ctypes.byref(layer_c), ctypes.byref(c), _ptr(x_in), _ptr(x_out),
                             int(phase), int(T), int(pos), _pad(pad, cache.B), policy,
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)))
