"""The C-ABI library loads, exports every symbol include/fg.h declares, and
rejects invalid arguments on the host before any launch (no GPU needed:
validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

from bit_group_quant_gb300 import fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    src = open(os.path.join(ROOT, "include", "fg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fg_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return fg.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fg.EXPORTS)


def test_version_and_status_strings(lib):
    assert fg.fg_version() >> 16 == 4
    assert lib.fg_status_str(fg.FG_ERR_TIMEOUT) == b"device wait timed out"


def _status(call):
    with pytest.raises(fg.FgError) as e:
        call()
    return e.value.status


def test_host_validation_rejects_without_launch(lib):
    P = ctypes.c_void_p
    q = fg.c_q4(P(0x1000), P(0x2000), 128, 100)            # cols not a multiple of 64
    assert lib.fg_quantize_g4(P(0x3000), 128, 100, ctypes.byref(q), None) == fg.FG_ERR_SHAPE
    q = fg.c_q4(P(0x1008), P(0x2000), 128, 128)            # misaligned codes
    assert lib.fg_quantize_g4(P(0x3000), 128, 128, ctypes.byref(q), None) == fg.FG_ERR_ALIGN
    q = fg.c_q4(None, P(0x2000), 128, 128)
    assert lib.fg_quantize_g4(P(0x3000), 128, 128, ctypes.byref(q), None) == fg.FG_ERR_NULL
    q = fg.c_q4(P(0x1000), P(0x2000), 100, 128)            # N % 16 != 0
    assert lib.fg_dequant_gemm_g4(P(0x3000), 4, ctypes.byref(q), None, None, 0, P(0x4000),
                                  None, 0, None) == fg.FG_ERR_SHAPE
    q = fg.c_q4(P(0x1000), P(0x2000), 128, 128)
    assert lib.fg_dequant_gemm_g4(P(0x3000), 4, ctypes.byref(q), None, None, 7, P(0x4000),
                                  None, 0, None) == fg.FG_ERR_SHAPE      # bad act
    assert lib.fg_dequant_gemm_g4(P(0x3000), 0, ctypes.byref(q), None, None, 0, P(0x4000),
                                  None, 0, None) == fg.FG_OK            # M == 0: no work
    kv = fg.c_kv4(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 2, 2, 96, 8)   # d = 96
    assert lib.fg_decode_attn_g4(P(0x5000), 576, ctypes.byref(kv), 0, None, 1, P(0x6000),
                                 None) == fg.FG_ERR_UNSUPPORTED
    kv = fg.c_kv4(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 2, 2, 64, 8)
    assert lib.fg_decode_attn_g4(P(0x5000), 384, ctypes.byref(kv), 8, None, 1, P(0x6000),
                                 None) == fg.FG_ERR_SHAPE               # pos == cap
    assert lib.fg_decode_attn_g4(P(0x5000), 384, ctypes.byref(kv), 7, P(0x7002), 1, P(0x6000),
                                 None) == fg.FG_ERR_ALIGN               # pad misaligned
    for pct in (0, 101, -5):                                            # keep_pct outside [1, 100]
        assert lib.fg_decode_attn_topk_g4(P(0x5000), 384, ctypes.byref(kv), 7, None, pct, 1,
                                          P(0x6000), None, P(0x8000), 1 << 20,
                                          None) == fg.FG_ERR_SHAPE
    assert lib.fg_decode_attn_topk_g4(P(0x5000), 384, ctypes.byref(kv), 7, None, 10, 1,
                                      P(0x6000), P(0x7001), P(0x8000), 1 << 20,
                                      None) == fg.FG_ERR_ALIGN                         # sel_out
    assert lib.fg_decode_attn_topk_g4(P(0x5000), 384, ctypes.byref(kv), 8, None, 10, 1,
                                      P(0x6000), None, P(0x8000), 1 << 20,
                                      None) == fg.FG_ERR_SHAPE                         # pos == cap
    assert lib.fg_decode_attn_topk_g4(P(0x5000), 384, ctypes.byref(kv), 7, None, 10, 1,
                                      P(0x6000), None, P(0x8010), 1 << 20,
                                      None) == fg.FG_ERR_ALIGN                         # workspace
    need = lib.fg_decode_attn_topk_workspace_bytes(2, 2, 7)   # scores 2*2*8 fp32 + stats, 256-aligned
    assert need == 512
    assert lib.fg_decode_attn_topk_g4(P(0x5000), 384, ctypes.byref(kv), 7, None, 10, 1,
                                      P(0x6000), None, P(0x8000), need - 1,
                                      None) == fg.FG_ERR_WORKSPACE
    for n, pct, want in [(513, 10, 52), (1, 10, 1), (10, 10, 1), (11, 10, 2), (7, 100, 7),
                         (0, 10, 0), (5, 0, -1), (5, 101, -1), (-1, 10, -1)]:
        assert lib.fg_topk_count(n, pct) == want
    kv16 = fg.c_kv16(P(0x1000), P(0x2000), 2, 2, 96, 8)                      # d = 96
    assert lib.fg_decode_attn_f16(P(0x5000), 576, ctypes.byref(kv16), 0, None, 1, P(0x6000),
                                  None) == fg.FG_ERR_UNSUPPORTED
    kv16 = fg.c_kv16(P(0x1000), P(0x2008), 2, 2, 64, 8)                      # v misaligned
    assert lib.fg_kv_store_f16(P(0x5000), 384, 1, ctypes.byref(kv16), 0, None) == fg.FG_ERR_ALIGN
    kv16 = fg.c_kv16(P(0x1000), P(0x2000), 2, 2, 64, 8)
    assert lib.fg_decode_attn_f16(P(0x5000), 384, ctypes.byref(kv16), 8, None, 1, P(0x6000),
                                  None) == fg.FG_ERR_SHAPE                 # pos == cap
    assert lib.fg_kv_store_f16(P(0x5000), 384, 4, ctypes.byref(kv16), 5, None) == fg.FG_ERR_SHAPE
    assert lib.fg_kv_store_f16(P(0x5000), 100, 1, ctypes.byref(kv16), 0, None) == fg.FG_ERR_SHAPE
    assert lib.fg_kv_store_f16(P(0x5000), 384, 0, ctypes.byref(kv16), 0, None) == fg.FG_OK
    assert lib.fg_kv_append_g4(P(0x5000), 100, ctypes.byref(kv), 0, None) == fg.FG_ERR_SHAPE
    assert lib.fg_layernorm(P(0x1000), 4, 100, 100, P(0x2000), P(0x3000), 1e-5, P(0x4000),
                            None) == fg.FG_ERR_SHAPE
    assert lib.fg_prefill_attn(P(0x1000), 1, 4, 2, 80, None, None, P(0x2000),
                               None) == fg.FG_ERR_UNSUPPORTED
    assert lib.fg_prefill_attn(P(0x1000), 1, 4, 2, 64, P(0x3001), None, P(0x2000),
                               None) == fg.FG_ERR_ALIGN
    assert lib.fg_argmax(P(0x1000), 4, 0, P(0x2000), None) == fg.FG_ERR_SHAPE
    assert lib.fg_argmax(P(0x1000), 4, 10, None, None) == fg.FG_ERR_NULL
    assert lib.fg_argmax(P(0x1000), 0, 10, None, None) == fg.FG_OK      # B == 0: no work
    assert lib.fg_embed(P(0x1000), 8, 3, 0, None, P(0x2000), 10, P(0x3000), 16, 64, P(0x4000),
                        None) == fg.FG_ERR_SHAPE                        # ntok % T != 0
    assert lib.fg_debug_set(99, 1) == fg.FG_ERR_UNSUPPORTED
    assert b"unknown knob" in lib.fg_last_error()


def test_layer_step_validation(lib):
    P = ctypes.c_void_p
    h1, H, h2 = 128, 2, 256
    q = lambda r, c: fg.c_q4(P(0x10000), P(0x20000), r, c)
    L = fg.c_layer(q(3 * h1, h1), q(h1, h1), q(h2, h1), q(h1, h2), *([P(0x30000)] * 8),
                   h1, H, h2, 1e-5)
    kv = fg.c_kv4(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 4, H, 64, 16)
    pol = fg.c_policy(2, 3, 0)                                # bls 6 != cache B 4
    need = lib.fg_layer_workspace_bytes(ctypes.byref(L), 0, 6, 8, 16, pol)
    assert need > 0
    st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 0, 8, 0,
                           None, pol, P(0x100000), need, None)
    assert st == fg.FG_ERR_SHAPE and b"bls" in lib.fg_last_error()
    pol = fg.c_policy(2, 2, 0)
    st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 1, 2, 0,
                           None, pol, P(0x100000), 1 << 30, None)
    assert st == fg.FG_ERR_SHAPE                              # decode needs T == 1
    st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 1, 1, 3,
                           None, pol, P(0x100000), 16, None)
    assert st == fg.FG_ERR_WORKSPACE
    dense = lib.fg_layer_workspace_bytes(ctypes.byref(L), 1, 4, 1, 16, pol)
    topk = lib.fg_layer_workspace_bytes(ctypes.byref(L), 1, 4, 1, 16, fg.c_policy(2, 2, 0, 10))
    assert topk == dense + lib.fg_decode_attn_topk_workspace_bytes(4, H, 15)
    assert lib.fg_layer_workspace_bytes(ctypes.byref(L), 1, 4, 1, 16, fg.c_policy(2, 2, 0, 100)) == dense
    st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 1, 1, 15,
                           None, fg.c_policy(2, 2, 0, 10), P(0x100000), dense, None)
    assert st == fg.FG_ERR_WORKSPACE                          # top-K needs its scores space
    for bad in (-1, 101):
        st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 1, 1, 3,
                               None, fg.c_policy(2, 2, 0, bad), P(0x100000), 1 << 30, None)
        assert st == fg.FG_ERR_SHAPE and b"topk_pct" in lib.fg_last_error()
    kv16 = fg.c_kv16(P(0x1000), P(0x2000), 4, H, 64, 16)
    st = lib.fg_layer_step_kv16(ctypes.byref(L), ctypes.byref(kv16), P(0x5000), P(0x6000), 1, 1, 3,
                                None, fg.c_policy(2, 2, 0, 10), P(0x100000), 1 << 30, None)
    assert st == fg.FG_ERR_UNSUPPORTED and b"4-bit" in lib.fg_last_error()
    st = lib.fg_layer_step_kv16(ctypes.byref(L), ctypes.byref(kv16), P(0x5000), P(0x6000), 1, 1, 3,
                                None, fg.c_policy(2, 3, 0), P(0x100000), 1 << 30, None)
    assert st == fg.FG_ERR_SHAPE and b"bls" in lib.fg_last_error()
    L.fc1 = q(h2 + 64, h1)
    st = lib.fg_layer_step(ctypes.byref(L), ctypes.byref(kv), P(0x5000), P(0x6000), 1, 1, 3,
                           None, pol, P(0x100000), 1 << 30, None)
    assert st == fg.FG_ERR_SHAPE
