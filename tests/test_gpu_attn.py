"""Decode attention over the 4-bit cache (with fused append) and causal
prefill attention against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg

from gpu_util import DEV, rel_l2, to_np

pytestmark = pytest.mark.gpu


def _fill_cache(B, H, d, cap, L, seed):
    """Cache slots 0..L-1 from N(0,1) fp16 rows, quantised by the oracle
    (the same bytes go to both sides)."""
    g = synth.generator(seed)
    rows = synth.normal_f16((2, B * H * L, d), 1.0, g).numpy()
    oc = oracle.KVCache(B, H, d, cap)
    if L:
        kc, km = oracle.quantize_g4(rows[0])
        vc, vm = oracle.quantize_g4(rows[1])
        oc.k_codes[:, :, :L] = kc.reshape(B, H, L, -1)
        oc.k_meta[:, :, :L] = km.reshape(B, H, L, -1, 2)
        oc.v_codes[:, :, :L] = vc.reshape(B, H, L, -1)
        oc.v_meta[:, :, :L] = vm.reshape(B, H, L, -1, 2)
    gc = fg.KV4(*(torch.from_numpy(a.copy()).to(DEV) for a in
                  (oc.k_codes, oc.v_codes, oc.k_meta, oc.v_meta)), B, H, d, cap)
    return oc, gc


def _attn_tol(out_ref, cache, L):
    """Output is a convex combination of dequantised V rows: score
    perturbations of size e move it by at most ~2e * max|V^|; plus fp16
    rounding of the result."""
    vmax = 0.0
    for meta, codes in ((cache.v_meta, cache.v_codes),):
        m = meta[:, :, :L, :, 0]
        s = meta[:, :, :L, :, 1]
        vmax = float(np.max(np.abs(m) + 15 * np.abs(s)))
    return 4e-3 * vmax + np.maximum(np.abs(out_ref), 2.0 ** -14) * 2.0 ** -10


@pytest.mark.parametrize("B,H,d,L", [
    (1, 1, 64, 1), (2, 3, 64, 63), (2, 2, 64, 64), (3, 2, 128, 65), (4, 12, 64, 40),
    (2, 4, 128, 513), (1, 2, 128, 2048),
])
def test_decode_attn_matches_oracle(B, H, d, L):
    cap = L + 2
    oc, gc = _fill_cache(B, H, d, cap, L - 1, B * 100 + L)
    h1 = H * d
    g = synth.generator(L)
    qkv = synth.normal_f16((B, 3 * h1), 1.0, g)
    out = fg.fg_decode_attn_g4(qkv.to(DEV), gc, L - 1, fuse_append=True)
    fg.fg_check()
    ref = oracle.decode_attn_g4(qkv.numpy(), oc, L - 1, append=True)
    # the fused append wrote exactly the oracle's bytes
    for a, b in ((gc.k_codes, oc.k_codes), (gc.v_codes, oc.v_codes),
                 (gc.k_meta, oc.k_meta), (gc.v_meta, oc.v_meta)):
        assert np.array_equal(to_np(a), b)
    got = to_np(out).astype(np.float64)
    want = ref.astype(np.float64)
    assert np.all(np.abs(got - want) <= _attn_tol(want, oc, L))
    assert rel_l2(got, want) < 2e-3


def test_decode_attn_without_append_matches_separate_append():
    B, H, d, L = 2, 4, 128, 100
    oc, gc = _fill_cache(B, H, d, L + 1, L - 1, 11)
    _, gc2 = _fill_cache(B, H, d, L + 1, L - 1, 11)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(12)).to(DEV)
    a = fg.fg_decode_attn_g4(qkv, gc, L - 1, fuse_append=True)
    fg.fg_kv_append_g4(qkv, gc2, L - 1)
    b = fg.fg_decode_attn_g4(qkv, gc2, L - 1, fuse_append=False)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(gc.k_codes, gc2.k_codes) and torch.equal(gc.v_meta, gc2.v_meta)


@pytest.mark.parametrize("B,s,H,d", [(1, 1, 1, 64), (2, 33, 3, 64), (1, 70, 2, 128), (4, 32, 12, 64)])
def test_prefill_attn_and_store_match_oracle(B, s, H, d):
    g = synth.generator(B * s + H)
    h1 = H * d
    qkv = synth.normal_f16((B * s, 3 * h1), 1.0, g)
    gc = fg.KV4.empty(B, H, d, s + 3, DEV)
    out = fg.fg_prefill_attn(qkv.to(DEV), B, s, H, d, cache=gc)
    fg.fg_check()
    ref = oracle.prefill_attn(qkv.numpy(), B, s, H, d)
    oc = oracle.KVCache(B, H, d, s + 3)
    oracle.kv_store_prefill(qkv.numpy(), B, s, oc)
    for a, b in ((gc.k_codes, oc.k_codes), (gc.v_codes, oc.v_codes),
                 (gc.k_meta, oc.k_meta), (gc.v_meta, oc.v_meta)):
        assert np.array_equal(to_np(a), b)
    got = to_np(out).astype(np.float64)
    want = ref.astype(np.float64)
    vmax = float(np.abs(qkv.numpy()[:, 2 * h1:]).max())
    assert np.all(np.abs(got - want) <= 4e-3 * vmax + np.maximum(np.abs(want), 2.0 ** -14) * 2.0 ** -10)
    assert rel_l2(got, want) < 2e-3
