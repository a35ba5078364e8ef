"""Pins for the oracle's top-K sparse decode attention ("FlexGen 完全拆解",
section on the paper's further approximations: scores from every cached key,
only the V rows of the highest-scoring 10% loaded).

Readings pinned here: the softmax is the full one over all attended rows;
rows not kept add nothing (no renormalisation); ceil(n * pct / 100) rows are
kept; equal scores are kept lowest slot first.  The checks use facts outside
the oracle's own arithmetic: an fp64 softmax (scipy) over the dequantised
rows with a numpy ranking, the closed form of the kept count, keeping every
row (the dense attention, pinned separately), all-equal keys (the first
rows), a single kept row (its own V times its weight), and the padding
shift."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle

H16 = 2.0 ** -11


def f16(a):
    return np.asarray(a, dtype=np.float16)


def _filled_cache(rng, B, H, d, cap, L):
    c = oracle.KVCache(B, H, d, cap)
    for b in range(B):
        for h in range(H):
            kc, km = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            vc, vm = oracle.quantize_g4(f16(rng.standard_normal((L, d))))
            c.k_codes[b, h, :L], c.k_meta[b, h, :L] = kc, km
            c.v_codes[b, h, :L], c.v_meta[b, h, :L] = vc, vm
    return c


def _qkv(rng, B, H, d):
    return f16(rng.standard_normal((B, 3 * H * d)))


def _rows(c, b, h, lo, hi, v):
    codes = c.v_codes if v else c.k_codes
    meta = c.v_meta if v else c.k_meta
    return oracle.dequant_g4(codes[b, h, lo:hi], meta[b, h, lo:hi]).astype(np.float64)


def _ref(qkv, c, pos, pct, pad=None):
    """fp64: full softmax over slots p0..pos, sum over the top rows only.
    Returns (out, kept slots per (b, h), score gap at the cut per (b, h))."""
    B, H, d = c.B, c.H, c.d
    out = np.zeros((B, H * d))
    kept, gaps = {}, {}
    for b in range(B):
        p0 = 0 if pad is None else int(pad[b])
        n = pos + 1 - p0
        ks = -(-n * pct // 100)
        for h in range(H):
            q = qkv[b, h * d:(h + 1) * d].astype(np.float64)
            s = _rows(c, b, h, p0, pos + 1, False) @ q / np.sqrt(d)
            p = softmax(s)
            order = np.lexsort((np.arange(n), -s))      # score desc, slot asc
            top = np.sort(order[:ks])
            out[b, h * d:(h + 1) * d] = p[top] @ _rows(c, b, h, p0, pos + 1, True)[top]
            kept[b, h] = top + p0
            gaps[b, h] = (s[order[ks - 1]] - s[order[ks]]) if ks < n else np.inf
    return out, kept, gaps


def test_kept_count_closed_form():
    for n, pct, want in [(1, 10, 1), (9, 10, 1), (10, 10, 1), (11, 10, 2), (100, 10, 10),
                         (101, 10, 11), (513, 10, 52), (544, 10, 55), (1056, 10, 106),
                         (7, 100, 7), (7, 1, 1), (300, 33, 99), (301, 33, 100)]:
        assert oracle.topk_count(n, pct) == want


@pytest.mark.parametrize("B,H,d,L,pct", [(2, 2, 64, 40, 10), (1, 3, 128, 97, 10),
                                         (2, 1, 128, 64, 25), (1, 2, 64, 5, 50)])
def test_topk_against_fp64_ranking(B, H, d, L, pct):
    rng = np.random.default_rng(L * 31 + pct)
    c = _filled_cache(rng, B, H, d, L + 1, L - 1)
    qkv = _qkv(rng, B, H, d)
    out, sel = oracle.decode_attn_topk_g4(qkv, c, L - 1, pct, append=True)
    ref, kept, gaps = _ref(qkv, c, L - 1, pct)
    ks = oracle.topk_count(L, pct)
    assert sel.shape == (B, H, ks)
    for (b, h), top in kept.items():
        if gaps[b, h] > 1e-4:   # the fp32 scores cannot reorder the cut
            assert np.array_equal(sel[b, h], top)
    o = out.astype(np.float64)
    assert np.all(np.abs(o - ref) <= np.maximum(np.abs(ref), 2.0 ** -14) * H16 + 2e-5)
    # rows were dropped: the output differs from the dense attention
    if ks < L:
        assert not np.array_equal(out, oracle.decode_attn_g4(qkv, c, L - 1, append=False))


def test_keep_all_equals_dense():
    rng = np.random.default_rng(51)
    B, H, d, L = 2, 2, 128, 33
    c = _filled_cache(rng, B, H, d, L, L - 1)
    c2 = _filled_cache(np.random.default_rng(51), B, H, d, L, L - 1)
    qkv = _qkv(rng, B, H, d)
    pad = np.array([0, 7], np.int32)
    a, sel = oracle.decode_attn_topk_g4(qkv, c, L - 1, 100, append=True, pad=pad)
    b = oracle.decode_attn_g4(qkv, c2, L - 1, append=True, pad=pad)
    assert np.array_equal(a, b)
    assert np.array_equal(sel[0, 0], np.arange(L))
    assert np.array_equal(sel[1, 0], np.r_[np.arange(7, L), -np.ones(7, np.int32)])


def test_equal_keys_keep_lowest_slots():
    rng = np.random.default_rng(52)
    B, H, d, L, pct = 1, 1, 64, 30, 10
    c = _filled_cache(rng, B, H, d, L, L)
    c.k_codes[:] = c.k_codes[:, :, :1]
    c.k_meta[:] = c.k_meta[:, :, :1]
    qkv = _qkv(rng, B, H, d)
    out, sel = oracle.decode_attn_topk_g4(qkv, c, L - 1, pct, append=False)
    assert np.array_equal(sel[0, 0], [0, 1, 2])
    # equal weights 1/L on the three kept rows
    ref = _rows(c, 0, 0, 0, 3, True).sum(0) / L
    assert np.all(np.abs(out[0].astype(np.float64) - ref) <= np.abs(ref) * H16 + 1e-6)


def test_single_kept_row_is_its_weighted_v():
    rng = np.random.default_rng(53)
    B, H, d, L = 1, 1, 128, 9
    c = _filled_cache(rng, B, H, d, L, L)
    qkv = _qkv(rng, B, H, d)
    # slot 4's key is q itself (quantised): it has the largest score
    kc, km = oracle.quantize_g4(qkv[:, :d] * 3)
    c.k_codes[0, 0, 4], c.k_meta[0, 0, 4] = kc[0], km[0]
    out, sel = oracle.decode_attn_topk_g4(qkv, c, L - 1, 10, append=False)
    assert np.array_equal(sel[0, 0], [4])
    q = qkv[0, :d].astype(np.float64)
    p = softmax(_rows(c, 0, 0, 0, L, False) @ q / np.sqrt(d))
    assert np.argmax(p) == 4
    ref = p[4] * _rows(c, 0, 0, 4, 5, True)[0]
    assert np.all(np.abs(out[0].astype(np.float64) - ref) <= np.abs(ref) * H16 + 1e-6)


def test_padded_equals_shifted_and_given_selection_round_trips():
    rng = np.random.default_rng(54)
    B, H, d, L, p0, pct = 1, 2, 64, 41, 9, 10
    c = _filled_cache(rng, B, H, d, L, L - 1)
    qkv = _qkv(rng, B, H, d)
    a, sa = oracle.decode_attn_topk_g4(qkv, c, L - 1, pct, append=True,
                                       pad=np.array([p0], np.int32))
    c2 = oracle.KVCache(B, H, d, L)
    for src, dst in ((c.k_codes, c2.k_codes), (c.k_meta, c2.k_meta),
                     (c.v_codes, c2.v_codes), (c.v_meta, c2.v_meta)):
        dst[:, :, :L - p0] = src[:, :, p0:L]
    b, sb = oracle.decode_attn_topk_g4(qkv, c2, L - 1 - p0, pct, append=False)
    assert np.array_equal(a, b)
    ks = oracle.topk_count(L - p0, pct)
    assert np.array_equal(sa[:, :, :ks], sb[:, :, :ks] + p0)
    assert np.all(sa[:, :, ks:] == -1) and np.all(sa[:, :, :ks] >= p0)
    # the oracle's own choice handed back reproduces its output bit for bit
    again, s2 = oracle.decode_attn_topk_g4(qkv, c, L - 1, pct, append=False,
                                           pad=np.array([p0], np.int32), sel=sa)
    assert np.array_equal(again, a) and np.array_equal(s2, sa)
    # another choice changes it
    other = sa.copy()
    other[0, 0, 0] = next(j for j in range(p0, L) if j not in set(sa[0, 0]))
    other[0, 0, :ks] = np.sort(other[0, 0, :ks])
    moved, _ = oracle.decode_attn_topk_g4(qkv, c, L - 1, pct, append=False,
                                          pad=np.array([p0], np.int32), sel=other)
    assert not np.array_equal(moved[0, :d], a[0, :d])
    assert np.array_equal(moved[0, d:], a[0, d:])
