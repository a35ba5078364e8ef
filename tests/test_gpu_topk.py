"""Top-K sparse decode attention through the C ABI against the oracle
("FlexGen 完全拆解", section on the paper's further approximations: scores
from every cached key, only the highest-scoring rows' V loaded).

Which rows are kept is an integer decided by floating point: the kernel ranks
its fp32 scores of the unrounded dequantised keys (m + c s), the oracle its
fp32 scores of fp16-rounded keys, so two keys whose scores differ by less
than those roundings may be kept by one side and not the other.  The tests
therefore check (1) that the kernel's kept set is a valid top set against
fp64 scores, and equal to the fp64 top set wherever the cut is clear of
rounding; (2) the weighted sum against the oracle run on the kernel's own
kept set; (3) identities: keeping every row keeps every slot and gives the
dense result, equal keys keep the lowest slots, the layer step's wiring
equals the composition of the public calls bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, quantize_layer

from gpu_util import DEV, rel_l2, to_np, unpack_codes
from test_gpu_attn import _attn_tol, _fill_cache

pytestmark = pytest.mark.gpu


def _scores64(oc, qkv, b, h, p0, L):
    """fp64 scores of slots p0..L-1 over the unrounded dequantised keys."""
    d = oc.d
    c = unpack_codes(oc.k_codes[b, h, p0:L]).astype(np.float64)
    m = np.repeat(oc.k_meta[b, h, p0:L, :, 0].astype(np.float64), 64, axis=1)
    s = np.repeat(oc.k_meta[b, h, p0:L, :, 1].astype(np.float64), 64, axis=1)
    q = np.asarray(qkv[b, h * d:(h + 1) * d], np.float64)
    return (m + c * s) @ q / np.sqrt(d)


def _check_selection(sel, oc, qkv, pos, pct, pad, bs=None):
    """Valid kept sets; returns how many (b, h) had a clear cut and matched
    the fp64 top set exactly."""
    B, H = sel.shape[:2]
    kmax = oracle.topk_count(pos + 1, pct)
    assert sel.shape == (B, H, kmax)
    exact = 0
    for i in range(B):
        b = i if bs is None else bs[i]
        p0 = 0 if pad is None else int(pad[i])
        n = pos + 1 - p0
        ks = oracle.topk_count(n, pct)
        for h in range(H):
            row = sel[i, h]
            assert np.all(row[ks:] == -1)
            kept = row[:ks]
            assert np.all(np.diff(kept) > 0) and kept[0] >= p0 and kept[-1] <= pos
            if ks == n:
                continue
            s = _scores64(oc, qkv, b, h, p0, pos + 1)
            eps = 1e-4 * (1.0 + np.abs(s).max())
            mask = np.zeros(n, bool)
            mask[kept - p0] = True
            assert s[mask].min() >= s[~mask].max() - eps
            order = np.lexsort((np.arange(n), -s))
            if s[order[ks - 1]] - s[order[ks]] > eps:
                assert np.array_equal(np.sort(order[:ks]) + p0, kept)
                exact += 1
    return exact


CASES = [
    (1, 1, 64, 1, 10, False), (2, 3, 64, 63, 10, False), (4, 12, 64, 40, 10, True),
    (2, 2, 128, 65, 10, False), (3, 2, 128, 513, 10, True), (2, 4, 64, 300, 25, True),
    (2, 2, 128, 1100, 50, False), (1, 2, 128, 2048, 10, False), (2, 3, 128, 200, 1, True),
]


@pytest.mark.parametrize("B,H,d,L,pct,padded", CASES)
def test_topk_matches_oracle(B, H, d, L, pct, padded):
    cap = L + 2
    oc, gc = _fill_cache(B, H, d, cap, L - 1, B * 1000 + L + pct)
    h1 = H * d
    g = synth.generator(L + 7)
    qkv = synth.normal_f16((B, 3 * h1), 1.0, g)
    pad = None
    if padded:
        pad = synth.pad_counts(B, L, g, min_len=1)
        pad = pad.numpy().astype(np.int32)
    out, sel = fg.fg_decode_attn_topk_g4(qkv.to(DEV), gc, L - 1, pct, fuse_append=True,
                                         sel_out=True,
                                         pad=None if pad is None else torch.from_numpy(pad).to(DEV))
    fg.fg_check()
    q = qkv.numpy()
    oracle.decode_attn_topk_g4(q, oc, L - 1, pct, append=True, pad=pad)
    for a, b in ((gc.k_codes, oc.k_codes), (gc.v_codes, oc.v_codes),
                 (gc.k_meta, oc.k_meta), (gc.v_meta, oc.v_meta)):
        assert np.array_equal(to_np(a), b)     # the fused append wrote the oracle's bytes
    sel = to_np(sel)
    exact = _check_selection(sel, oc, q, L - 1, pct, pad)
    if L >= 200:
        assert exact >= (B * H) // 2
    ref, used = oracle.decode_attn_topk_g4(q, oc, L - 1, pct, append=False, pad=pad, sel=sel)
    assert np.array_equal(used, sel)
    got = to_np(out).astype(np.float64)
    want = ref.astype(np.float64)
    assert np.all(np.abs(got - want) <= _attn_tol(want, oc, L))
    assert rel_l2(got, want) < 2e-3


@pytest.mark.parametrize("d,L,padded", [(64, 65, False), (128, 65, True), (128, 513, True),
                                        (64, 300, True), (128, 1100, False)])
def test_keep_all_matches_dense(d, L, padded):
    """Keeping 100% of the rows keeps every slot and gives the dense result
    (within the attention tolerance: the gather sums the same weights in
    another order)."""
    B, H = 3, 2
    oc, g1 = _fill_cache(B, H, d, L + 1, L - 1, 77 + L)
    _, g2 = _fill_cache(B, H, d, L + 1, L - 1, 77 + L)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(78)).to(DEV)
    pad = torch.tensor([0, 5, L - 1], dtype=torch.int32, device=DEV) if padded else None
    a, sel = fg.fg_decode_attn_topk_g4(qkv, g1, L - 1, 100, sel_out=True, pad=pad)
    b = fg.fg_decode_attn_g4(qkv, g2, L - 1, pad=pad)
    fg.fg_check()
    got, want = to_np(a).astype(np.float64), to_np(b).astype(np.float64)
    assert np.all(np.abs(got - want) <= _attn_tol(want, oc, L))
    assert rel_l2(got, want) < 2e-3
    s = to_np(sel)
    p0 = [0, 5, L - 1] if padded else [0, 0, 0]
    for i in range(B):
        n = L - p0[i]
        assert np.array_equal(s[i, :, :n], np.broadcast_to(np.arange(p0[i], L), (H, n)))
        assert np.all(s[i, :, n:] == -1)


def test_kept_list_is_optional_and_does_not_change_the_output():
    B, H, d, L = 2, 4, 128, 400
    _, g1 = _fill_cache(B, H, d, L, L - 1, 91)
    _, g2 = _fill_cache(B, H, d, L, L - 1, 91)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(92)).to(DEV)
    a, _ = fg.fg_decode_attn_topk_g4(qkv, g1, L - 1, 10, sel_out=True)
    b = fg.fg_decode_attn_topk_g4(qkv, g2, L - 1, 10)
    dense = fg.fg_decode_attn_g4(qkv, g2, L - 1, fuse_append=False)
    fg.fg_check()
    assert torch.equal(a, b)
    assert not torch.equal(a, dense)


@pytest.mark.parametrize("d", [64, 128])
def test_equal_keys_keep_lowest_slots(d):
    B, H, L, pct = 2, 3, 150, 10
    oc, _ = _fill_cache(B, H, d, L, L, 93)
    oc.k_codes[:] = oc.k_codes[:, :, :1]
    oc.k_meta[:] = oc.k_meta[:, :, :1]
    gc = fg.KV4(*(torch.from_numpy(a.copy()).to(DEV) for a in
                  (oc.k_codes, oc.v_codes, oc.k_meta, oc.v_meta)), B, H, d, L)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(94))
    pad = torch.tensor([0, 17], dtype=torch.int32, device=DEV)
    out, sel = fg.fg_decode_attn_topk_g4(qkv.to(DEV), gc, L - 1, pct, fuse_append=False,
                                         sel_out=True, pad=pad)
    fg.fg_check()
    s = to_np(sel)
    for i, p0 in enumerate((0, 17)):
        ks = oracle.topk_count(L - p0, pct)
        assert np.array_equal(s[i, :, :ks], np.broadcast_to(np.arange(p0, p0 + ks), (H, ks)))
    ref, used = oracle.decode_attn_topk_g4(qkv.numpy(), oc, L - 1, pct, append=False,
                                           pad=np.array([0, 17], np.int32))
    assert np.array_equal(used, s)
    got = to_np(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= _attn_tol(ref.astype(np.float64), oc, L))


def test_opt30b_shape_full_block_sampled():
    """The 30B shape at its benchmark block: 144 sequences x 56 heads of
    d 128 at context 513 (prompt 512 + the appended row), keep 10%, a
    synthetic 4-bit cache (codes uniform, group min and scale of N(0,1)
    rows); six sequences checked head by head against the oracle."""
    B, H, d, L, pct = 144, 56, 128, 513, 10
    g = synth.generator(2024, DEV)
    shp = (B, H, L, d // 2)
    kc = torch.randint(0, 256, shp, dtype=torch.uint8, device=DEV, generator=g)
    vc = torch.randint(0, 256, shp, dtype=torch.uint8, device=DEV, generator=g)
    meta = lambda: torch.stack([-2.4 + 0.3 * torch.randn((B, H, L, d // 64), device=DEV, generator=g),
                                0.32 + 0.03 * torch.randn((B, H, L, d // 64), device=DEV, generator=g)], -1)
    km, vm = meta(), meta()
    gc = fg.KV4(kc, vc, km.contiguous(), vm.contiguous(), B, H, d, L)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, g, DEV)
    pad = synth.pad_counts(B, L - 1, g, min_len=64, device=DEV)
    host = [t.cpu().numpy() for t in (kc, vc, km, vm)]
    out, sel = fg.fg_decode_attn_topk_g4(qkv, gc, L - 1, pct, sel_out=True, pad=pad)
    fg.fg_check()
    bs = [0, 1, 47, 90, 128, 143]
    oc = oracle.KVCache(len(bs), H, d, L)
    oc.k_codes[:], oc.v_codes[:] = host[0][bs], host[1][bs]
    oc.k_meta[:], oc.v_meta[:] = host[2][bs], host[3][bs]
    q = qkv.cpu().numpy()[bs]
    p = pad.cpu().numpy().astype(np.int32)[bs]
    oracle.decode_attn_topk_g4(q, oc, L - 1, pct, append=True, pad=p)
    got_sel = to_np(sel)[bs]
    exact = _check_selection(got_sel, oc, q, L - 1, pct, p)
    assert exact >= len(bs) * H // 2
    ref, _ = oracle.decode_attn_topk_g4(q, oc, L - 1, pct, append=False, pad=p, sel=got_sel)
    got = to_np(out)[bs].astype(np.float64)
    want = ref.astype(np.float64)
    assert np.all(np.abs(got - want) <= _attn_tol(want, oc, L))
    assert rel_l2(got, want) < 2e-3


def test_layer_step_topk_equals_public_calls():
    """fg_layer_step with topk_pct 10 (block order) equals, bit for bit, the
    decode layer composed from the public calls with fg_decode_attn_topk_g4;
    every block order agrees; topk_pct 100 is the dense step."""
    h1, H, h2, gbs, k, s = 256, 2, 1024, 3, 2, 150
    g = synth.generator(95)
    w = synth.layer_weights(h1, h2, g)
    w.update(synth.random_affine_params(h1, h2, g))
    gl = quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2)
    bls = gbs * k
    x0 = synth.normal_f16((bls * s, h1), 1.0, g).to(DEV)
    x1 = synth.normal_f16((bls, h1), 1.0, g).to(DEV)
    outs = {}
    for name, pct, order in (("topk", 10, fg.FG_ORDER_BLOCK), ("topk_b", 10, fg.FG_ORDER_BATCHES),
                             ("topk_r", 10, fg.FG_ORDER_BATCHES_REV), ("dense", 0, fg.FG_ORDER_BLOCK),
                             ("all", 100, fg.FG_ORDER_BLOCK), ("manual", 0, fg.FG_ORDER_BLOCK)):
        st = LayerStack([gl], gbs, k, s + 1, DEV)
        st.topk_pct = pct
        st.run(x0, fg.FG_PHASE_PREFILL, s, 0, fg.FG_ORDER_BLOCK)
        if name != "manual":
            outs[name] = st.run(x1, fg.FG_PHASE_DECODE, 1, s, order).clone()
            continue
        c = st.caches[0]
        a = fg.fg_layernorm(x1, gl.ln1_g, gl.ln1_b, gl.eps)
        qkv = fg.fg_dequant_gemm_g4(a, gl.qkv, bias=gl.b_qkv)
        attn = fg.fg_decode_attn_topk_g4(qkv, c, s, 10)
        hh = fg.fg_dequant_gemm_g4(attn, gl.out, bias=gl.b_out, residual=x1)
        a2 = fg.fg_layernorm(hh, gl.ln2_g, gl.ln2_b, gl.eps)
        u = fg.fg_dequant_gemm_g4(a2, gl.fc1, bias=gl.b_fc1, act=fg.FG_ACT_RELU)
        outs[name] = fg.fg_dequant_gemm_g4(u, gl.fc2, bias=gl.b_fc2, residual=hh)
    fg.fg_check()
    assert torch.equal(outs["topk"], outs["manual"])
    assert torch.equal(outs["topk"], outs["topk_b"]) and torch.equal(outs["topk"], outs["topk_r"])
    assert torch.equal(outs["dense"], outs["all"])
    assert not torch.equal(outs["topk"], outs["dense"])
