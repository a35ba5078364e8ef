"""The uncompressed (fp16) KV cache -- the setting the pages compare the 4-bit
cache against ("FlexGen 完全拆解", results for input length 512) -- through
the C ABI against the oracle: the stores are bit-exact copies, the decode
attention agrees within fp32 summation-order error, and the layer and model
agree with the oracle run over an fp16 cache."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, Model, quantize_layer
from oracle.model import DECODE, PREFILL, OracleModel, generate, layer_step
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, rel_l2, to_np, ulp16  # noqa: F401

pytestmark = pytest.mark.gpu


def _filled(B, H, d, cap, L, seed):
    g = synth.generator(seed)
    oc = oracle.KVCache16(B, H, d, cap)
    if L:
        oc.k[:, :, :L] = synth.normal_f16((B, H, L, d), 1.0, g).numpy()
        oc.v[:, :, :L] = synth.normal_f16((B, H, L, d), 1.0, g).numpy()
    gc = fg.KV16(torch.from_numpy(oc.k.copy()).to(DEV), torch.from_numpy(oc.v.copy()).to(DEV),
                 B, H, d, cap)
    return oc, gc


def _tol(want, oc):
    """Both sides sum the same fp16 products in fp32, in different orders:
    a few fp32 ulps of the sums (the output is a convex combination of V
    rows, |out| <= max|V|), plus one fp16 rounding of the result."""
    vmax = float(np.max(np.abs(oc.v.astype(np.float64))))
    return ulp16(want) + 2e-5 * vmax


@pytest.mark.parametrize("B,H,d,L,padded", [
    (1, 1, 64, 1, False), (2, 3, 64, 63, True), (2, 2, 64, 64, False), (3, 2, 128, 65, True),
    (4, 12, 64, 40, False), (2, 4, 128, 513, True), (1, 2, 128, 1100, False),
    (1, 2, 128, 2048, False),
])
def test_decode_attn_f16_matches_oracle(B, H, d, L, padded):
    cap = L + 2
    oc, gc = _filled(B, H, d, cap, L - 1, B * 10 + L)
    g = synth.generator(L + 3)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, g)
    pad = synth.pad_counts(B, L, g).numpy().astype(np.int32) if padded else None
    out = fg.fg_decode_attn_f16(qkv.to(DEV), gc, L - 1, fuse_append=True,
                                pad=None if pad is None else torch.from_numpy(pad).to(DEV))
    fg.fg_check()
    ref = oracle.decode_attn_f16(qkv.numpy(), oc, L - 1, append=True, pad=pad)
    assert np.array_equal(to_np(gc.k), oc.k) and np.array_equal(to_np(gc.v), oc.v)
    got = to_np(out).astype(np.float64)
    want = ref.astype(np.float64)
    assert np.all(np.abs(got - want) <= _tol(want, oc))
    assert rel_l2(got, want) < 1e-3


def test_separate_store_equals_fused_append():
    B, H, d, L = 3, 4, 128, 130
    _, g1 = _filled(B, H, d, L, L - 1, 5)
    _, g2 = _filled(B, H, d, L, L - 1, 5)
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, synth.generator(6)).to(DEV)
    a = fg.fg_decode_attn_f16(qkv, g1, L - 1, fuse_append=True)
    fg.fg_kv_store_f16(qkv, 1, g2, slot0=L - 1)
    b = fg.fg_decode_attn_f16(qkv, g2, L - 1, fuse_append=False)
    fg.fg_check()
    assert torch.equal(a, b) and torch.equal(g1.k, g2.k) and torch.equal(g1.v, g2.v)


@pytest.mark.parametrize("B,T,H,d,slot0", [(2, 7, 3, 64, 0), (3, 33, 2, 128, 5), (1, 1, 56, 128, 9)])
def test_kv_store_f16_matches_oracle(B, T, H, d, slot0):
    g = synth.generator(B * T + slot0)
    qkv = synth.normal_f16((B * T, 3 * H * d), 1.0, g)
    oc, gc = _filled(B, H, d, slot0 + T + 2, 0, 1)
    fg.fg_kv_store_f16(qkv.to(DEV), T, gc, slot0=slot0)
    fg.fg_check()
    if slot0 == 0:
        oracle.kv_store_prefill_f16(qkv.numpy(), B, T, oc)
    else:   # the oracle's prefill store at slot 0, moved to slot0
        tmp = oracle.KVCache16(B, H, d, T)
        oracle.kv_store_prefill_f16(qkv.numpy(), B, T, tmp)
        oc.k[:, :, slot0:slot0 + T], oc.v[:, :, slot0:slot0 + T] = tmp.k, tmp.v
    assert np.array_equal(to_np(gc.k), oc.k) and np.array_equal(to_np(gc.v), oc.v)


def _layer(h1, H, h2, seed):
    g = synth.generator(seed)
    w = synth.layer_weights(h1, h2, g)
    w.update(synth.random_affine_params(h1, h2, g))
    gl = quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2)
    ol = oracle_layer({n: t.numpy() for n, t in w.items()}, h1, H, h2)
    return gl, ol, g


def test_opt125m_layer_with_f16_cache():
    """One OPT-125M-shaped layer over the fp16 cache, prompt 32 and 8 decode
    steps: per-step output relative L2 <= 5e-3 against the oracle, the
    stored rows within the projections' rounding."""
    wl = synth.OPT125M_LAYER
    gl, ol, g = _layer(wl.h1, wl.H, wl.h2, 0)
    stack = LayerStack([gl], wl.gbs, wl.k, wl.cap, DEV, kv="f16")
    oc = oracle.KVCache16(wl.bls, wl.H, wl.d, wl.cap)
    x = synth.normal_f16((wl.bls * wl.s, wl.h1), 1.0, g)
    y = stack.run(x.to(DEV), fg.FG_PHASE_PREFILL, wl.s, 0, fg.FG_ORDER_BLOCK)
    ref = layer_step(ol, x.numpy(), oc, PREFILL, wl.bls, wl.s)
    assert rel_l2(to_np(y), ref) <= 5e-3
    for t in range(1, wl.decode_steps + 1):
        xt = synth.normal_f16((wl.bls, wl.h1), 1.0, g)
        y = stack.run(xt.to(DEV), fg.FG_PHASE_DECODE, 1, wl.s + t - 1, fg.FG_ORDER_BLOCK)
        ref = layer_step(ol, xt.numpy(), oc, DECODE, wl.bls, 1, pos=wl.s + t - 1)
        assert rel_l2(to_np(y), ref) <= 5e-3, t
    fg.fg_check()
    # the stored rows are the projections' outputs as they are, which the two
    # sides round in different summation orders
    assert rel_l2(to_np(stack.caches[0].k), oc.k) <= 1e-3
    assert rel_l2(to_np(stack.caches[0].v), oc.v) <= 1e-3


def test_small_model_logits_with_f16_cache_match_oracle_and_orders_agree():
    h1, H, h2, V, gbs, k, s, D = 512, 8, 1024, 1000, 2, 2, 24, 3
    g = synth.generator(31)
    ws = []
    for _ in range(2):
        w = synth.layer_weights(h1, h2, g)
        w.update(synth.random_affine_params(h1, h2, g))
        ws.append(w)
    et, ep = synth.embeddings(V, s + D + 1, h1, g)
    lnf_g = (1 + synth.normal_f16((h1,), 0.1, g).float()).half()
    lnf_b = synth.normal_f16((h1,), 0.1, g)
    prompt = synth.token_ids((gbs * k, s), V, g)
    dec = synth.token_ids((gbs * k, D), V, g)
    om = OracleModel([oracle_layer({n: t.numpy() for n, t in w.items()}, h1, H, h2) for w in ws],
                     et.numpy(), ep.numpy(), lnf_g.numpy(), lnf_b.numpy())
    ref = generate(om, prompt.numpy(), dec.numpy(), gbs, k, order="block",
                   caches=om.new_caches(gbs * k, s + D + 1, kv="f16"))
    outs = []
    for order in ("block", "zigzag"):
        layers = [quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2) for w in ws]
        m = Model(LayerStack(layers, gbs, k, s + D + 1, DEV, kv="f16"), et.to(DEV), ep.to(DEV),
                  lnf_g.to(DEV), lnf_b.to(DEV))
        got = m.generate(prompt.to(DEV), dec.t().contiguous().to(DEV), order=order)
        fg.fg_check()
        outs.append([x.clone() for x in got])
        for t, (a, b) in enumerate(zip(got, ref)):
            a = to_np(a)
            assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(b)), (order, t)
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_layer_step_kv16_rejects_topk():
    gl, _, _ = _layer(128, 2, 256, 3)
    st = LayerStack([gl], 2, 1, 8, DEV, kv="f16")
    st.topk_pct = 10
    x = torch.zeros((2, 128), dtype=torch.float16, device=DEV)
    with pytest.raises(fg.FgError) as e:
        st.run(x, fg.FG_PHASE_DECODE, 1, 0, fg.FG_ORDER_BLOCK)
    assert e.value.status == fg.FG_ERR_UNSUPPORTED
