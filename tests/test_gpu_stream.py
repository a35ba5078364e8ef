"""Weights streamed from pinned host memory one layer ahead (HostLayerStack)
give, bit for bit, the tokens and logits of the same weights resident in
HBM: the same kernels read the same bytes; only where the bytes come from
and when they arrive differ.  Covers the block and zig-zag orders, prefill
and greedy decode steps, and the fetch that crosses token steps (the last
layer's successor is layer 0 of the next step)."""
import pytest
import torch

import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import HostLayerStack, LayerStack, Model, quantize_layer

from gpu_util import DEV

pytestmark = pytest.mark.gpu


def _layers(ws, h1, H, h2):
    return [quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2) for w in ws]


@pytest.mark.parametrize("order", ["block", "zigzag"])
def test_host_streamed_weights_bitwise_equal_resident(order):
    h1, H, h2, V, gbs, k, s, n, nl = 512, 4, 1024, 700, 2, 3, 40, 6, 5   # odd layer count
    g = synth.generator(300)
    ws = []
    for _ in range(nl):
        w = synth.layer_weights(h1, h2, g)
        w.update(synth.random_affine_params(h1, h2, g))
        ws.append(w)
    et, ep = synth.embeddings(V, s + n + 1, h1, g)
    ones = torch.ones(h1, dtype=torch.float16, device=DEV)
    zeros = torch.zeros(h1, dtype=torch.float16, device=DEV)
    prompt = synth.token_ids((gbs * k, s), V, g).to(DEV)
    res = Model(LayerStack(_layers(ws, h1, H, h2), gbs, k, s + n + 1, DEV), et.to(DEV), ep.to(DEV),
                ones, zeros)
    hst = Model(HostLayerStack(_layers(ws, h1, H, h2), gbs, k, s + n + 1, DEV), et.to(DEV),
                ep.to(DEV), ones, zeros)
    assert all(getattr(L, "qkv") is None for L in hst.stack.layers)   # no device copy kept
    t1, l1 = res.generate_greedy(prompt, n, order=order, keep_logits=True)
    t2, l2 = hst.generate_greedy(prompt, n, order=order, keep_logits=True)
    fg.fg_check()
    assert torch.equal(t1, t2)
    for a, b in zip(l1, l2):
        assert torch.equal(a, b)


def test_host_streamed_model_logits_match_oracle():
    """The host-streamed model against the oracle directly (not only against
    the resident stack): 3 layers of h1 512 / 4 heads / h2 1024, vocab 700,
    gbs 2 x k 2, prompt 24, 4 teacher-forced decode steps, zig-zag order;
    logits every step within max-abs 1e-2 * max|ref|."""
    import numpy as np
    from oracle.model import OracleModel, generate
    from oracle.model import quantize_layer as oracle_layer
    from gpu_util import to_np
    h1, H, h2, V, gbs, k, s, D, nl = 512, 4, 1024, 700, 2, 2, 24, 4, 3
    g = synth.generator(301)
    ws = []
    for _ in range(nl):
        w = synth.layer_weights(h1, h2, g)
        w.update(synth.random_affine_params(h1, h2, g))
        ws.append(w)
    et, ep = synth.embeddings(V, s + D + 1, h1, g)
    lnf_g = (1 + synth.normal_f16((h1,), 0.1, g).float()).half()
    lnf_b = synth.normal_f16((h1,), 0.1, g)
    prompt = synth.token_ids((gbs * k, s), V, g)
    dec = synth.token_ids((gbs * k, D), V, g)
    hst = Model(HostLayerStack(_layers(ws, h1, H, h2), gbs, k, s + D + 1, DEV), et.to(DEV),
                ep.to(DEV), lnf_g.to(DEV), lnf_b.to(DEV))
    got = hst.generate(prompt.to(DEV), dec.t().contiguous().to(DEV), order="zigzag")
    fg.fg_check()
    om = OracleModel([oracle_layer({n: t.numpy() for n, t in w.items()}, h1, H, h2) for w in ws],
                     et.numpy(), ep.numpy(), lnf_g.numpy(), lnf_b.numpy())
    ref = generate(om, prompt.numpy(), dec.numpy(), gbs, k, order="zigzag")
    for t, (a, b) in enumerate(zip(got, ref)):
        a = to_np(a)
        assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(b)), t
