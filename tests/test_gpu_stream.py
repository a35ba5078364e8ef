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
