"""Decoder layer step and model under the block schedule, through the C ABI,
against the oracle; the block orders agree bit for bit on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, Model, quantize_layer
from oracle.model import DECODE, PREFILL, OracleModel, generate, layer_step
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, rel_l2, to_np

pytestmark = pytest.mark.gpu


def _layer(h1, H, h2, seed, affine=True):
    g = synth.generator(seed)
    w = synth.layer_weights(h1, h2, g)
    if affine:
        w.update(synth.random_affine_params(h1, h2, g))
    gl = quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2)
    ol = oracle_layer({n: t.numpy() for n, t in w.items()}, h1, H, h2)
    return gl, ol, g


@pytest.mark.parametrize("affine", [False, True])
def test_opt125m_layer_prefill_and_8_decode_steps(affine):
    """One OPT-125M-shaped layer (h1 768, 12 heads of 64, h2 3072), gbs 4,
    k 1, prompt 32, 8 teacher-forced decode steps, N(0,1) hidden inputs:
    per-step layer output relative L2 <= 5e-3 against the oracle."""
    wl = synth.OPT125M_LAYER
    gl, ol, g = _layer(wl.h1, wl.H, wl.h2, 0, affine)
    stack = LayerStack([gl], wl.gbs, wl.k, wl.cap, DEV)
    oc = oracle.KVCache(wl.bls, wl.H, wl.d, wl.cap)
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


def _stacks_run(order_codes, h1=256, H=4, h2=512, gbs=3, k=3, s=20, D=4):
    outs = []
    for oc_fn in order_codes:
        gl, _, g = _layer(h1, H, h2, 5)
        stack = LayerStack([gl, _layer(h1, H, h2, 6)[0]], gbs, k, s + D + 1, DEV)
        x = synth.normal_f16((gbs * k * s, h1), 1.0, synth.generator(9)).to(DEV)
        ys = [stack.run(x, fg.FG_PHASE_PREFILL, s, 0, oc_fn(0)).clone()]
        for t in range(1, D + 1):
            xt = synth.normal_f16((gbs * k, h1), 1.0, synth.generator(100 + t)).to(DEV)
            ys.append(stack.run(xt, fg.FG_PHASE_DECODE, 1, s + t - 1, oc_fn(t)).clone())
        outs.append(ys)
    torch.cuda.synchronize()
    return outs


def test_block_orders_bitwise_identical_on_gpu():
    block = lambda t: fg.FG_ORDER_BLOCK
    batches = lambda t: fg.FG_ORDER_BATCHES
    zigzag = lambda t: fg.FG_ORDER_BATCHES if t % 2 == 0 else fg.FG_ORDER_BATCHES_REV
    a, b, c = _stacks_run([block, batches, zigzag])
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y) and torch.equal(x, z)


def test_block_orders_identical_when_block_exceeds_one_token_tile():
    """gbs 64 x k 5 = 320 sequences, h1 256 / 4 heads / h2 1024: a decode
    block of 320 rows takes two token tiles, while each 64-row batch alone
    would fit one (where the K = 1024 projection splits K across CTAs).  The
    batches plan their split from the block, so all orders still agree bit
    for bit."""
    h1, H, h2, gbs, k, s = 256, 4, 1024, 64, 5, 8
    gl, _, g = _layer(h1, H, h2, 11)
    assert fg.fg_dequant_gemm_workspace_bytes(gbs, h1, h2) > 0      # split alone
    assert fg.fg_dequant_gemm_workspace_bytes(gbs * k, h1, h2) == 0
    x = synth.normal_f16((gbs * k * s, h1), 1.0, g).to(DEV)
    xs = [synth.normal_f16((gbs * k, h1), 1.0, g).to(DEV) for _ in range(2)]
    outs = []
    for order in (lambda t: fg.FG_ORDER_BLOCK, lambda t: fg.FG_ORDER_BATCHES,
                  lambda t: fg.FG_ORDER_BATCHES if t % 2 == 0 else fg.FG_ORDER_BATCHES_REV):
        stack = LayerStack([gl], gbs, k, s + 3, DEV)
        ys = [stack.run(x, fg.FG_PHASE_PREFILL, s, 0, order(0)).clone()]
        for t in (1, 2):
            ys.append(stack.run(xs[t - 1], fg.FG_PHASE_DECODE, 1, s + t - 1, order(t)).clone())
        outs.append(ys)
    fg.fg_check()
    for a, b, c in zip(*outs):
        assert torch.equal(a, b) and torch.equal(a, c)


def test_small_model_logits_match_oracle():
    """2 layers of h1 512 / 8 heads / h2 1024, vocab 1000, gbs 2 x k 2,
    prompt 24, 3 decode steps: teacher-forced logits every step within
    max-abs 1e-2 * max|ref|, for the block and zig-zag orders."""
    h1, H, h2, V, gbs, k, s, D = 512, 8, 1024, 1000, 2, 2, 24, 3
    g = synth.generator(21)
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
    ref = generate(om, prompt.numpy(), dec.numpy(), gbs, k, order="block")
    for order in ("block", "zigzag"):
        layers = [quantize_layer({n: t.to(DEV) for n, t in w.items()}, h1, H, h2) for w in ws]
        m = Model(LayerStack(layers, gbs, k, s + D + 1, DEV), et.to(DEV), ep.to(DEV),
                  lnf_g.to(DEV), lnf_b.to(DEV))
        got = m.generate(prompt.to(DEV), dec.t().contiguous().to(DEV), order=order)
        fg.fg_check()
        for t, (a, b) in enumerate(zip(got, ref)):
            a = to_np(a)
            assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(b)), (order, t)
