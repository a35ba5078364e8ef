"""Per-workload parity of the whole models against the oracle, at full size.

* OPT-1.3B shape (24 layers, vocab 50272), gbs 16, prompt 512, 32 tokens:
  teacher-forced logits of sampled sequences at every one of the 32 steps
  within max-abs 1e-2 * max|ref| (the oracle runs the sampled sequences
  alone: sequences never mix, which the block-order tests prove bit for bit).
* OPT-6.7B (gbs 32 x k 8 = 256) and OPT-30B (gbs 48 x k 3 = 144) shapes,
  prompt 512: the full model runs on the GPU; at layers 0 and l-1 the oracle
  takes the GPU's inputs of that layer for 2 sampled sequences (hidden
  states, and for a decode step the cache rows it attends over), runs the
  prefill and two decode steps, and the GPU's output hidden states match at
  relative L2 <= 5e-3.

The dataflow follows "FlexGen 完全拆解" (section 从 Transformer 推理的数据流重新
定义卸载: prefill over the prompt, then one new row per decode step), with
the pages' synthetic workload of 512-token inputs and 32 generated tokens
(section on reading the experimental results).
"""
import numpy as np
import pytest
import torch

import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, Model, quantize_layer
from oracle import KVCache
from oracle.model import DECODE, PREFILL, OracleModel, generate, layer_step
from oracle.model import quantize_layer as oracle_layer

from gpu_util import DEV, rel_l2, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _build(wl, seed, keep=()):
    """Seeded layers of workload wl, quantised on the GPU; the fp16 weights
    of the layers in `keep` are returned as numpy for the oracle."""
    g = synth.generator(seed, DEV)
    layers, kept = [], {}
    for j in range(wl.layers):
        w = synth.layer_weights(wl.h1, wl.h2, g, DEV)
        if j in keep:
            kept[j] = {n: to_np(t) for n, t in w.items()}
        layers.append(quantize_layer(w, wl.h1, wl.H, wl.h2))
        del w
    e_tok, e_pos = synth.embeddings(wl.vocab, wl.cap, wl.h1, g, DEV)
    return layers, kept, e_tok, e_pos, g


def test_opt13b_full_model_teacher_forced_logits_sampled():
    wl = synth.OPT1_3B
    keep = tuple(range(wl.layers))
    layers, kept, e_tok, e_pos, g = _build(wl, 1300, keep)
    ones = torch.ones(wl.h1, dtype=torch.float16, device=DEV)
    zeros = torch.zeros(wl.h1, dtype=torch.float16, device=DEV)
    prompt = synth.token_ids((wl.bls, wl.s), wl.vocab, g, DEV)
    dec = synth.token_ids((wl.decode_steps, wl.bls), wl.vocab, g, DEV)   # time-major
    m = Model(LayerStack(layers, wl.gbs, wl.k, wl.cap, DEV), e_tok, e_pos, ones, zeros)
    seqs = [3, 14]
    got = [to_np(lg[seqs]) for lg in m.generate(prompt, dec)]
    fg.fg_check()
    assert len(got) == wl.n
    del m, layers
    torch.cuda.empty_cache()
    om = OracleModel([oracle_layer(kept[j], wl.h1, wl.H, wl.h2) for j in keep],
                     to_np(e_tok), to_np(e_pos), to_np(ones), to_np(zeros))
    ref = generate(om, to_np(prompt[seqs]), to_np(dec[:, seqs]).T, len(seqs), 1, order="block")
    for t, (a, b) in enumerate(zip(got, ref)):
        assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(b)), t


def _layer_inputs_outputs(wl, seed, n_decode=2):
    """Runs the full model on the GPU (prefill of the whole block, then
    n_decode teacher-forced decode steps, block order), keeping for layers 0
    and l-1 and sequences 0 and bls-1: the input and output hidden states of
    every step and, before each decode step, the 4-bit cache rows the layer
    is about to attend over (the layer's other input)."""
    last = wl.layers - 1
    layers, kept, e_tok, e_pos, g = _build(wl, seed, keep=(0, last))
    stack = LayerStack(layers, wl.gbs, wl.k, wl.cap, DEV)
    pol = stack.policy(fg.FG_ORDER_BLOCK)
    seqs = [0, wl.bls - 1]
    rec = {0: [], last: []}
    prompt = synth.token_ids((wl.bls, wl.s), wl.vocab, g, DEV)

    def run(x, phase, T, pos):
        ws = stack.workspace(phase, T, fg.FG_ORDER_BLOCK)
        cur, nxt = x, torch.empty_like(x)
        for j, Lc in enumerate(stack.c_layers):
            snap = None
            if j in rec and phase == fg.FG_PHASE_DECODE:
                c = stack.caches[j]
                snap = {n: to_np(getattr(c, n)[seqs, :, :pos])
                        for n in ("k_codes", "k_meta", "v_codes", "v_meta")}
            fg.fg_layer_step(Lc, stack.caches[j], cur, nxt, phase, T, pos, pol, ws)
            if j in rec:
                rows = lambda t: to_np(t.view(wl.bls, T, wl.h1)[seqs]).reshape(-1, wl.h1)
                rec[j].append((rows(cur), rows(nxt), snap))
            cur, nxt = nxt, cur

    x = fg.fg_embed(prompt.reshape(-1), wl.s, 0, e_tok, e_pos)
    run(x, fg.FG_PHASE_PREFILL, wl.s, 0)
    for t in range(1, n_decode + 1):
        ids = synth.token_ids((wl.bls,), wl.vocab, g, DEV)
        run(fg.fg_embed(ids, 1, wl.s + t - 1, e_tok, e_pos), fg.FG_PHASE_DECODE, 1, wl.s + t - 1)
    fg.fg_check()
    del stack, layers
    torch.cuda.empty_cache()
    return kept, rec, len(seqs)


@pytest.mark.parametrize("wl", [synth.OPT6_7B, synth.OPT30B], ids=["opt-6.7b", "opt-30b"])
def test_first_and_last_layer_prefill_and_decode_sampled(wl):
    """Each step of the layer gets, on both sides, the same inputs: the GPU's
    input hidden states and, for a decode step, the GPU's cache rows (the
    prefill attends over its own fresh fp16 K/V).  Feeding the oracle its own
    cache instead would compare the 4-bit codes of two slightly different
    fp16 K/V computations, where a one-ulp difference can move a code by a
    whole quantisation step."""
    kept, rec, B = _layer_inputs_outputs(wl, 670 if wl is synth.OPT6_7B else 3000)
    for j, steps in rec.items():
        ol = oracle_layer(kept[j], wl.h1, wl.H, wl.h2)
        for t, (x_in, y_gpu, snap) in enumerate(steps):
            cache = KVCache(B, wl.H, wl.d, wl.cap)
            if t == 0:
                ref = layer_step(ol, x_in, cache, PREFILL, B, wl.s)
            else:
                pos = wl.s + t - 1
                for n, a in snap.items():
                    getattr(cache, n)[:, :, :pos] = a
                ref = layer_step(ol, x_in, cache, DECODE, B, 1, pos=pos)
            assert rel_l2(y_gpu, ref) <= 5e-3, (j, t, rel_l2(y_gpu, ref))
