"""Decode steps recorded as CUDA graphs (one per step: embedding, every
layer step, final LayerNorm, LM head, argmax) replay exactly what the eager
calls compute: greedy tokens and logits bit-identical, for the block and
zig-zag orders and with left-padded prompts."""
import pytest
import torch

import synth
from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import LayerStack, Model, quantize_layer

from gpu_util import DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("order,padded", [("block", False), ("zigzag", False), ("block", True)])
def test_decode_graph_replay_equals_eager(order, padded):
    h1, H, h2, V, gbs, k, s, n = 512, 4, 1024, 900, 3, 2, 40, 6
    g = synth.generator(500, DEV)
    layers = [quantize_layer(synth.layer_weights(h1, h2, g, DEV), h1, H, h2) for _ in range(3)]
    et, ep = synth.embeddings(V, s + n, h1, g, DEV)
    ones = torch.ones(h1, dtype=torch.float16, device=DEV)
    zeros = torch.zeros(h1, dtype=torch.float16, device=DEV)
    m = Model(LayerStack(layers, gbs, k, s + n, DEV), et, ep, ones, zeros)
    prompt = synth.token_ids((gbs * k, s), V, g, DEV)
    pad = synth.pad_counts(gbs * k, s, g, device=DEV) if padded else None
    logits = [torch.empty((gbs * k, V), dtype=torch.float32, device=DEV) for _ in range(2)]

    def prefill(toks):
        lg = m.prefill(prompt, order, logits=logits[0], pad=pad)
        fg.fg_argmax(lg, out=toks[0])

    toks_e = torch.empty((n, gbs * k), dtype=torch.int32, device=DEV)
    prefill(toks_e)
    kept = []
    for t in range(1, n):
        lg = m.decode_step(toks_e[t - 1], t, s, order, logits=logits[t % 2], pad=pad)
        fg.fg_argmax(lg, out=toks_e[t])
        kept.append(lg.clone())
    fg.fg_check()

    toks_g = torch.zeros_like(toks_e)
    graphs = m.capture_decode_steps(toks_g, s, logits, order, pad=pad)
    assert len(graphs) == n - 1
    for _ in range(2):                       # two generations in a row from the same graphs
        toks_g.zero_()
        prefill(toks_g)
        for t, gph in enumerate(graphs, start=1):
            gph.replay()
            torch.cuda.synchronize()
            assert torch.equal(logits[t % 2], kept[t - 1]), t
        fg.fg_check()
        assert torch.equal(toks_g, toks_e)


def test_split_tile_gemm_with_residual_graph_replay_bitwise():
    """A decode-regime projection whose weight tiles are split over clusters
    (the later parts meet behind flags tagged with the launch's epoch) and
    whose residual is staged by TMA, recorded in a CUDA graph: every replay
    (same tag) equals the eager result bit for bit, because the consumed
    flags are reset after use and each replay waits for its own parts."""
    M, N, K = 37, 1040, 512   # 9 weight tiles (1-CTA clusters), 18 units over 6 clusters
    g = synth.generator(600, DEV)
    x = synth.normal_f16((M, K), 1.0, g, DEV)
    w = synth.normal_f16((N, K), 0.02, g, DEV)
    b = synth.normal_f16((N,), 0.1, g, DEV)
    r = synth.normal_f16((M, N), 1.0, g, DEV)
    q = fg.fg_quantize_g4(w)
    ws = torch.empty(max(fg.fg_dequant_gemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device=DEV)
    eager = fg.fg_dequant_gemm_g4(x, q, bias=b, residual=r, workspace=ws)
    fg.fg_check()
    y = torch.empty_like(eager)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fg.fg_dequant_gemm_g4(x, q, bias=b, residual=r, Y=y, workspace=ws)
    for _ in range(3):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, eager)
    fg.fg_check()
