"""Pins for the oracle's size formulas, layer composition and block orders.

Size formulas and worked numbers: "FlexGen 完全拆解" (M_W = l(8h1^2+4h1h2),
M_KV = 4blh1(s+n); OPT-175B about 325 GB of fp16 weights and about 1.2 TB of
KV at b=512, s=512, n=32, 3.8x the weights; 162.5 s to read 325 GB at 2 GB/s;
bls = gbs * number of GPU batches).  Block orders: batches are independent,
so row-by-row, zig-zag and whole-block orders must agree bit for bit.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.model import (DECODE, PREFILL, OracleModel, generate, generate_greedy,
                          layer_step, quantize_layer)

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def _np(d):
    return {k: v.numpy() for k, v in d.items()}


# ------------------------------------------------------------------ sizes

@pytest.mark.parametrize("w", list(synth.WORKLOADS.values()))
def test_m_w_is_exact_fp16_allocation(w):
    """M_W equals the byte count of the six fp16 projection matrices."""
    shapes = [(3 * w.h1, w.h1), (w.h1, w.h1), (w.h2, w.h1), (w.h1, w.h2)]
    per_layer = sum(2 * a * b for a, b in shapes)
    assert oracle.size_m_w(w.layers, w.h1, w.h2) == w.layers * per_layer


@pytest.mark.parametrize("w", list(synth.WORKLOADS.values()))
def test_m_kv_is_exact_fp16_allocation(w):
    """M_KV equals K plus V, fp16, [b][l][s+n][h1] each."""
    b = w.bls
    alloc = 2 * (2 * b * w.layers * w.cap * w.h1)
    assert oracle.size_m_kv(b, w.layers, w.h1, w.s, w.n) == alloc


def test_q4_size_per_layer():
    # 0.5 byte per element plus 8 bytes per group of 64
    assert oracle.size_q4(768, 768) == 768 * 384 + 768 * 12 * 8
    w = synth.OPT125M_LAYER
    per_layer = sum(oracle.size_q4(r, c) for r, c in
                    [(3 * w.h1, w.h1), (w.h1, w.h1), (w.h2, w.h1), (w.h1, w.h2)])
    assert per_layer == 4_423_680


def test_pages_175b_examples():
    g = GOLD["opt175b_shape"]
    mw = oracle.size_m_w(g["l"], g["h1"], g["h2"])
    assert abs(mw - g["fp16_weight_bytes_about"]) / g["fp16_weight_bytes_about"] < g["rel_tol"]
    k = GOLD["opt175b_kv_example"]
    mkv = oracle.size_m_kv(k["b"], g["l"], g["h1"], k["s"], k["n"])
    assert abs(mkv - k["kv_bytes_about"]) / k["kv_bytes_about"] < k["rel_tol"]
    assert abs(mkv / mw - k["kv_over_weights_about"]) < 0.05
    e = GOLD["ssd_read_example"]
    assert e["bytes"] / e["bandwidth"] == e["seconds"]


def test_block_sizes():
    for gbs, k, bls in GOLD["block_sizes"]["cases"]:
        assert gbs * k == bls
    assert synth.OPT30B.bls == 144 and synth.OPT6_7B.bls == 256


# ------------------------------------------------------------------ layer / model

def _tiny_model(seed=0, layers=2, h1=128, H=2, h2=256, V=300, P=16):
    g = synth.generator(seed)
    ls = []
    for _ in range(layers):
        w = synth.layer_weights(h1, h2, g)
        w.update(synth.random_affine_params(h1, h2, g))
        ls.append(quantize_layer(_np(w), h1, H, h2))
    et, ep = synth.embeddings(V, P, h1, g)
    return OracleModel(ls, et.numpy(), ep.numpy(), np.ones(h1, np.float16),
                       np.zeros(h1, np.float16))


def test_block_orders_identical():
    m = _tiny_model()
    g = synth.generator(1)
    gbs, k, s, D = 2, 3, 5, 3
    prompt = synth.token_ids((gbs * k, s), 300, g).numpy()
    dec = synth.token_ids((gbs * k, D), 300, g).numpy()
    a = generate(m, prompt, dec, gbs, k, order="row")
    b = generate(m, prompt, dec, gbs, k, order="zigzag")
    c = generate(m, prompt, dec, gbs, k, order="block")
    assert len(a) == D + 1                    # prefill token + D decode steps
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y) and np.array_equal(x, z)
        assert np.all(np.isfinite(x))


def test_sequences_independent():
    """A sequence's logits do not depend on the other sequences of its block."""
    m = _tiny_model(seed=3, layers=1)
    g = synth.generator(4)
    prompt = synth.token_ids((4, 6), 300, g).numpy()
    dec = synth.token_ids((4, 2), 300, g).numpy()
    full = generate(m, prompt, dec, 4, 1, order="block")
    one = generate(m, prompt[2:3], dec[2:3], 1, 1, order="block")
    for x, y in zip(full, one):
        assert np.array_equal(x[2:3], y)


def _layer_fp64(L, x):
    """Textbook OPT pre-LN layer in fp64 on the dequantised weights, for a
    prefill of one sequence (no fp16 rounding anywhere)."""
    deq = lambda cm: oracle.dequant_g4(*cm).astype(np.float64)
    def ln(v, g, b):
        mu = v.mean(-1, keepdims=True)
        var = ((v - mu) ** 2).mean(-1, keepdims=True)
        return (v - mu) / np.sqrt(var + L.eps) * g.astype(np.float64) + b.astype(np.float64)
    s = x.shape[0]
    d = L.d
    a = ln(x, L.ln1_g, L.ln1_b)
    qkv = a @ deq(L.qkv).T + L.b_qkv.astype(np.float64)
    q, k, v = np.split(qkv, 3, axis=1)
    o = np.zeros_like(q)
    for h in range(L.H):
        sl = slice(h * d, (h + 1) * d)
        sc = q[:, sl] @ k[:, sl].T / np.sqrt(d)
        sc = np.where(np.tril(np.ones((s, s), bool)), sc, -np.inf)
        p = np.exp(sc - sc.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o[:, sl] = p @ v[:, sl]
    h_ = x + o @ deq(L.out).T + L.b_out.astype(np.float64)
    u = np.maximum(ln(h_, L.ln2_g, L.ln2_b) @ deq(L.fc1).T + L.b_fc1.astype(np.float64), 0)
    return h_ + u @ deq(L.fc2).T + L.b_fc2.astype(np.float64)


def test_layer_h1_64_matches_textbook_fp64():
    g = synth.generator(5)
    h1, H, h2, s = 64, 1, 128, 10
    w = synth.layer_weights(h1, h2, g, std=0.2)
    w.update(synth.random_affine_params(h1, h2, g))
    L = quantize_layer(_np(w), h1, H, h2)
    x = synth.normal_f16((s, h1), 1.0, g).numpy()
    cache = oracle.KVCache(1, H, h1 // H, s + 1)
    y = layer_step(L, x, cache, PREFILL, 1, s).astype(np.float64)
    ref = _layer_fp64(L, x.astype(np.float64))
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 5e-3


def test_decode_step_extends_prefill():
    """Prefill of s tokens then one decode step equals (in the attention
    sense) a prefill of s+1 tokens, up to the 4-bit cache: the decode output
    stays within the 4-bit quantisation error of the s+1 prefill's last row."""
    g = synth.generator(6)
    h1, H, h2, s = 128, 2, 256, 9
    w = synth.layer_weights(h1, h2, g)
    L = quantize_layer(_np(w), h1, H, h2)
    x = synth.normal_f16((s + 1, h1), 1.0, g).numpy()
    c1 = oracle.KVCache(1, H, h1 // H, s + 2)
    layer_step(L, x[:s], c1, PREFILL, 1, s)
    yd = layer_step(L, x[s:], c1, DECODE, 1, 1, pos=s).astype(np.float64)
    c2 = oracle.KVCache(1, H, h1 // H, s + 2)
    yp = layer_step(L, x, c2, PREFILL, 1, s + 1)[-1:].astype(np.float64)
    rel = np.linalg.norm(yd - yp) / np.linalg.norm(yp)
    assert rel < 2e-2


# ------------------------------------------------------------------ padding and greedy

@pytest.mark.parametrize("order", ["row", "zigzag", "block"])
def test_padded_prompt_equals_unpadded_run(order):
    """Left padding reaches no real token: a prompt padded inside a block of
    longer prompts gives, bit for bit, the logits (teacher-forced) and the
    tokens (greedy) of the same prompt run alone at its own length."""
    m = _tiny_model(seed=7)
    g = synth.generator(8)
    gbs, k, s, D = 2, 2, 9, 3
    pad = np.array([0, 4, 8, 1], np.int32)
    prompt = synth.token_ids((gbs * k, s), 300, g).numpy()
    dec = synth.token_ids((gbs * k, D), 300, g).numpy()
    full = generate(m, prompt, dec, gbs, k, order=order, pad=pad)
    toks, glog = generate_greedy(m, prompt, D + 1, gbs, k, order=order, pad=pad)
    for b in range(gbs * k):
        p0 = pad[b]
        one = generate(m, prompt[b:b + 1, p0:], dec[b:b + 1], 1, 1, order="block")
        for x, y in zip(full, one):
            assert np.array_equal(x[b:b + 1], y)
        t1, _ = generate_greedy(m, prompt[b:b + 1, p0:], D + 1, 1, 1, order="block")
        assert np.array_equal(toks[b:b + 1], t1)


def test_greedy_feeds_back_its_argmax():
    """Greedy tokens are the argmax of each step's logits, and feeding them
    back teacher-forced reproduces the same logits."""
    m = _tiny_model(seed=9)
    g = synth.generator(10)
    gbs, k, s, n = 3, 2, 6, 4
    prompt = synth.token_ids((gbs * k, s), 300, g).numpy()
    pad = np.array([0, 2, 5, 0, 3, 1], np.int32)
    toks, logits = generate_greedy(m, prompt, n, gbs, k, order="zigzag", pad=pad)
    assert toks.shape == (gbs * k, n)
    for t in range(n):
        assert np.array_equal(toks[:, t], np.argmax(logits[t], axis=1))
    tf = generate(m, prompt, toks[:, :n - 1], gbs, k, order="block", pad=pad)
    for x, y in zip(logits, tf):
        assert np.array_equal(x, y)
