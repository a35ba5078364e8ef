"""Oracle OPT decoder layer, model, block schedules and size formulas.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every step calls the
plain C primitives of this package; the composition follows the pages:

* OPT pre-LN decoder layer: h = x + OutProj(Attn(LN1(x)));
  y = h + FC2(ReLU(FC1(LN2(h)))); q, k, v of head h are columns
  [h*d, (h+1)*d) of the three h1-wide blocks of the fused QKV projection.
* Prefill computes Q, K, V for all s prompt tokens and stores K, V; each
  decode step appends one K/V row per sequence and attends over s+t rows
  ("FlexGen 完全拆解", section on the inference dataflow).
* Block schedule ("FlexGen 完全拆解", section on the computation graph and
  the zig-zag block schedule): a block of bls = gbs * k sequences; one layer's
  weights stay loaded while the k GPU batches of the block pass through it,
  and the traversal direction reverses at each token boundary.  Row-by-row
  order runs one GPU batch through every layer and token before the next.
  Batches are independent, so all orders must give identical results.
* The first generated token comes out of the prefill, so n generated tokens
  take n-1 decode steps (T = l*T_pre + l*(n-1)*T_gen on the same page).
* Prompts of different lengths share one block by left padding to the
  common length s (the pages' workloads pad every prompt to 512 or 1024,
  "FlexGen 完全拆解", section on reading the
  experimental results).  The pages do not spell the
  masking out; the reading taken here: prompt b occupies slots pad[b]..s-1,
  its tokens take positions 0..s-1-pad[b] (decode step t: position
  s+t-1-pad[b]), every query attends only keys at slots >= pad[b] (and, in
  the prefill, <= its own slot), and queries in padding slots give zero
  attention output.  A padded prompt then yields exactly the results of the
  same prompt run unpadded.
* Greedy generation: the next token is the argmax of the logits, the lowest
  index among equal maxima.
* Size formulas on the same page: M_W = l(8 h1^2 + 4 h1 h2) bytes of fp16
  weights (embeddings ignored) and M_KV = 4 b l h1 (s + n) bytes of fp16 KV.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import (GROUP, KVCache, KVCache16, argmax, decode_attn_f16, decode_attn_g4, embed,
               kv_store_prefill, kv_store_prefill_f16,
               layernorm, linear_f16_f32out, linear_g4, prefill_attn,
               quantize_g4)

PREFILL, DECODE = 0, 1


# --------------------------------------------------------------------------
# sizes
# --------------------------------------------------------------------------

def size_m_w(l: int, h1: int, h2: int) -> int:
    """fp16 weight bytes of l decoder layers: l(8 h1^2 + 4 h1 h2)."""
    return l * (8 * h1 * h1 + 4 * h1 * h2)


def size_m_kv(b: int, l: int, h1: int, s: int, n: int) -> int:
    """fp16 K+V cache bytes at full length: 4 b l h1 (s + n)."""
    return 4 * b * l * h1 * (s + n)


def size_q4(rows: int, cols: int) -> int:
    """Bytes of a 4-bit group-quantised [rows][cols] tensor: half a byte per
    element plus (min, scale) fp32 per group of 64."""
    assert cols % GROUP == 0
    return rows * cols // 2 + rows * (cols // GROUP) * 8


# --------------------------------------------------------------------------
# layer
# --------------------------------------------------------------------------

@dataclass
class OracleLayer:
    h1: int
    H: int
    h2: int
    qkv: tuple      # (codes, meta) of W_qkv [3 h1][h1]
    out: tuple      # W_out [h1][h1]
    fc1: tuple      # W_fc1 [h2][h1]
    fc2: tuple      # W_fc2 [h1][h2]
    b_qkv: np.ndarray
    b_out: np.ndarray
    b_fc1: np.ndarray
    b_fc2: np.ndarray
    ln1_g: np.ndarray
    ln1_b: np.ndarray
    ln2_g: np.ndarray
    ln2_b: np.ndarray
    eps: float = 1e-5

    @property
    def d(self):
        return self.h1 // self.H


def quantize_layer(w: dict, h1: int, H: int, h2: int, eps: float = 1e-5) -> OracleLayer:
    """w: fp16 numpy arrays named w_qkv, w_out, w_fc1, w_fc2 (torch Linear
    layout [out][in]), b_*, ln1_g, ln1_b, ln2_g, ln2_b."""
    f16 = lambda a: np.ascontiguousarray(a, dtype=np.float16)
    return OracleLayer(
        h1=h1, H=H, h2=h2,
        qkv=quantize_g4(w["w_qkv"]), out=quantize_g4(w["w_out"]),
        fc1=quantize_g4(w["w_fc1"]), fc2=quantize_g4(w["w_fc2"]),
        b_qkv=f16(w["b_qkv"]), b_out=f16(w["b_out"]), b_fc1=f16(w["b_fc1"]),
        b_fc2=f16(w["b_fc2"]), ln1_g=f16(w["ln1_g"]), ln1_b=f16(w["ln1_b"]),
        ln2_g=f16(w["ln2_g"]), ln2_b=f16(w["ln2_b"]), eps=eps)


def layer_step(L: OracleLayer, x, cache: KVCache, phase: int, B: int, T: int,
               pos: int = 0, trace: dict | None = None, pad=None):
    """One decoder layer for B sequences of T new tokens each.

    x: fp16 [B*T][h1] (sequence-major rows).  PREFILL: T = s prompt tokens in
    slots 0..s-1.  DECODE: T = 1, the new token sits at cache slot pos.
    pad: None or [B] left-padding counts (attention sees slots >= pad[b]).
    """
    a = layernorm(x, L.ln1_g, L.ln1_b, L.eps)
    qkv = linear_g4(a, *L.qkv, bias=L.b_qkv)
    f16 = isinstance(cache, KVCache16)   # uncompressed cache (the A/B setting)
    if phase == PREFILL:
        attn = prefill_attn(qkv, B, T, L.H, L.d, pad=pad)
        (kv_store_prefill_f16 if f16 else kv_store_prefill)(qkv, B, T, cache)
    else:
        assert T == 1
        attn = (decode_attn_f16 if f16 else decode_attn_g4)(qkv, cache, pos, append=True, pad=pad)
    h = linear_g4(attn, *L.out, bias=L.b_out, residual=x)
    u = linear_g4(layernorm(h, L.ln2_g, L.ln2_b, L.eps), *L.fc1, bias=L.b_fc1, act=1)
    y = linear_g4(u, *L.fc2, bias=L.b_fc2, residual=h)
    if trace is not None:
        trace.update(ln1=a, qkv=qkv, attn=attn, h=h, u=u)
    return y


# --------------------------------------------------------------------------
# model and block schedules
# --------------------------------------------------------------------------

@dataclass
class OracleModel:
    layers: list
    e_tok: np.ndarray          # [V][h1] fp16, tied LM head
    e_pos: np.ndarray          # [P][h1] fp16
    lnf_g: np.ndarray
    lnf_b: np.ndarray
    eps: float = 1e-5
    caches: list = field(default_factory=list)

    @property
    def h1(self):
        return self.e_tok.shape[1]

    def new_caches(self, B, cap, kv="g4"):
        """kv "g4": the 4-bit cache; "f16": the uncompressed one."""
        L0 = self.layers[0]
        cls = KVCache16 if kv == "f16" else KVCache
        return [cls(B, L0.H, L0.d, cap) for _ in self.layers]

    def head(self, x):
        """Final LayerNorm then logits against the tied token embedding (fp32)."""
        return linear_f16_f32out(layernorm(x, self.lnf_g, self.lnf_b, self.eps),
                                 self.e_tok)


def _embed_rows(m: OracleModel, ids, positions):
    return embed(ids, positions, m.e_tok, m.e_pos)


def positions_of(slots, pad_b: int):
    """Positions of a sequence's slots under left padding by pad_b (padding
    slots take position 0; nothing real reads them)."""
    return np.maximum(np.asarray(slots, np.int64) - pad_b, 0).astype(np.int32)


def generate(m: OracleModel, prompt_ids, decode_ids, gbs: int, k: int,
             order: str = "zigzag", caches=None, pad=None):
    """Teacher-forced generation of a block of bls = gbs*k sequences.

    prompt_ids: int [bls][s]; decode_ids: int [bls][D] fed at decode steps
    1..D (slot s+t-1).  pad: None or int [bls] left-padding counts (prompt b
    is prompt_ids[b, pad[b]:]).  Returns the list of fp32 logits [bls][V]:
    entry 0 from the prefill's last slot, entry t from decode step t.

    order: "row" (one GPU batch through all layers and tokens, then the next),
    "zigzag" (per token step and layer, the k batches in turn, direction
    reversed on odd token steps) or "block" (per token step and layer, one
    call over all bls rows).  All three give identical logits.
    """
    decode_ids = np.asarray(decode_ids, np.int32)
    D = decode_ids.shape[1]
    return _run(m, prompt_ids, D, lambda t, prev, b0, b1: decode_ids[b0:b1, t - 1],
                gbs, k, order, caches, pad)


def generate_greedy(m: OracleModel, prompt_ids, n_new: int, gbs: int, k: int,
                    order: str = "zigzag", caches=None, pad=None):
    """Greedy generation of n_new tokens per sequence: token 1 is the argmax
    of the prefill's logits, token t+1 the argmax of decode step t's logits
    (fed back at step t).  Returns (tokens int32 [bls][n_new], logits list as
    generate() gives it)."""
    assert n_new >= 1
    out = _run(m, prompt_ids, n_new - 1, lambda t, prev, b0, b1: argmax(prev[b0:b1]),
               gbs, k, order, caches, pad)
    toks = np.stack([argmax(lg) for lg in out], axis=1).astype(np.int32)
    return toks, out


def _run(m: OracleModel, prompt_ids, D: int, ids_for_step, gbs: int, k: int,
         order: str, caches, pad):
    """Shared driver: ids_for_step(t, logits of step t-1, b0, b1) gives the
    ids of sequences [b0, b1) at decode step t."""
    prompt_ids = np.asarray(prompt_ids, np.int32)
    bls, s = prompt_ids.shape
    assert bls == gbs * k
    pad = np.zeros(bls, np.int32) if pad is None else np.asarray(pad, np.int32)
    assert pad.shape == (bls,) and np.all((pad >= 0) & (pad < s))
    cap = s + D + 1
    if caches is None:
        caches = m.new_caches(bls, cap)
    nl = len(m.layers)
    batches = [(i * gbs, (i + 1) * gbs) for i in range(k)]
    out = [np.zeros((bls, m.e_tok.shape[0]), np.float32) for _ in range(D + 1)]

    def prefill_rows(b0, b1):
        ids = prompt_ids[b0:b1].reshape(-1)
        pos = np.concatenate([positions_of(np.arange(s), pad[b]) for b in range(b0, b1)])
        return _embed_rows(m, ids, pos)

    def decode_rows(b0, b1, t):
        ids = np.asarray(ids_for_step(t, out[t - 1], b0, b1), np.int32)
        pos = np.array([s + t - 1 - pad[b] for b in range(b0, b1)], np.int32)
        return _embed_rows(m, ids, pos)

    def last_rows(x, nb):
        return x.reshape(nb, s, -1)[:, -1, :]

    if order == "row":
        for (b0, b1) in batches:
            pb = pad[b0:b1]
            x = prefill_rows(b0, b1)
            for j in range(nl):
                x = layer_step(m.layers[j], x, caches[j].view(b0, b1), PREFILL, b1 - b0, s,
                               pad=pb)
            out[0][b0:b1] = m.head(last_rows(x, b1 - b0))
            for t in range(1, D + 1):
                x = decode_rows(b0, b1, t)
                for j in range(nl):
                    x = layer_step(m.layers[j], x, caches[j].view(b0, b1), DECODE,
                                   b1 - b0, 1, pos=s + t - 1, pad=pb)
                out[t][b0:b1] = m.head(x)
        return out

    if order == "block":
        groups = [[(0, bls)]] * (D + 1)
    elif order == "zigzag":
        groups = [batches if t % 2 == 0 else batches[::-1] for t in range(D + 1)]
    else:
        raise ValueError(order)

    xs = {bb: prefill_rows(*bb) for bb in groups[0]}
    for j in range(nl):
        for bb in groups[0]:
            xs[bb] = layer_step(m.layers[j], xs[bb], caches[j].view(*bb), PREFILL,
                                bb[1] - bb[0], s, pad=pad[bb[0]:bb[1]])
    for (b0, b1) in groups[0]:
        out[0][b0:b1] = m.head(last_rows(xs[(b0, b1)], b1 - b0))
    for t in range(1, D + 1):
        xs = {bb: decode_rows(*bb, t) for bb in groups[t]}
        for j in range(nl):
            for bb in groups[t]:
                xs[bb] = layer_step(m.layers[j], xs[bb], caches[j].view(*bb), DECODE,
                                    bb[1] - bb[0], 1, pos=s + t - 1, pad=pad[bb[0]:bb[1]])
        for (b0, b1) in groups[t]:
            out[t][b0:b1] = m.head(xs[(b0, b1)])
    return out
