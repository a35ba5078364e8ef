"""OPT decoder driver over libfg: weights stored 4-bit and resident in HBM,
a 4-bit KV cache, and generation under the block schedule.

Torch supplies device memory, streams and the synthetic inputs; every step
of prefill and decode is a libfg call (embedding, layer steps, final
LayerNorm, LM head).  Schedule ("FlexGen 完全拆解", computation-graph
section): for each token step and each layer, the k GPU batches of the block
pass through that layer's weights before the next layer; with order "block"
the k batches are one launch per projection (weights read once per block),
with order "zigzag" they are k launches whose order reverses at every token
step.  The first generated token comes from the prefill, so n tokens take
n-1 decode steps.

Prompts of different lengths share a block by left padding to the common
length s (pad: int32 [bls] counts on the device); positions count from each
prompt's first real slot and the attention kernels mask the padding, so a
padded prompt gives the results of the same prompt run alone.  Greedy
generation feeds back fg_argmax of each step's logits without leaving the
device.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import fg
import synth


@dataclass
class Layer:
    qkv: fg.Q4
    out: fg.Q4
    fc1: fg.Q4
    fc2: fg.Q4
    b_qkv: torch.Tensor
    b_out: torch.Tensor
    b_fc1: torch.Tensor
    b_fc2: torch.Tensor
    ln1_g: torch.Tensor
    ln1_b: torch.Tensor
    ln2_g: torch.Tensor
    ln2_b: torch.Tensor
    h1: int
    H: int
    h2: int
    eps: float = 1e-5

    def c(self) -> fg.c_layer:
        p = lambda t: t.data_ptr()
        return fg.c_layer(self.qkv.c(), self.out.c(), self.fc1.c(), self.fc2.c(),
                          p(self.b_qkv), p(self.b_out), p(self.b_fc1), p(self.b_fc2),
                          p(self.ln1_g), p(self.ln1_b), p(self.ln2_g), p(self.ln2_b),
                          self.h1, self.H, self.h2, self.eps)

    @property
    def nbytes_q4(self):
        return self.qkv.nbytes + self.out.nbytes + self.fc1.nbytes + self.fc2.nbytes


def quantize_layer(w: dict, h1: int, H: int, h2: int, eps: float = 1e-5) -> Layer:
    """w: fp16 CUDA tensors (torch Linear layout).  The projections are
    quantised on the GPU by fg_quantize_g4; the fp16 copies can be dropped."""
    q = lambda name: fg.fg_quantize_g4(w[name].contiguous())
    c = lambda name: w[name].contiguous()
    return Layer(q("w_qkv"), q("w_out"), q("w_fc1"), q("w_fc2"), c("b_qkv"), c("b_out"),
                 c("b_fc1"), c("b_fc2"), c("ln1_g"), c("ln1_b"), c("ln2_g"), c("ln2_b"),
                 h1, H, h2, eps)


def order_for(step: int, order: str) -> int:
    if order == "block":
        return fg.FG_ORDER_BLOCK
    if order == "batches":
        return fg.FG_ORDER_BATCHES
    if order == "zigzag":
        return fg.FG_ORDER_BATCHES if step % 2 == 0 else fg.FG_ORDER_BATCHES_REV
    raise ValueError(order)


class LayerStack:
    """l decoder layers with their KV caches and one shared workspace for a
    block of bls = gbs * k sequences.  topk_pct: 0 for dense decode
    attention, 1..99 for top-K sparse decode attention keeping that percent
    of the cached rows' V (the prefill stays dense)."""

    topk_pct = 0

    def __init__(self, layers, gbs: int, k: int, cap: int, device="cuda", kv="g4"):
        self.layers = layers
        self.c_layers = [L.c() for L in layers]
        self.gbs, self.k, self.cap = gbs, k, cap
        L0 = layers[0]
        self.h1, self.H, self.h2 = L0.h1, L0.H, L0.h2
        self.d = self.h1 // self.H
        self.device = device
        self.kv = kv
        self.caches = [self.new_cache(cap, device) for _ in layers]
        self._ws = {}

    @property
    def bls(self):
        return self.gbs * self.k

    def new_cache(self, cap, device):
        """kv "g4": the 4-bit cache; "f16": the uncompressed one (the A/B)."""
        cls = fg.KV16 if self.kv == "f16" else fg.KV4
        return cls.empty(self.bls, self.H, self.d, cap, device)

    def policy(self, order_code: int) -> fg.c_policy:
        return fg.c_policy(self.gbs, self.k, order_code, self.topk_pct)

    def workspace(self, phase, T, order_code):
        key = (phase, T, order_code != fg.FG_ORDER_BLOCK, self.topk_pct)
        if key not in self._ws:
            n = fg.fg_layer_workspace_bytes(self.c_layers[0], phase, self.bls, T,
                                            self.policy(order_code), cap=self.cap)
            self._ws[key] = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def run(self, x, phase, T, pos, order_code, out=None, stream=None, pad=None):
        """x: [bls*T][h1] fp16 -> hidden states after every layer.  pad: None
        or int32 [bls] left-padding counts on the device."""
        ws = self.workspace(phase, T, order_code)
        pol = self.policy(order_code)
        bufs = [out if out is not None else torch.empty_like(x), torch.empty_like(x)]
        n = len(self.c_layers)
        cur = x
        for j, Lc in enumerate(self.c_layers):
            nxt = bufs[(n - 1 - j) % 2]        # the last layer writes bufs[0]
            fg.fg_layer_step(Lc, self.caches[j], cur, nxt, phase, T, pos, pol, ws, stream,
                             pad=pad)
            cur = nxt
        return cur


class Model:
    """Embeddings + LayerStack + final LayerNorm + LM head tied to the token
    embedding (fp16, not quantised: the size formula M_W leaves the small
    embedding out)."""

    def __init__(self, stack: LayerStack, e_tok, e_pos, lnf_g, lnf_b, eps=1e-5):
        self.stack = stack
        self.e_tok, self.e_pos = e_tok, e_pos
        self.lnf_g, self.lnf_b, self.eps = lnf_g, lnf_b, eps
        self.vocab = e_tok.shape[0]

    def head(self, x, rows, x_ld, logits=None, stream=None):
        h = fg.fg_layernorm(x, self.lnf_g, self.lnf_b, self.eps, rows=rows, x_ld=x_ld,
                            stream=stream)
        return fg.fg_gemm_f16_f32out(h, self.e_tok, Y=logits, stream=stream)

    def prefill(self, prompt_ids, order="block", logits=None, stream=None, pad=None):
        """prompt_ids: int32 CUDA [bls][s] (left-padded by pad, int32 CUDA [bls]
        or None).  Returns fp32 logits [bls][V] of the last prompt slot (the
        first generated token)."""
        bls, s = prompt_ids.shape
        x = fg.fg_embed(prompt_ids.reshape(-1), s, 0, self.e_tok, self.e_pos, stream=stream,
                        pad=pad)
        y = self.stack.run(x, fg.FG_PHASE_PREFILL, s, 0, order_for(0, order), stream=stream,
                           pad=pad)
        last = y[s - 1:]          # row b of the view starts at (b*s + s-1) * h1
        return self.head(last, bls, s * self.stack.h1, logits=logits, stream=stream)

    def decode_step(self, ids, t, s, order="block", logits=None, stream=None, pad=None):
        """ids: int32 CUDA [bls], fed at slot s+t-1 (decode step t >= 1)."""
        pos = s + t - 1
        x = fg.fg_embed(ids, 1, pos, self.e_tok, self.e_pos, stream=stream, pad=pad)
        y = self.stack.run(x, fg.FG_PHASE_DECODE, 1, pos, order_for(t, order), stream=stream,
                           pad=pad)
        return self.head(y, ids.shape[0], self.stack.h1, logits=logits, stream=stream)

    def capture_decode_steps(self, toks, s, logits, order="block", pad=None, steps=None):
        """One CUDA graph per greedy decode step t = 1..D (D = toks.shape[0]-1,
        or `steps`): the embedding of toks[t-1] at slot s+t-1, every layer
        step, the final LayerNorm, the LM head into logits[t % 2] and
        fg_argmax into toks[t] -- the launches decode_step and fg_argmax make,
        recorded once and replayed without host work.  A step's slot (pos) is
        a launch argument, so each step has its own graph.  Replays compute
        exactly what the eager calls compute (same kernels, arguments and
        buffers); the workspaces must already exist (run one eager step
        first).  HBM-resident weights only."""
        if isinstance(self.stack, HostLayerStack):
            raise ValueError("decode graphs need the HBM-resident stack")
        D = toks.shape[0] - 1 if steps is None else steps
        graphs = []
        side = torch.cuda.Stream(toks.device)
        side.wait_stream(torch.cuda.current_stream(toks.device))
        for t in range(1, D + 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                lg = self.decode_step(toks[t - 1], t, s, order, logits=logits[t % 2], pad=pad)
                fg.fg_argmax(lg, out=toks[t])
            graphs.append(g)
        torch.cuda.current_stream(toks.device).wait_stream(side)
        return graphs

    def generate(self, prompt_ids, decode_ids_tm, order="block", stream=None, pad=None):
        """Teacher-forced generation.  prompt_ids: int32 [bls][s]; decode_ids_tm:
        int32 [D][bls] (time-major, row t-1 fed at decode step t).  Returns
        [logits of the prefill] + [logits of decode step t for t = 1..D], each
        fp32 [bls][V] on the device."""
        s = prompt_ids.shape[1]
        out = [self.prefill(prompt_ids, order, stream=stream, pad=pad)]
        for t in range(1, decode_ids_tm.shape[0] + 1):
            out.append(self.decode_step(decode_ids_tm[t - 1], t, s, order, stream=stream,
                                        pad=pad))
        return out

    def generate_greedy(self, prompt_ids, n_new, order="block", stream=None, pad=None,
                        keep_logits=False):
        """Greedy generation of n_new tokens per sequence: token 1 is
        fg_argmax of the prefill's logits, token t+1 fg_argmax of decode step
        t's logits, fed back at step t; nothing leaves the device.  Returns
        (tokens int32 [n_new][bls] time-major on the device, the list of
        logits per step if keep_logits else None)."""
        bls, s = prompt_ids.shape
        toks = torch.empty((n_new, bls), dtype=torch.int32, device=prompt_ids.device)
        keep = [] if keep_logits else None
        lg = self.prefill(prompt_ids, order, stream=stream, pad=pad)
        fg.fg_argmax(lg, out=toks[0], stream=stream)
        if keep is not None:
            keep.append(lg)
        for t in range(1, n_new):
            lg = self.decode_step(toks[t - 1], t, s, order, stream=stream, pad=pad,
                                  logits=None if keep is not None else lg)
            fg.fg_argmax(lg, out=toks[t], stream=stream)
            if keep is not None:
                keep.append(lg)
        return toks, keep


def random_layers(wl, gen, device="cuda", affine=False, n_layers=None):
    """Random fp16 weights ~N(0, 0.02) per layer, quantised at once on the GPU
    so the fp16 copy of the whole model never exists."""
    layers = []
    for _ in range(wl.layers if n_layers is None else n_layers):
        w = synth.layer_weights(wl.h1, wl.h2, gen, device)
        if affine:
            w.update(synth.random_affine_params(wl.h1, wl.h2, gen, device))
        layers.append(quantize_layer(w, wl.h1, wl.H, wl.h2))
        del w
    return layers


def random_model(wl, seed=0, device="cuda", n_layers=None, cap=None, host_weights=False,
                 kv="g4"):
    """host_weights: keep the 4-bit weights in pinned host memory and stream
    them one layer ahead (HostLayerStack).  kv: "g4" (4-bit KV cache) or
    "f16" (uncompressed)."""
    gen = synth.generator(seed, device)
    layers = random_layers(wl, gen, device, n_layers=n_layers)
    cls = HostLayerStack if host_weights else LayerStack
    stack = cls(layers, wl.gbs, wl.k, cap or wl.cap, device, kv=kv)
    e_tok, e_pos = synth.embeddings(wl.vocab, wl.cap, wl.h1, gen, device)
    ones = torch.ones(wl.h1, dtype=torch.float16, device=device)
    zeros = torch.zeros(wl.h1, dtype=torch.float16, device=device)
    return Model(stack, e_tok, e_pos, ones, zeros)


class HostLayerStack(LayerStack):
    """A LayerStack whose 4-bit weights live in pinned host memory and are
    streamed to the GPU one layer ahead ("FlexGen 完全拆解", section on how
    the three data paths overlap: while the k batches of a block run on layer
    j, the weights of layer j+1 are fetched; the weight-read bound per
    sequence is W / (B beta), section on the problem).

    Each layer's four projections (codes and min/scale pairs) are packed into
    one pinned host buffer, at 1 KB-aligned offsets, so that a fetch is a
    single asynchronous copy.  Two device buffers of that size form a ring.
    A copy stream fetches the next layer into the buffer the previous layer
    released: each copy waits for the compute that last read its buffer, and
    each layer's compute waits for its copy.  The last layer's successor is
    layer 0 of the next token step, so the fetch runs across step boundaries
    too.  Biases, LayerNorm parameters and the KV cache stay on the device.
    Results are bit-identical to the resident stack (same kernels, same
    bytes)."""

    NAMES = ("qkv", "out", "fc1", "fc2")
    ALIGN = 1024

    @classmethod
    def _layout(cls, L0):
        """(name, codes offset, meta offset, rows, cols) per projection, and
        the packed size in bytes."""
        lay, off = [], 0
        up = lambda v: (v + cls.ALIGN - 1) // cls.ALIGN * cls.ALIGN
        for nm in cls.NAMES:
            q = getattr(L0, nm)
            oc = off
            om = up(oc + q.codes.numel())
            off = up(om + q.meta.numel() * 4)
            lay.append((nm, oc, om, q.rows, q.cols))
        return lay, off

    @staticmethod
    def _views(buf, lay):
        out = {}
        for nm, oc, om, rows, cols in lay:
            codes = buf[oc:oc + rows * cols // 2].view(rows, cols // 2)
            meta = buf[om:om + rows * cols // 64 * 8].view(torch.float32).view(rows, cols // 64, 2)
            out[nm] = fg.Q4(codes, meta, rows, cols)
        return out

    def __init__(self, layers, gbs: int, k: int, cap: int, device="cuda", kv="g4"):
        L0 = layers[0]
        self.layout, self.bytes_per_layer = self._layout(L0)
        # host copies of the quantised projections, one pinned buffer per
        # layer; the device copies are dropped
        self.host = []
        for L in layers:
            hb = torch.empty(self.bytes_per_layer, dtype=torch.uint8).pin_memory()
            hv = self._views(hb, self.layout)
            for nm in self.NAMES:
                hv[nm].codes.copy_(getattr(L, nm).codes)
                hv[nm].meta.copy_(getattr(L, nm).meta)
                setattr(L, nm, None)
            self.host.append(hb)
        self.layers = list(layers)
        self.dev = [torch.empty(self.bytes_per_layer, dtype=torch.uint8, device=device)
                    for _ in range(2)]
        self.buf = [self._views(b, self.layout) for b in self.dev]
        self.gbs, self.k, self.cap = gbs, k, cap
        self.h1, self.H, self.h2 = L0.h1, L0.H, L0.h2
        self.d = self.h1 // self.H
        self.device = device
        self.kv = kv
        self.caches = [self.new_cache(cap, device) for _ in layers]
        self._ws = {}
        self.copy_stream = torch.cuda.Stream(device)
        self.freed = [torch.cuda.Event(), torch.cuda.Event()]
        self.fetched = [torch.cuda.Event(), torch.cuda.Event()]
        self.next = None          # (layer, slot): the fetch already issued
        # the C layer descriptors, one per (layer, slot)
        self.c_slot = [[self._c_layer(j, s) for s in range(2)] for j in range(len(layers))]
        self.c_layers = None

    def _c_layer(self, j, slot):
        L = self.layers[j]
        b = self.buf[slot]
        p = lambda t: t.data_ptr()
        return fg.c_layer(b["qkv"].c(), b["out"].c(), b["fc1"].c(), b["fc2"].c(),
                          p(L.b_qkv), p(L.b_out), p(L.b_fc1), p(L.b_fc2),
                          p(L.ln1_g), p(L.ln1_b), p(L.ln2_g), p(L.ln2_b),
                          L.h1, L.H, L.h2, L.eps)

    def _fetch(self, j, slot):
        """Issue the copy of layer j's weights into device slot `slot`."""
        cp = self.copy_stream
        cp.wait_event(self.freed[slot])   # its last reader has finished
        with torch.cuda.stream(cp):
            self.dev[slot].copy_(self.host[j], non_blocking=True)
        self.fetched[slot].record(cp)

    def workspace(self, phase, T, order_code):
        key = (phase, T, order_code != fg.FG_ORDER_BLOCK, self.topk_pct)
        if key not in self._ws:
            n = fg.fg_layer_workspace_bytes(self.c_slot[0][0], phase, self.bls, T,
                                            self.policy(order_code), cap=self.cap)
            self._ws[key] = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def run(self, x, phase, T, pos, order_code, out=None, stream=None, pad=None):
        cs = stream if stream is not None else torch.cuda.current_stream()
        ws = self.workspace(phase, T, order_code)
        pol = self.policy(order_code)
        n = len(self.layers)
        bufs = [out if out is not None else torch.empty_like(x), torch.empty_like(x)]
        if self.next is None:
            self._fetch(0, 0)
            self.next = (0, 0)
        cur = x
        for j in range(n):
            lj, slot = self.next
            assert lj == j
            cs.wait_event(self.fetched[slot])
            nj = (j + 1) % n
            self._fetch(nj, 1 - slot)
            self.next = (nj, 1 - slot)
            nxt = bufs[(n - 1 - j) % 2]
            fg.fg_layer_step(self.c_slot[j][slot], self.caches[j], cur, nxt, phase, T, pos, pol,
                             ws, cs, pad=pad)
            self.freed[slot].record(cs)
            cur = nxt
        return cur
