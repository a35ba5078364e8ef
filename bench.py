"""Benchmark: decode tokens/s of 4-bit group-quantised, block-scheduled OPT
generation on GB300, plus the dequant-GEMM TFLOP/s and 4-bit KV-attention
GB/s measured inside the same timed region.

One step = one whole pass of the hot path over one block: greedy generation
of n tokens per prompt -- prefill of bls prompts (embedding, every layer,
final LayerNorm, LM head, argmax) followed by n-1 decode steps, each fed the
previous step's argmax on the device.  Default workload: OPT-30B-shaped model
(48 layers, h1 7168, 56 heads, h2 28672, vocab 50272), gbs 48 x k 3 =
bls 144, s 512, n 32, weights and KV cache 4-bit g64, all resident in HBM.

`value` = bls * (n-1) / (device time of the decode phase), summed over
ranks over the max-over-ranks time.  Inputs (18.5 GB of weights, 33.7 GB of
KV cache) are far larger than L2, so no flush is needed between steps.

python bench.py [--steps K] [--warmup W] [--impl reference]
The product runs on one GPU: under torchrun with more than one rank it
prints an "unavailable" line and touches no GPU (the GEMM kernels' cluster
multicast loads stay in single-GPU runs; sequences are independent, so N
GPUs are N separate jobs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = ("decode tokens/s at bls=144,s=512,n=32; dequant-GEMM TFLOP/s; "
          "4-bit KV-attn GB/s")
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------
# distributed helpers (replicas: no collective on the data path)
# --------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_scalar(x: float, op: str, device="cpu") -> float:
    """Max or sum of one float over all ranks (identity with one process)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    rop = torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM
    torch.distributed.all_reduce(t, op=rop)
    return float(t.item())


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def aggregate(units_per_rank: float, seconds_per_rank: float, device="cpu"):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    units = reduce_scalar(units_per_rank, "sum", device)
    secs = reduce_scalar(seconds_per_rank, "max", device)
    return units / secs, secs


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------------------
# peaks and committed ncu traffic
# --------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def committed_traffic(kernel_file: str, workload: str):
    """Per-launch DRAM bytes of the kernel from profiles/traffic.json, valid
    only while the kernel source is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_file + ":" + workload)
    src = os.path.join(ROOT, "bit_group_quant_gb300", "csrc", kernel_file)
    if not d or d.get("source_sha") != kernel_hash(src):
        return None
    return d.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# CPU baseline (the oracle, as it stands, on a bounded sample)
# --------------------------------------------------------------------------

def oracle_sample(wl, nseq: int, seed: int = 0, frac: int = 16):
    """Time the oracle on a bounded sample of one decode token step: every
    projection of one layer on a 1/frac row slice of its weight, the decode
    attention of nseq sequences over all heads at context s+1 (cache of
    quantised N(0,1) rows), both LayerNorms, and a 1/frac slice of the LM
    head; the slices are scaled by frac and the layer by the layer count.
    Returns (decode tokens/s, seconds of CPU work, threads used)."""
    import oracle

    g = synth.generator(seed)
    h1, h2 = wl.h1, wl.h2
    shapes = [(3 * h1, h1), (h1, h1), (h2, h1), (h1, h2)]
    slices = []
    for n, k in shapes:
        w = synth.normal_f16((n // frac, k), 0.02, g).numpy()
        x = synth.normal_f16((nseq, k), 1.0, g).numpy()
        slices.append((x, oracle.quantize_g4(w)))
    cache = oracle.KVCache(nseq, wl.H, wl.d, wl.s + 1)
    rows = synth.normal_f16((2, nseq * wl.H * wl.s, wl.d), 1.0, g).numpy()
    kc, km = oracle.quantize_g4(rows[0])
    vc, vm = oracle.quantize_g4(rows[1])
    cache.k_codes[:, :, :wl.s] = kc.reshape(nseq, wl.H, wl.s, -1)
    cache.k_meta[:, :, :wl.s] = km.reshape(nseq, wl.H, wl.s, -1, 2)
    cache.v_codes[:, :, :wl.s] = vc.reshape(nseq, wl.H, wl.s, -1)
    cache.v_meta[:, :, :wl.s] = vm.reshape(nseq, wl.H, wl.s, -1, 2)
    qkv = synth.normal_f16((nseq, 3 * h1), 1.0, g).numpy()
    xh = synth.normal_f16((nseq, h1), 1.0, g).numpy()
    e_tok = synth.normal_f16((max(wl.vocab // frac, 1), h1), 0.02, g).numpy()
    ones, zeros = np.ones(h1, np.float16), np.zeros(h1, np.float16)

    t0 = time.perf_counter()
    for x, (codes, meta) in slices:
        oracle.linear_g4(x, codes, meta)
    t1 = time.perf_counter()
    oracle.decode_attn_g4(qkv, cache, wl.s, append=True)
    oracle.layernorm(xh, ones, zeros)
    oracle.layernorm(xh, ones, zeros)
    t2 = time.perf_counter()
    oracle.linear_f16_f32out(oracle.layernorm(xh, ones, zeros), e_tok)
    t3 = time.perf_counter()
    layer = frac * (t1 - t0) + (t2 - t1)
    per_token_step = wl.layers * layer + frac * (t3 - t2)
    return nseq / per_token_step, (t3 - t0), oracle.num_threads()


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

# Why a run with more than one process is refused: the dequant-GEMM kernels
# share activation tiles across a thread-block cluster with multicast bulk
# tensor loads, which are kept to runs that use a single GPU.  Sequences are
# independent, so N GPUs are N separate single-GPU jobs.
MULTI_GPU_REFUSAL = ("one GPU per run: the dequant-GEMM kernels use cluster-multicast "
                     "bulk tensor loads, which stay in single-GPU runs; run N independent "
                     "single-GPU jobs instead")


def footprints(wl, kv="g4"):
    """Bytes of the model's 4-bit weights (codes, half a byte, plus (min,
    scale), 8 bytes per 64 weights) and of its K/V caches (every layer, cap =
    s + n slots; 4-bit rows of d/2 code bytes and d/8 (min, scale) bytes, or
    fp16 rows)."""
    wbytes = wl.layers * (4 * wl.h1 * wl.h1 + 2 * wl.h1 * wl.h2) * 0.625
    per = 2 * wl.d * 2 if kv == "f16" else wl.d * 1.25   # K and V together
    return wbytes, wl.layers * wl.bls * wl.H * wl.cap * per


def workload_config(wl, args, ws, wbytes=None, kvbytes=None):
    """The `config` object of a bench line: the workload and the options, with
    the weight and cache footprints computed from the shapes when not given
    (the oracle's line names the same configuration as the GPU arm's)."""
    D = wl.decode_steps
    if wl.vocab == 0:   # one decoder layer fed synthetic hidden states
        return {"workload": "%s: one decoder layer, h1 %d, %d heads, h2 %d; gbs %d x k %d, "
                            "s %d, %d teacher-forced decode steps; weights and KV 4-bit g64"
                            % (wl.name, wl.h1, wl.H, wl.h2, wl.gbs, wl.k, wl.s, D),
                "decode_launch": "eager" if args.no_graphs else "one CUDA graph per decode step",
                "l2": "inputs smaller than L2 (a latency-bound workload; no flush)"}
    host = args.weights == "host"
    graphs = not args.no_graphs and not host
    fw, fkv = footprints(wl, args.kv)
    wbytes = fw if wbytes is None else wbytes
    kvbytes = fkv if kvbytes is None else kvbytes
    return {"workload": "%s-shaped: %d layers, h1 %d, %d heads, h2 %d, vocab %d; "
                        "gbs %d x k %d = bls %d, s %d, n %d (%d decode steps); "
                        "weights 4-bit g64, KV cache %s, in HBM"
                        % (wl.name, wl.layers, wl.h1, wl.H, wl.h2, wl.vocab, wl.gbs,
                           wl.k, wl.bls, wl.s, wl.n, D,
                           "fp16 (uncompressed)" if args.kv == "f16" else "4-bit g64"),
            "kv_cache": args.kv,
            "decode_attention": ("top-K sparse, %d%% of the rows' V" % args.topk
                                 if 0 < args.topk < 100 else "dense"),
            "order": args.order, "decoding": "greedy (argmax on the device)",
            "decode_launch": "one CUDA graph per decode step" if graphs else "eager",
            "parallelism": "replicas" if ws > 1 else "single",
            "weights": ("4-bit, pinned host memory, streamed one layer ahead over "
                        "NVLink-C2C" if host else "4-bit, resident in HBM"),
            "l2": "inputs larger than L2 (weights %.1f GB, KV %.1f GB)"
                  % (wbytes / 1e9, kvbytes / 1e9)}


def run_fg(args, ws, rank, local):
    if ws > 1:
        # no GPU is touched; rank 0 alone says why
        return ({"metric": METRIC, "unit": UNIT, "n_gpus": ws, "unavailable": MULTI_GPU_REFUSAL}
                if rank == 0 else None)
    from bit_group_quant_gb300 import fg
    from bit_group_quant_gb300.model import random_model

    wl = synth.WORKLOADS[args.workload]
    D = wl.decode_steps
    if wl.vocab == 0:
        return run_layer_workload(args, wl, local)

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        v, secs, cores = oracle_sample(wl, args.cpu_seqs, frac=args.cpu_frac)
        cpu_base = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                    "sample": "one decode token step of %d sequences at context %d: 1/%d row "
                              "slices of the four projections and the LM head (scaled by %d), "
                              "full attention and LayerNorms, one layer scaled to %d "
                              "(%.1f s of CPU work)" % (args.cpu_seqs, wl.s, args.cpu_frac,
                                                        args.cpu_frac, wl.layers, secs)}

    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    init_dist(ws, "nccl")
    stream = torch.cuda.current_stream()

    host = args.weights == "host"
    model = random_model(wl, seed=0, device=dev, host_weights=host, kv=args.kv)
    model.stack.topk_pct = args.topk
    g = synth.generator(1000 + rank, dev)
    prompt = synth.token_ids((wl.bls, wl.s), wl.vocab, g, dev)
    logits_buf = [torch.empty((wl.bls, wl.vocab), dtype=torch.float32, device=dev)
                  for _ in range(2)]
    toks = torch.empty((wl.n, wl.bls), dtype=torch.int32, device=dev)   # generated, time-major

    graphs = []

    def step(evs=None, prompt_ids=prompt, eager=False):
        # greedy generation of n tokens per prompt: token 1 from the prefill,
        # token t+1 from decode step t fed token t; all on the device.  The
        # decode steps replay their CUDA graphs unless eager (the traced pass
        # times every launch from the host).
        if evs:
            evs[0].record(stream)
        lg = model.prefill(prompt_ids, args.order, logits=logits_buf[0])
        fg.fg_argmax(lg, out=toks[0])
        if evs:
            evs[1].record(stream)
        if graphs and not eager:
            for gph in graphs:
                gph.replay()
        else:
            for t in range(1, D + 1):
                lg = model.decode_step(toks[t - 1], t, wl.s, args.order, logits=logits_buf[t % 2])
                fg.fg_argmax(lg, out=toks[t])
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
    fg.fg_check()
    if not args.no_graphs and not host:
        graphs.extend(model.capture_decode_steps(toks, wl.s, logits_buf, args.order))
        step()
        fg.fg_check()

    # ---------------- timed region (device-resident inputs).  K steps timed
    # with one event pair per phase give the throughput; K more steps with an
    # event pair around every launch of the traced kernel classes give the
    # per-kernel durations behind the roofline (those events add a little
    # device time, so they stay out of the throughput steps).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    barrier()
    fg.fg_trace_begin(fg.FG_TRACE_GEMM_PREFILL | fg.FG_TRACE_GEMM_DECODE |
                      fg.FG_TRACE_ATTN_DECODE | fg.FG_TRACE_ATTN_PREFILL)
    for k in range(args.steps):
        step(eager=True)
    torch.cuda.synchronize()
    trace = fg.fg_trace_end()
    barrier()
    clk = clocks.stop()
    fg.fg_check()
    t_pre = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    value, t_dec_max = aggregate(wl.bls * D * args.steps, t_dec, dev)
    gen_value, t_all_max = aggregate(wl.bls * wl.n * args.steps, t_pre + t_dec, dev)

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_prompt = prompt.cpu().pin_memory()
        h_toks = torch.empty((wl.n, wl.bls), dtype=torch.int32).pin_memory()
        d_prompt = torch.empty_like(prompt)
        e2e_dec = e2e_all = 0.0
        barrier()
        torch.cuda.synchronize()
        for k in range(args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            ev[0].record(stream)
            d_prompt.copy_(h_prompt, non_blocking=True)
            ev[1].record(stream)
            step(ev[2:], prompt_ids=d_prompt)
            h_toks.copy_(toks, non_blocking=True)
            end = torch.cuda.Event(enable_timing=True)
            end.record(stream)
            torch.cuda.synchronize()
            # the decode phase plus the step's host copies (prompt ids in,
            # generated tokens out)
            e2e_dec += (ev[0].elapsed_time(ev[1]) + ev[3].elapsed_time(end)) / 1e3
            e2e_all += ev[0].elapsed_time(end) / 1e3
        e2e_value, _ = aggregate(wl.bls * D * args.steps, e2e_dec, dev)
        e2e_gen, _ = aggregate(wl.bls * wl.n * args.steps, e2e_all, dev)
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": int(h_prompt.numel() * 4),
               "d2h_bytes_per_step": int(h_toks.numel() * 4),
               "generation_tokens_per_s": e2e_gen,
               "note": "decode phase plus the step's host copies: the H2D copy of the prompt "
                       "ids from pinned memory and the D2H copy of the n generated tokens of "
                       "every sequence into pinned memory; generation_tokens_per_s times the "
                       "whole step, prefill included"}
        fg.fg_check()

    stream_info = None
    if host:
        # beta: one layer's weight copies alone (the copy stream idle otherwise)
        torch.cuda.synchronize()
        st = model.stack
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record(st.copy_stream)
        for r in range(reps):
            st.next = None
            st._fetch(r % len(st.layers), r % 2)
        b.record(st.copy_stream)
        torch.cuda.synchronize()
        st.next = None
        beta = st.bytes_per_layer * reps / (a.elapsed_time(b) / 1e3)
        W = st.bytes_per_layer * len(st.layers)
        t_step = t_dec / max(args.steps, 1) / D
        stream_info = {
            "bytes_per_layer": st.bytes_per_layer, "model_bytes": W,
            "h2d_gbs": beta / 1e9,
            "bound_ms_per_decode_step": W / beta * 1e3,
            "measured_ms_per_decode_step": t_step * 1e3,
            "note": "weights fetched once per token step for the whole block: per sequence at "
                    "least W/(B beta); the decode step is bound by W/beta when that exceeds "
                    "the resident step's compute"}

    if rank != 0:
        return None

    peaks, peak_kind = load_peaks()
    wbytes = (model.stack.bytes_per_layer * len(model.stack.layers) if host
              else sum(L.nbytes_q4 for L in model.stack.layers))
    gp = trace["gemm_prefill"]
    gd = trace["gemm_decode"]
    ad = trace["attn_decode"]
    ap = trace["attn_prefill"]
    tflops = lambda c: c["flops"] / (c["ms"] / 1e3) / 1e12 if c["ms"] > 0 else None
    gbs = lambda c: c["bytes"] / (c["ms"] / 1e3) / 1e9 if c["ms"] > 0 else None
    # The dominant kernel of the step is the prefill dequant-GEMM (tensor-bound);
    # it runs inside a seconds-long step, so the sustained cuBLAS figure is the peak.
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    achieved = tflops(gp)
    launches = sum(c["launches"] for c in trace.values())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_all_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic",
        "config": workload_config(wl, args, ws, wbytes,
                                  sum(c.nbytes for c in model.stack.caches)),
        "generation_tokens_per_s": gen_value,
        "gemm_tflops": {"prefill": tflops(gp), "decode": tflops(gd)},
        "attn_gbs": {("decode_f16" if args.kv == "f16" else "decode_4bit"): gbs(ad)},
        "phase_ms_per_step": {"prefill": t_pre / args.steps * 1e3,
                              "decode": t_dec / args.steps * 1e3},
        "kernel_ms_per_step": {k: c["ms"] / args.steps for k, c in trace.items()},
        "roofline": {"kernel": "prefill projections: dequant_g4_kernel (weights to fp16, once per "
                               "launch) + gemm_pf_kernel (CTA-pair tcgen05 GEMM); time of both",
                     "bound": "tensor",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak if achieved else None,
                     "peak_source": "%s bf16_tflops_sustained (fp16 dense rate = bf16)" % peak_kind,
                     "traffic": committed_traffic("gemm_pf.cu", wl.name),
                     "launches": gp["launches"],
                     "avg_launch_ms": gp["ms"] / max(gp["launches"], 1)},
        "decode_roofline": {
            "gemm": {"bound": "tensor", "achieved": tflops(gd), "unit": "TFLOP/s",
                     "peak": peak,
                     "frac": tflops(gd) / peak if tflops(gd) else None},
            "attn": {"bound": "hbm", "achieved": gbs(ad), "unit": "GB/s",
                     "peak": peaks["hbm_gbs"],
                     "frac": gbs(ad) / peaks["hbm_gbs"] if gbs(ad) else None}},
        "prefill_attn_tflops": tflops(ap),
        "cpu_baseline": cpu_base,
        "weight_stream": stream_info,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    return line


# --------------------------------------------------------------------------
# kernel micro-benchmarks: one kernel on one shape (ncu captures), and the
# OPT-175B single-layer sweep
# --------------------------------------------------------------------------

def _time_launches(fn, iters, stream):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters / 1e3


def gemm_case(M, N, K, iters, dev, seed=0, residual=False):
    """One dequant-GEMM launch shape with a bias (and, as the decoder's out
    and fc2 projections have, a residual); returns (seconds, TFLOP/s, GB/s)."""
    from bit_group_quant_gb300 import fg
    g = synth.generator(seed, dev)
    q = fg.fg_quantize_g4(synth.normal_f16((N, K), 0.02, g, dev))
    x = synth.normal_f16((M, K), 1.0, g, dev)
    b = synth.normal_f16((N,), 0.1, g, dev)
    r = synth.normal_f16((M, N), 1.0, g, dev) if residual else None
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    ws_n = fg.fg_dequant_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    fn = lambda: fg.fg_dequant_gemm_g4(x, q, bias=b, residual=r, Y=y, workspace=ws)
    sec = _time_launches(fn, iters, torch.cuda.current_stream())
    fg.fg_check()
    flops = 2.0 * M * N * K
    bytes_ = 0.625 * N * K + 2.0 * M * K + 2.0 * M * N * (2.0 if residual else 1.0)
    return sec, flops / sec / 1e12, bytes_ / sec / 1e9


def attn_case(B, H, d, L, iters, dev, seed=0, topk=0, kv="g4"):
    """One decode-attention launch over a full 4-bit cache of L rows
    (fused append at slot L-1); returns (seconds, GB/s).  topk 1..99: the
    top-K sparse attention keeping that percent of the rows' V (its bytes:
    every K row, the kept V rows).  kv "f16": the uncompressed cache."""
    from bit_group_quant_gb300 import fg
    g = synth.generator(seed, dev)
    if kv == "f16":
        c16 = fg.KV16.empty(B, H, d, L, dev, zero=False)
        c16.k.copy_(synth.normal_f16((B, H, L, d), 1.0, g, dev))
        c16.v.copy_(synth.normal_f16((B, H, L, d), 1.0, g, dev))
        qkv = synth.normal_f16((B, 3 * H * d), 1.0, g, dev)
        out = torch.empty((B, H * d), dtype=torch.float16, device=dev)
        sec = _time_launches(lambda: fg.fg_decode_attn_f16(qkv, c16, L - 1, out=out), iters,
                             torch.cuda.current_stream())
        fg.fg_check()
        return sec, B * H * (2.0 * L * d * 2 + 2 * d * 2 + 8.0 * d) / sec / 1e9
    cache = fg.KV4.empty(B, H, d, L, dev, zero=False)
    rows = synth.normal_f16((B * H * L, d), 1.0, g, dev)
    kq = fg.fg_quantize_g4(rows)
    cache.k_codes.copy_(kq.codes.view_as(cache.k_codes))
    cache.k_meta.copy_(kq.meta.view_as(cache.k_meta))
    vq = fg.fg_quantize_g4(synth.normal_f16((B * H * L, d), 1.0, g, dev))
    cache.v_codes.copy_(vq.codes.view_as(cache.v_codes))
    cache.v_meta.copy_(vq.meta.view_as(cache.v_meta))
    del rows, kq, vq
    qkv = synth.normal_f16((B, 3 * H * d), 1.0, g, dev)
    out = torch.empty((B, H * d), dtype=torch.float16, device=dev)
    if 0 < topk < 100:
        ws = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(B, H, L - 1), dtype=torch.uint8,
                         device=dev)
        fn = lambda: fg.fg_decode_attn_topk_g4(qkv, cache, L - 1, topk, fuse_append=True, out=out,
                                               workspace=ws)
        nv = fg.fg_topk_count(L, topk)
    else:
        fn = lambda: fg.fg_decode_attn_g4(qkv, cache, L - 1, fuse_append=True, out=out)
        nv = L
    sec = _time_launches(fn, iters, torch.cuda.current_stream())
    fg.fg_check()
    row = d / 2 + (d / 64) * 8
    bytes_ = B * H * ((L + nv) * row + 2 * row + 8.0 * d)
    return sec, bytes_ / sec / 1e9


def quant_case(iters, dev, seed=0):
    """The group-wise 4-bit quantiser at HBM rate: (1) fg_quantize_g4 on one
    OPT-30B fc1 matrix (28672 x 7168 fp16 -> codes + (min, scale)); (2) the
    prefill's K/V store (the same quantiser on every prompt row's k and v,
    into the cache) for 16 sequences of 512 tokens, 56 heads of 128, timed
    by its trace class inside fg_prefill_attn.  Algorithmic bytes: 2 read +
    0.625 written per element."""
    from bit_group_quant_gb300 import fg
    g = synth.generator(seed, dev)
    N, K = 28672, 7168
    x = synth.normal_f16((N, K), 0.02, g, dev)
    q = fg.Q4.empty(N, K, dev)
    sec = _time_launches(lambda: fg.fg_quantize_g4(x, out=q), iters, torch.cuda.current_stream())
    fg.fg_check()
    wq = {"elements": N * K, "ms": sec * 1e3, "gbs": 2.625 * N * K / sec / 1e9}
    del x, q
    B, S, H, d = 16, 512, 56, 128
    qkv = synth.normal_f16((B * S, 3 * H * d), 1.0, g, dev)
    cache = fg.KV4.empty(B, H, d, S, dev)
    out = torch.empty((B * S, H * d), dtype=torch.float16, device=dev)
    for _ in range(3):
        fg.fg_prefill_attn(qkv, B, S, H, d, cache=cache, out=out)
    torch.cuda.synchronize()
    fg.fg_trace_begin(fg.FG_TRACE_OTHER)
    for _ in range(iters):
        fg.fg_prefill_attn(qkv, B, S, H, d, cache=cache, out=out)
    torch.cuda.synchronize()
    tr = fg.fg_trace_end()["other"]
    fg.fg_check()
    n = 2 * B * S * H * d
    kv = {"elements": n, "ms": tr["ms"] / max(tr["launches"], 1),
          "gbs": 2.625 * n / (tr["ms"] / max(tr["launches"], 1) / 1e3) / 1e9}
    return wq, kv


def prefill_case(B, s, H, d, iters, dev, seed=0):
    """One causal prefill-attention launch over fp16 Q/K/V of B sequences of s
    tokens; returns (seconds, causal TFLOP/s)."""
    from bit_group_quant_gb300 import fg
    g = synth.generator(seed, dev)
    qkv = synth.normal_f16((B * s, 3 * H * d), 1.0, g, dev)
    out = torch.empty((B * s, H * d), dtype=torch.float16, device=dev)
    fn = lambda: fg.fg_prefill_attn(qkv, B, s, H, d, out=out)
    sec = _time_launches(fn, iters, torch.cuda.current_stream())
    fg.fg_check()
    flops = 4.0 * B * H * (s * (s + 1) / 2.0) * d
    return sec, flops / sec / 1e12


def decode_case(args, dev):
    """Decode steps only (greedy, block order) of the workload's model at
    bls = gbs * k, weights resident in HBM or streamed from pinned host
    memory: decode tokens/s.  The prompt's cache rows are left as allocated
    (zeros): a decode step's work does not depend on the cache contents."""
    import dataclasses
    from bit_group_quant_gb300 import fg
    from bit_group_quant_gb300.model import random_model
    wl = synth.WORKLOADS[args.workload]
    if args.gbs:
        wl = dataclasses.replace(wl, gbs=args.gbs, k=args.k or 1)
    host = args.weights == "host"
    model = random_model(wl, seed=0, device=dev, host_weights=host, kv=args.kv)
    model.stack.topk_pct = args.topk
    D = wl.decode_steps
    toks = torch.zeros((wl.n, wl.bls), dtype=torch.int32, device=dev)
    lg = [torch.empty((wl.bls, wl.vocab), dtype=torch.float32, device=dev) for _ in range(2)]
    def steps(n):
        for t in range(1, n + 1):
            l = model.decode_step(toks[t - 1], t, wl.s, "block", logits=lg[t % 2])
            fg.fg_argmax(l, out=toks[t])
    steps(3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    h0 = time.perf_counter()
    steps(D)
    h1 = time.perf_counter()
    b.record()
    torch.cuda.synchronize()
    fg.fg_check()
    sec = a.elapsed_time(b) / 1e3
    return {"micro": "decode", "weights": args.weights, "kv": args.kv, "s": wl.s,
            "topk_pct": args.topk,
            "bls": wl.bls, "gbs": wl.gbs, "k": wl.k,
            "decode_steps": D, "ms_per_decode_step": sec / D * 1e3,
            "host_enqueue_ms_per_decode_step": (h1 - h0) / D * 1e3,
            "decode_tokens_per_s": wl.bls * D / sec}


def run_micro(args):
    torch.cuda.set_device(0)
    dev = "cuda:0"
    peaks, kind = load_peaks()
    if args.micro == "decode":
        return decode_case(args, dev)
    if args.micro == "gemm":
        sec, tf, gb = gemm_case(args.M, args.N, args.K, args.iters, dev, residual=args.residual)
        return {"micro": "dequant_gemm", "M": args.M, "N": args.N, "K": args.K,
                "residual": args.residual,
                "ms": sec * 1e3, "tflops": tf, "gbs": gb,
                "frac_tensor": tf / peaks["bf16_tflops"], "peak_source": kind + " bf16_tflops"}
    if args.micro == "prefill":
        sec, tf = prefill_case(args.B, args.L, args.H, args.d, args.iters, dev)
        return {"micro": "prefill_attn", "B": args.B, "s": args.L, "H": args.H, "d": args.d,
                "ms": sec * 1e3, "tflops_causal": tf, "frac_tensor": tf / peaks["bf16_tflops"],
                "peak_source": kind + " bf16_tflops"}
    if args.micro == "quant":
        wq, kv = quant_case(args.iters, dev)
        return {"micro": "quantize_g4", "weights_28672x7168": wq, "kv_store_B16_s512_H56_d128": kv,
                "peak_hbm_gbs": peaks["hbm_gbs"], "frac_hbm": {"weights": wq["gbs"] / peaks["hbm_gbs"],
                                                               "kv_store": kv["gbs"] / peaks["hbm_gbs"]},
                "peak_source": kind + " hbm_gbs"}
    if args.micro == "attn":
        sec, gb = attn_case(args.B, args.H, args.d, args.L, args.iters, dev, topk=args.topk,
                            kv=args.kv)
        res = {"micro": ("decode_attn_f16" if args.kv == "f16" else
                         "decode_attn_topk_g4" if 0 < args.topk < 100 else "decode_attn_g4"),
               "B": args.B, "H": args.H, "d": args.d, "L": args.L,
               "ms": sec * 1e3, "gbs": gb, "frac_hbm": gb / peaks["hbm_gbs"],
               "peak_source": kind + " hbm_gbs"}
        if 0 < args.topk < 100:
            dsec, _ = attn_case(args.B, args.H, args.d, args.L, args.iters, dev)
            res.update({"keep_pct": args.topk, "dense_ms": dsec * 1e3, "speedup": dsec / sec})
        return res
    # OPT-175B single-layer sweep: dequant-GEMM at bls in {32,144,256,512} for
    # the four projection shapes, decode attention at bls 144 for three contexts
    h1, H, h2 = synth.OPT175B_H1, synth.OPT175B_H, synth.OPT175B_H2
    shapes = {"qkv": (3 * h1, h1), "out": (h1, h1), "fc1": (h2, h1), "fc2": (h1, h2)}
    gemm = {}
    for bls in synth.SWEEP_GEMM_BLS:
        tot_f = tot_s = tot_b = 0.0
        per = {}
        for name, (N, K) in shapes.items():
            sec, tf, gb = gemm_case(bls, N, K, args.iters, dev)
            per[name] = {"ms": sec * 1e3, "tflops": tf, "gbs": gb}
            tot_f += 2.0 * bls * N * K
            tot_b += 0.625 * N * K + 2.0 * bls * (K + N)
            tot_s += sec
        tf = tot_f / tot_s / 1e12
        gb = tot_b / tot_s / 1e9
        bound = "hbm" if bls < 144 else "tensor"
        frac = gb / peaks["hbm_gbs"] if bound == "hbm" else tf / peaks["bf16_tflops"]
        gemm[str(bls)] = {"layer_ms": tot_s * 1e3, "tflops": tf, "gbs": gb, "bound": bound,
                          "frac": frac, "per_projection": per}
    attn = {}
    for L in synth.SWEEP_ATTN_CTX:
        sec, gb = attn_case(synth.SWEEP_ATTN_BLS, H, h1 // H, L, args.iters, dev)
        attn[str(L)] = {"ms": sec * 1e3, "gbs": gb, "frac_hbm": gb / peaks["hbm_gbs"]}
    return {"sweep": "opt-175b layer: h1 12288, 96 heads of 128, h2 49152",
            "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops")}, "peak_source": kind,
            "dequant_gemm": gemm, "decode_attn_bls144": attn}


def run_layer_workload(args, wl, local):
    """The single-decoder-layer workload (no embedding, no LM head): a block
    of bls sequences fed N(0, 1) hidden states, prefill of s prompt tokens,
    then decode_steps teacher-forced decode steps, each fed a new hidden
    state per sequence.  value = bls * decode_steps / decode time."""
    import oracle
    from bit_group_quant_gb300 import fg
    from bit_group_quant_gb300.model import LayerStack, quantize_layer
    from oracle.model import DECODE, PREFILL, layer_step
    from oracle.model import quantize_layer as oracle_layer

    D = wl.decode_steps
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    stream = torch.cuda.current_stream()
    gw = synth.generator(0, dev)
    w = synth.layer_weights(wl.h1, wl.h2, gw, dev)
    stack = LayerStack([quantize_layer(w, wl.h1, wl.H, wl.h2)], wl.gbs, wl.k, wl.s + D, dev)
    g = synth.generator(1000, dev)
    x_pre = synth.normal_f16((wl.bls * wl.s, wl.h1), 1.0, g, dev)
    x_dec = synth.normal_f16((D, wl.bls, wl.h1), 1.0, g, dev)
    y_pre = torch.empty_like(x_pre)
    y_dec = torch.empty_like(x_dec)
    order = fg.FG_ORDER_BLOCK

    graphs = []

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        stack.run(x_pre, fg.FG_PHASE_PREFILL, wl.s, 0, order, out=y_pre)
        if evs:
            evs[1].record(stream)
        if graphs:
            for gph in graphs:
                gph.replay()
        else:
            for t in range(1, D + 1):
                stack.run(x_dec[t - 1], fg.FG_PHASE_DECODE, 1, wl.s + t - 1, order, out=y_dec[t - 1])
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
    fg.fg_check()
    launches_eager = 0
    fg.fg_trace_begin(0)
    step()
    torch.cuda.synchronize()
    launches_eager = sum(c["launches"] for c in fg.fg_trace_end().values())
    if not args.no_graphs:
        # one CUDA graph per decode step (its slot is a launch argument)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        for t in range(1, D + 1):
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=side):
                stack.run(x_dec[t - 1], fg.FG_PHASE_DECODE, 1, wl.s + t - 1, order, out=y_dec[t - 1],
                          stream=side)
            graphs.append(gph)
        stream.wait_stream(side)
        step()
        fg.fg_check()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    clocks.start()
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    clk = clocks.stop()
    fg.fg_check()
    t_pre = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    value = wl.bls * D * args.steps / t_dec
    # end to end: hidden states in from pinned host memory, the last decode
    # step's output back, every step
    e2e = None
    if not args.no_e2e:
        h_pre = x_pre.cpu().pin_memory()
        h_dec = x_dec.cpu().pin_memory()
        h_out = torch.empty_like(y_dec[-1], device="cpu").pin_memory()
        tot_dec = 0.0
        for k in range(args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            ev[0].record(stream)
            x_pre.copy_(h_pre, non_blocking=True)
            x_dec.copy_(h_dec, non_blocking=True)
            ev[1].record(stream)
            step(ev[2:5])
            h_out.copy_(y_dec[-1], non_blocking=True)
            ev[5].record(stream)
            torch.cuda.synchronize()
            # the copies in (prompt and decode inputs), the decode phase, the copy out
            tot_dec += (ev[0].elapsed_time(ev[1]) + ev[3].elapsed_time(ev[5])) / 1e3
        e2e = {"value": wl.bls * D * args.steps / tot_dec, "unit": UNIT,
               "h2d_bytes_per_step": int(h_pre.numel() * 2 + h_dec.numel() * 2),
               "d2h_bytes_per_step": int(h_out.numel() * 2),
               "note": "decode phase plus the read-back of the last decode step's hidden states; "
                       "the hidden-state inputs are copied in from pinned memory every step"}
    cpu_base = None
    if not args.no_cpu_baseline:
        # the oracle on the whole workload (it is small): prefill + D decode steps
        ol = oracle_layer({n: t.cpu().numpy() for n, t in w.items()}, wl.h1, wl.H, wl.h2)
        cache = oracle.KVCache(wl.bls, wl.H, wl.d, wl.s + D)
        xp, xd = x_pre.cpu().numpy(), x_dec.cpu().numpy()
        t0 = time.perf_counter()
        layer_step(ol, xp, cache, PREFILL, wl.bls, wl.s)
        t1 = time.perf_counter()
        for t in range(1, D + 1):
            layer_step(ol, xd[t - 1], cache, DECODE, wl.bls, 1, pos=wl.s + t - 1)
        t2 = time.perf_counter()
        cpu_base = {"value": wl.bls * D / (t2 - t1), "unit": UNIT, "cores": oracle.num_threads(),
                    "kind": "oracle",
                    "sample": "the whole workload (prefill %.2f s, %d decode steps %.2f s)"
                              % (t1 - t0, D, t2 - t1)}
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": (t_pre + t_dec) / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
            "data": "synthetic",
            "config": workload_config(wl, args, 1),
            "phase_ms_per_step": {"prefill": t_pre / args.steps * 1e3,
                                  "decode": t_dec / args.steps * 1e3},
            "gpu_launches": int(launches_eager) * args.steps,
            "cpu_baseline": cpu_base, "e2e": e2e, "clocks": clk}


def run_reference(args, ws, rank):
    """The oracle timed on this host's cores: each step is a bounded sample."""
    if rank != 0:
        return None
    wl = synth.WORKLOADS[args.workload]
    for _ in range(args.warmup):
        oracle_sample(wl, args.ref_seqs, seed=1, frac=args.ref_frac)
    vals, secs = [], 0.0
    cores = 1
    for k in range(args.steps):
        v, s, cores = oracle_sample(wl, args.ref_seqs, seed=2 + k, frac=args.ref_frac)
        vals.append(v)
        secs += s
    value = len(vals) / sum(1.0 / v for v in vals)
    sample = ("per step: one decode token step of %d sequences at context %d: 1/%d row slices "
              "of the four projections and the LM head (scaled by %d), full attention and "
              "LayerNorms, one layer scaled to %d layers (%.1f s of CPU work per step)"
              % (args.ref_seqs, wl.s, args.ref_frac, args.ref_frac, wl.layers,
                 secs / max(args.steps, 1)))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(wl, args, ws),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fg", choices=["fg", "reference"])
    ap.add_argument("--workload", default="opt-30b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--order", default="block", choices=["block", "zigzag"])
    ap.add_argument("--weights", default="hbm", choices=["hbm", "host"],
                    help="host: 4-bit weights in pinned host memory, streamed one layer ahead")
    ap.add_argument("--cpu-seqs", type=int, default=24)
    ap.add_argument("--ref-seqs", type=int, default=2)
    ap.add_argument("--cpu-frac", type=int, default=1)
    ap.add_argument("--ref-frac", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch the decode steps eagerly instead of replaying CUDA graphs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gbs", type=int, default=0, help="--micro decode: override gbs")
    ap.add_argument("--k", type=int, default=0, help="--micro decode: override k")
    ap.add_argument("--kv", choices=["g4", "f16"], default="g4",
                    help="KV cache: 4-bit g64 (the method) or fp16 (the uncompressed A/B)")
    ap.add_argument("--topk", type=int, default=0,
                    help="top-K sparse decode attention keeping this percent of the rows "
                         "(0: dense); the step, --micro attn and --micro decode")
    ap.add_argument("--micro", choices=["gemm", "attn", "prefill", "sweep175b", "decode", "quant"],
                    default=None,
                    help="time one kernel shape (or the OPT-175B layer sweep) instead")
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--residual", action="store_true",
                    help="--micro gemm: add a residual operand (the out and fc2 projections)")
    ap.add_argument("--N", type=int, default=28672)
    ap.add_argument("--K", type=int, default=7168)
    ap.add_argument("--B", type=int, default=144)
    ap.add_argument("--H", type=int, default=56)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--L", type=int, default=513)
    ap.add_argument("--iters", type=int, default=10)
    args = ap.parse_args(argv)
    ws, rank, local = dist_env()
    if ws > 1 and args.impl != "reference":
        line = run_fg(args, ws, rank, local)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.micro:
        print(json.dumps(run_micro(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_fg(args, ws, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
