"""Seeded synthetic inputs and workload shapes.

This module is shared by the CUDA path's driver, the tests and the oracle
harness.  It holds no arithmetic of the method (no quantisation, no layer
math): only random tensors drawn with torch generators and the shape tables
of the workloads.  Recipe: seed 0; weights fp16 ~ N(0, 0.02); biases 0;
LayerNorm gamma 1, beta 0; hidden-state inputs fp16 ~ N(0, 1); token ids
uniform over [0, vocab); KV-sweep rows fp16 ~ N(0, 1).  The pages benchmark
with dummy weights, so random weights of the right shapes are the workload.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    h1: int
    H: int
    h2: int
    vocab: int        # 0: single decoder layer fed with hidden states
    gbs: int
    k: int
    s: int
    n: int            # generated tokens per sequence
    decode_steps: int

    @property
    def d(self):
        return self.h1 // self.H

    @property
    def bls(self):
        return self.gbs * self.k

    @property
    def cap(self):
        return self.s + self.n


# One OPT-125M-shaped decoder layer, fed N(0,1) hidden states; 8 teacher-forced
# decode steps after a 32-token prompt.
OPT125M_LAYER = Workload("opt125m-layer", 1, 768, 12, 3072, 0, 4, 1, 32, 8, 8)
# Full models: the prefill yields the first token, so n = 32 tokens take 31
# decode steps.
OPT1_3B = Workload("opt-1.3b", 24, 2048, 32, 8192, 50272, 16, 1, 512, 32, 31)
OPT6_7B = Workload("opt-6.7b", 32, 4096, 32, 16384, 50272, 32, 8, 512, 32, 31)
OPT30B = Workload("opt-30b", 48, 7168, 56, 28672, 50272, 48, 3, 512, 32, 31)
# The same model on the pages' longer synthetic input (prompts padded to 1024).
OPT30B_S1024 = Workload("opt-30b-s1024", 48, 7168, 56, 28672, 50272, 48, 3, 1024, 32, 31)
# OPT-175B single-layer kernel sweep shapes.
OPT175B_H1, OPT175B_H, OPT175B_H2 = 12288, 96, 49152
SWEEP_GEMM_BLS = (32, 144, 256, 512)
SWEEP_ATTN_BLS = 144
SWEEP_ATTN_CTX = (512, 1024, 2048)

WORKLOADS = {w.name: w for w in (OPT125M_LAYER, OPT1_3B, OPT6_7B, OPT30B, OPT30B_S1024)}


def generator(seed: int = 0, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_f16(shape, std: float, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """fp16 tensor drawn from N(0, std^2) (drawn in fp32, rounded once)."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t.to(torch.float16)


def token_ids(shape, vocab: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randint(0, vocab, shape, generator=gen, device=device,
                         dtype=torch.int64).to(torch.int32)


def layer_weights(h1: int, h2: int, gen: torch.Generator, device="cpu",
                  std: float = 0.02) -> dict:
    """fp16 weights of one OPT decoder layer in torch Linear layout [out][in];
    fused QKV = rows q | k | v.  Biases 0, LayerNorm gamma 1 and beta 0."""
    z = lambda n: torch.zeros(n, dtype=torch.float16, device=device)
    o = lambda n: torch.ones(n, dtype=torch.float16, device=device)
    return {
        "w_qkv": normal_f16((3 * h1, h1), std, gen, device),
        "w_out": normal_f16((h1, h1), std, gen, device),
        "w_fc1": normal_f16((h2, h1), std, gen, device),
        "w_fc2": normal_f16((h1, h2), std, gen, device),
        "b_qkv": z(3 * h1), "b_out": z(h1), "b_fc1": z(h2), "b_fc2": z(h1),
        "ln1_g": o(h1), "ln1_b": z(h1), "ln2_g": o(h1), "ln2_b": z(h1),
    }


def random_affine_params(h1: int, h2: int, gen: torch.Generator, device="cpu") -> dict:
    """Non-trivial biases and LayerNorm affine parameters (for tests that must
    exercise every epilogue term; the benchmark workload keeps 0 / 1 / 0)."""
    return {
        "b_qkv": normal_f16((3 * h1,), 0.1, gen, device),
        "b_out": normal_f16((h1,), 0.1, gen, device),
        "b_fc1": normal_f16((h2,), 0.1, gen, device),
        "b_fc2": normal_f16((h1,), 0.1, gen, device),
        "ln1_g": (1.0 + normal_f16((h1,), 0.1, gen, device).float()).half(),
        "ln1_b": normal_f16((h1,), 0.1, gen, device),
        "ln2_g": (1.0 + normal_f16((h1,), 0.1, gen, device).float()).half(),
        "ln2_b": normal_f16((h1,), 0.1, gen, device),
    }


def embeddings(vocab: int, positions: int, h1: int, gen: torch.Generator,
               device="cpu", std: float = 0.02):
    return (normal_f16((vocab, h1), std, gen, device),
            normal_f16((positions, h1), std, gen, device))


def pad_counts(n: int, s: int, gen: torch.Generator, min_len: int = 1, device="cpu") -> torch.Tensor:
    """Left-padding counts of n prompts padded to the common length s: each
    real length is uniform in [min_len, s] (a mix of short and full prompts),
    pad = s - length.  int32 [n]."""
    lengths = torch.randint(min_len, s + 1, (n,), generator=gen, device=device, dtype=torch.int64)
    return (s - lengths).to(torch.int32)
