"""Seeded synthetic inputs and the workload shapes.

This module is the only code that the CUDA path and the CPU oracle share.  It
draws random numbers and names shapes; it holds none of the quantization or
product arithmetic.

Workloads (no trained weights or datasets exist on this machine, so every
tensor is synthetic with the shapes of the model families the pages name):

* ``tiny_int8``  - one 256x256 weight ~ N(0, 0.02^2), x ~ N(0, 1), seed 0 (CPU).
* ``gemma2_9b_int8`` - Gemma-2-9B-shaped decoder linears, 42 layers, INT8
  per tensor (ELG Stream Layer runs Gemma 2 9B).
* ``llama32_3b_int4o`` - Llama-3.2-3B shapes, 28 layers, outlier-aware INT4
  (OTF-LLM validates on Llama-3.2-3B).
* ``llama_7b_int4o`` - 7B Llama-style shapes, 32 layers, batch 1/4/16/64.
* ``llama_70b_int4o`` - 70B shapes, 80 layers (NTransformer runs Llama 3.1 70B).
* ``llama32_3b_head`` - the steps either side of the 3B stack: an INT8
  vocabulary table of 128256 x 3072 (embed_tokens) and the output projection
  (lm_head) of the same shape, tied (the INT8 table itself) or untied
  (outlier-aware INT4); OTF-LLM key innovation 4.

Weights are 0.02 * StudentT(4) in fp16, drawn as z0 / sqrt((z1^2+..+z4^2)/4)
from five standard normals; activations x ~ N(0, 1) fp16; the activation
profile is |N(0, 1)| with a seeded random 1% of channels multiplied by 20.
Head seeds: table = base, untied lm_head = base + 1, its profile base + 2,
hidden states base + 3, token ids base + 4 (uniform over the vocabulary).
Seeds: matrix m of layer l uses base + 16*l + m (m = 0..6 for q,k,v,o,gate,
up,down); the input of group g uses base + 16*l + 8 + g; the profile of
permutation table p uses base + 16*l + 12 + p.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# matrix names in one decoder layer, in seed order
MATS = ("q", "k", "v", "o", "gate", "up", "down")
# launch groups: matrices of one group read the same input vector
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
# permutation tables (input spaces) of one layer, and which groups use each
PERM_TABLES = {"hidden": ("q", "k", "v", "gate", "up"), "attn": ("o",), "mlp": ("down",)}


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str                 # "int8" or "int4o"
    hidden: int
    q_out: int
    kv_out: int
    inter: int
    layers: int
    seed_base: int
    batches: tuple = (1,)
    dist: str = "studentt4"
    extra: dict = field(default_factory=dict)

    def shape(self, m: str) -> tuple[int, int]:
        """(N, K) of matrix m."""
        h, qo, kv, it = self.hidden, self.q_out, self.kv_out, self.inter
        return {"q": (qo, h), "k": (kv, h), "v": (kv, h), "o": (h, qo),
                "gate": (it, h), "up": (it, h), "down": (h, it)}[m]

    def mats(self):
        return MATS


WORKLOADS = {
    "tiny_int8": Workload("tiny_int8", "int8", 256, 256, 256, 256, 1, 0, dist="normal"),
    "gemma2_9b_int8": Workload("gemma2_9b_int8", "int8", 3584, 4096, 2048, 14336, 42, 42),
    "llama32_3b_int4o": Workload("llama32_3b_int4o", "int4o", 3072, 3072, 1024, 8192, 28, 3000),
    "llama_7b_int4o": Workload("llama_7b_int4o", "int4o", 4096, 4096, 4096, 11008, 32, 7000,
                               batches=(1, 4, 16, 64)),
    "llama_70b_int4o": Workload("llama_70b_int4o", "int4o", 8192, 8192, 1024, 28672, 80, 70000),
    # the same decoder shapes in the per-tensor INT8 format
    "llama_7b_int8": Workload("llama_7b_int8", "int8", 4096, 4096, 4096, 11008, 32, 7500),
    "llama_70b_int8": Workload("llama_70b_int8", "int8", 8192, 8192, 1024, 28672, 80, 70500),
}


@dataclass(frozen=True)
class Head:
    """Vocabulary table and output projection of one model family."""
    name: str
    vocab: int
    hidden: int
    seed_base: int


HEADS = {"llama32_3b_head": Head("llama32_3b_head", 128256, 3072, 3900)}


def tokens(B: int, V: int, seed: int, device="cpu") -> torch.Tensor:
    """int32 [B] token ids, uniform over [0, V)."""
    g = _gen(seed, device)
    return torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def matrix_seed(wl: Workload, layer: int, m: str) -> int:
    return wl.seed_base + 16 * layer + MATS.index(m)


def input_seed(wl: Workload, layer: int, g: int) -> int:
    return wl.seed_base + 16 * layer + 8 + g


def profile_seed(wl: Workload, layer: int, table: str) -> int:
    return wl.seed_base + 16 * layer + 12 + list(PERM_TABLES).index(table)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weight(N: int, K: int, seed: int, device="cpu", dist: str = "studentt4") -> torch.Tensor:
    """fp16 [N, K] weight, 0.02 * StudentT(4) (or 0.02 * N(0,1))."""
    g = _gen(seed, device)
    if dist == "normal":
        z = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
        return (0.02 * z).to(torch.float16)
    z = torch.randn((5, N, K), generator=g, device=device, dtype=torch.float32)
    t = z[0] / torch.sqrt((z[1:] * z[1:]).sum(0) / 4.0)
    return (0.02 * t).to(torch.float16)


def activation(B: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp16 [B, K] activations ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((B, K), generator=g, device=device, dtype=torch.float32).to(torch.float16)


def x_profile(K: int, n_boost: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [K] profile |N(0,1)| with n_boost random channels times 20."""
    g = _gen(seed, device)
    p = torch.randn((K,), generator=g, device=device, dtype=torch.float32).abs()
    idx = torch.randperm(K, generator=g, device=device)[:n_boost]
    p[idx] *= 20.0
    return p


def tiny_int8_inputs():
    """The 256x256 INT8 check: W ~ N(0, 0.02^2) then x ~ N(0,1), one CPU
    generator seeded 0, W drawn first."""
    g = _gen(0, "cpu")
    W = (0.02 * torch.randn((256, 256), generator=g)).to(torch.float16)
    x = torch.randn((1, 256), generator=g).to(torch.float16)
    return W, x
