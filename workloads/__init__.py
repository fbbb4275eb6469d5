"""Seeded synthetic workloads for Flash-LoRA-Attention.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds shapes and random draws only: none of the method's arithmetic (no
products, no softmax, no LoRA expansion) lives here.

Distributions (LRAgent workloads, shape-only):
  Q, K_base, V_base, X, L ~ N(0, 1)
  A ~ N(0, 1/d_model)         (variance 1/d_model)
  B ~ N(0, 0.02^2)            (std 0.02)

L ~ N(0, 1) is drawn directly for decode workloads: an entry of X.A_i with
X ~ N(0, 1) and A_i ~ N(0, 1/d_model) is a sum of d_model products of
variance 1/d_model, so it has unit variance.  Drawing it avoids generating
a full-context X (10 GB for the ragged serving workload).

Values are drawn in fp32 from a CPU torch.Generator and then rounded to the
storage dtype, so the CPU oracle and the GPU path see bit-identical inputs.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One shape configuration of the decode / prefill / LR-build path."""

    name: str
    n_agents: int          # A
    hq: int                # query heads
    hkv: int               # key/value heads (GQA groups)
    head_dim: int          # d
    d_model: int           # D
    rank: int              # r
    dtype: str             # "f32" or "bf16" storage
    lengths: tuple = ()    # per-request context lengths (decode)
    n0: int = 0            # cached tokens before the prefill chunk
    chunk: int = 0         # new tokens per agent in the prefill chunk
    build_tokens: int = 0  # rows of X for the LR-cache build (0 = none)

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def n_req(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def ragged_lengths(n_req: int = 32, lo: int = 4096, hi: int = 32768, seed: int = 0) -> List[int]:
    """Per-request context lengths, uniform in [lo, hi] (inclusive)."""
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi, size=n_req, endpoint=True)]


# The five shape configurations the path is measured on.
WORKLOADS: Dict[str, Workload] = {
    # 2 agents, 4 q heads = 4 kv heads, d 64, d_model 256, n 256, r 8, fp32.
    "tiny_decode": Workload("tiny_decode", 2, 4, 4, 64, 256, 8, "f32", lengths=(256,),
                            build_tokens=256),
    # Llama-3-8B-shaped layer: 3 agents, 32/8 heads, d 128, d_model 4096, r 16, n 16384.
    "llama8b_decode": Workload("llama8b_decode", 3, 32, 8, 128, 4096, 16, "bf16", lengths=(16384,)),
    # Chunked prefill: 4 agents, 8192 cached + 512 new tokens, causal, r 16; the
    # LR cache of the 512 new tokens is built first (X 512x4096 . A_i 4096x16).
    "llama8b_prefill": Workload("llama8b_prefill", 4, 32, 8, 128, 4096, 16, "bf16",
                                n0=8192, chunk=512, build_tokens=512),
    # Concurrent serving: 32 requests x 4 agents, r 32, ragged lengths in [4096, 32768].
    "llama8b_ragged": Workload("llama8b_ragged", 4, 32, 8, 128, 4096, 32, "bf16",
                               lengths=tuple(ragged_lengths())),
    # Llama-70B-shaped long context: 5 agents, 64/8 heads, d_model 8192, r 64,
    # n 131072, plus the full LR-cache build X (131072x8192) . A_cat (8192x320).
    "llama70b_decode": Workload("llama70b_decode", 5, 64, 8, 128, 8192, 64, "bf16",
                                lengths=(131072,), build_tokens=131072),
}


def _randn(gen: torch.Generator, shape, std: float, dtype, device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) draw from `gen`, rounded to `dtype`, placed on `device`.

    Large tensors are drawn in 64 Mi-element slices so that peak host memory
    stays bounded; the slices consume the generator in order, so the values do
    not depend on where the tensor ends up.
    """
    numel = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(numel, dtype=dtype, device=device)
    step = 1 << 26
    for s in range(0, numel, step):
        e = min(numel, s + step)
        t = torch.randn(e - s, generator=gen, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        out[s:e].copy_(t.to(dtype))
    return out.view(*shape)


def make_decode_inputs(w: Workload, seed: int = 0, device="cpu", shared_L: bool = False,
                       lengths: Optional[List[int]] = None) -> Dict[str, torch.Tensor]:
    """Decode inputs: one query token per agent per request.

    Layouts (row-major):
      Q       [R, A, Hq, d]
      K_base  [N, Hkv, d]      N = sum of lengths (packed by `offsets`)
      V_base  [N, Hkv, d]
      L       [N, A*r]         agent-major column blocks ([N, r] when shared_L)
      B       [A, r, Hkv*d]
      offsets [R+1] int32      prefix sums of the lengths, offsets[0] = 0
    """
    lengths = list(w.lengths if lengths is None else lengths)
    gen = torch.Generator("cpu").manual_seed(seed)
    dt = w.torch_dtype
    A, hq, hkv, d, r = w.n_agents, w.hq, w.hkv, w.head_dim, w.rank
    N = int(sum(lengths))
    R = len(lengths)
    Q = _randn(gen, (R, A, hq, d), 1.0, dt, device)
    K = _randn(gen, (N, hkv, d), 1.0, dt, device)
    V = _randn(gen, (N, hkv, d), 1.0, dt, device)
    L = _randn(gen, (N, r if shared_L else A * r), 1.0, dt, device)
    B = _randn(gen, (A, r, hkv * d), 0.02, dt, device)
    offs = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=device)
    return dict(Q=Q, K_base=K, V_base=V, L=L, B=B, offsets=offs)


def make_prefill_inputs(w: Workload, seed: int = 0, device="cpu", with_X: bool = True
                        ) -> Dict[str, torch.Tensor]:
    """Chunked-prefill inputs (one shared context, one new chunk for every agent).

    Layouts:
      Q       [A, c, Hq, d]     each agent's queries for the c new tokens
      K_base  [n0+c, Hkv, d]    base keys (the chunk's own keys appended)
      V_base  [n0+c, Hkv, d]
      L       [n0+c, A*r]       LR cache; rows [n0, n0+c) are rebuilt from X
      X       [c, D]            hidden states of the chunk
      A_cat   [D, A*r]          [A_1 | ... | A_A]
      B       [A, r, Hkv*d]
    """
    gen = torch.Generator("cpu").manual_seed(seed)
    dt = w.torch_dtype
    A, hq, hkv, d, r, D = w.n_agents, w.hq, w.hkv, w.head_dim, w.rank, w.d_model
    c, n0 = w.chunk, w.n0
    Q = _randn(gen, (A, c, hq, d), 1.0, dt, device)
    K = _randn(gen, (n0 + c, hkv, d), 1.0, dt, device)
    V = _randn(gen, (n0 + c, hkv, d), 1.0, dt, device)
    out = dict(Q=Q, K_base=K, V_base=V)
    if with_X:
        out["X"] = _randn(gen, (c, D), 1.0, dt, device)
        out["A_cat"] = _randn(gen, (D, A * r), D ** -0.5, dt, device)
    out["B"] = _randn(gen, (A, r, hkv * d), 0.02, dt, device)
    out["L"] = _randn(gen, (n0 + c, A * r), 1.0, dt, device)
    return out


def make_build_inputs(n_tokens: int, d_model: int, n_agents: int, rank: int, dtype,
                      seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """LR-cache build inputs: X [n, D] ~ N(0,1), A_cat [D, A*r] ~ N(0, 1/D)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    X = _randn(gen, (n_tokens, d_model), 1.0, dtype, device)
    A_cat = _randn(gen, (d_model, n_agents * rank), d_model ** -0.5, dtype, device)
    return dict(X=X, A_cat=A_cat)


def make_rebase_inputs(n_tokens: int, d_model: int, hkv: int, head_dim: int, n_agents: int, rank: int, dtype,
                       seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """Base-cache rebuild inputs: X [n, D] ~ N(0,1); the pretrained projections
    W_k, W_v [D, Hkv*d] and A_cat [D, A*r] ~ N(0, 1/D) (unit-variance outputs)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    X = _randn(gen, (n_tokens, d_model), 1.0, dtype, device)
    W_k = _randn(gen, (d_model, hkv * head_dim), d_model ** -0.5, dtype, device)
    W_v = _randn(gen, (d_model, hkv * head_dim), d_model ** -0.5, dtype, device)
    A_cat = _randn(gen, (d_model, n_agents * rank), d_model ** -0.5, dtype, device)
    return dict(X=X, W_k=W_k, W_v=W_v, A_cat=A_cat)
