"""Seeded synthetic inputs for per-token adapter routing, shared by the tests and the benchmark.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no routing, no dispatch, no LoRA math), so both the CUDA path and the CPU
oracle may consume what it produces.

Every tensor comes from a torch CPU generator seeded with ``seed`` (default 1234 + the
workload's index below); floating tensors are drawn in fp32 and rounded to bf16 by
round-to-nearest-even where the workload is bf16.  Shapes and distributions follow the
workloads measured in "MoLoRA: Composable Specialization via Per-Token Adapter Routing":

  0 tiny_vocab    N=256, d_in=d_out=512, K=4, r=8, fp32, vocabulary routing.
  1 modality4     N=2048, d_in=d_out=4096, K=4, r=16, bf16 (Table 3's 4-modality kernel
                  benchmark: text / image / audio / video vocabulary ranges).  Tokens come in
                  runs of geometric length (mean 64), one uniformly drawn modality per run;
                  ``dist`` "80-10-5-5" or "95-2-2-1" draws each run's modality with those
                  shares instead (Table 9's group-size distributions); "70-10-10-10" is the
                  text-heavy interleaving of Table 6.
  2 topk_mlp      N=4096, d_in=2048, d_out=6144, K=4, r=16, k=2, bf16, learned router
                  (Figure 2's top-2 weighted sum at a Qwen3-1.7B MLP shape).
  3 decode_sweep  b tokens x K hot-set adapters, d_in=d_out=4096, r=16, bf16, top-1; adapter
                  drawn uniformly or Zipf(s=1.1) (Figures 5 and 9: scalar vs tensor-core).
  4 topk_scaling  N=8192, d_in=d_out=4096, K=8, r=64, k in 1..4, learned router (Table 16).

Common init: x ~ N(0,1); A_a ~ N(0, 1/d_in); B_a ~ N(0, 1/r); y0 ~ N(0,1); scale = 2.0;
router W1 ~ N(0, 1/d_in) [d_in x 64], W2 ~ N(0, 1/64) [64 x K], no biases.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

VOCAB = 32000
ROUTER_HIDDEN = 64
WORKLOADS = ("tiny_vocab", "modality4", "topk_mlp", "decode_sweep", "topk_scaling")


@dataclasses.dataclass
class Workload:
    name: str
    N: int
    d_in: int
    d_out: int
    K: int
    r: int
    k: int
    dtype: torch.dtype
    scale: float
    x: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor
    y0: torch.Tensor
    # vocabulary routing (k == 1): token ids and K+1 range starts
    tok: Optional[torch.Tensor] = None
    starts: Optional[torch.Tensor] = None
    # learned routing: router weights
    W1: Optional[torch.Tensor] = None
    W2: Optional[torch.Tensor] = None
    seed: int = 0

    @property
    def routing(self) -> str:
        return "vocab" if self.tok is not None else "router"

    def describe(self) -> dict:
        return {"workload": self.name, "N": self.N, "d_in": self.d_in, "d_out": self.d_out,
                "K": self.K, "r": self.r, "k": self.k, "dtype": str(self.dtype).replace("torch.", ""),
                "routing": self.routing, "seed": self.seed}


def equal_vocab_starts(K: int, vocab: int = VOCAB) -> torch.Tensor:
    """K equal contiguous vocabulary ranges covering [0, vocab): K+1 strictly increasing starts."""
    return torch.tensor([(a * vocab) // K for a in range(K + 1)], dtype=torch.int32)


def _randn(g, shape, std, dtype):
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * std).to(dtype)


def _adapters(g, K, d_in, d_out, r, dtype):
    A = _randn(g, (K, d_in, r), 1.0 / math.sqrt(d_in), dtype)
    B = _randn(g, (K, r, d_out), 1.0 / math.sqrt(r), dtype)
    return A, B


def _tokens_in_ranges(g, modality: torch.Tensor, starts: torch.Tensor) -> torch.Tensor:
    """A token id drawn uniformly inside the vocabulary range of each position's modality."""
    lo = starts[modality.long()].to(torch.int64)
    hi = starts[modality.long() + 1].to(torch.int64)
    u = torch.rand(modality.numel(), generator=g, dtype=torch.float64)
    return (lo + torch.floor(u * (hi - lo).to(torch.float64)).to(torch.int64)).to(torch.int32)


SHARES = {"80-10-5-5": (0.80, 0.10, 0.05, 0.05), "95-2-2-1": (0.95, 0.02, 0.02, 0.01),
          "70-10-10-10": (0.70, 0.10, 0.10, 0.10)}


def modality_runs(g, N: int, K: int, mean_run: float = 64.0, shares=None) -> torch.Tensor:
    """Per-position modality for N tokens laid out as runs of geometric length (mean
    ``mean_run``, success probability 1/mean_run) with one modality per run, drawn uniformly
    or, when ``shares`` (K probabilities) is given, with those probabilities."""
    p = 1.0 / mean_run
    out = torch.empty(N, dtype=torch.int32)
    pos = 0
    probs = None if shares is None else torch.tensor(shares, dtype=torch.float64)
    while pos < N:
        u = torch.rand(1, generator=g, dtype=torch.float64).item()
        length = 1 + int(math.floor(math.log1p(-u) / math.log1p(-p))) if u > 0 else 1
        if probs is None:
            m = int(torch.randint(0, K, (1,), generator=g).item())
        else:
            m = int(torch.multinomial(probs, 1, generator=g).item())
        out[pos:pos + length] = m
        pos += length
    return out


def zipf_choice(g, n: int, K: int, s: float = 1.1) -> torch.Tensor:
    """n draws from Zipf(s) over ranks 1..K, returned as 0-based indices."""
    p = torch.tensor([1.0 / (i ** s) for i in range(1, K + 1)], dtype=torch.float64)
    return torch.multinomial(p / p.sum(), n, replacement=True, generator=g).to(torch.int32)


def make(name: str, seed: Optional[int] = None, *, N: Optional[int] = None, d_in: Optional[int] = None,
         d_out: Optional[int] = None, K: Optional[int] = None, r: Optional[int] = None,
         k: Optional[int] = None, dist: str = "uniform", dtype: Optional[torch.dtype] = None) -> Workload:
    """Build workload ``name`` (see module docstring); keyword overrides shrink or vary it."""
    idx = WORKLOADS.index(name)
    seed = 1234 + idx if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    scale = 2.0
    if name == "tiny_vocab":
        N, d_in, d_out = N or 256, d_in or 512, d_out or d_in or 512
        K, r, dt = K or 4, r or 8, dtype or torch.float32
        starts = equal_vocab_starts(K)
        tok = torch.randint(0, VOCAB, (N,), generator=g, dtype=torch.int32)
        x = _randn(g, (N, d_in), 1.0, dt)
        A, B = _adapters(g, K, d_in, d_out, r, dt)
        y0 = _randn(g, (N, d_out), 1.0, torch.float32)
        return Workload(name, N, d_in, d_out, K, r, 1, dt, scale, x, A, B, y0, tok=tok, starts=starts, seed=seed)
    if name == "modality4":
        N, d_in = N or 2048, d_in or 4096
        d_out = d_out or d_in
        K, r, dt = K or 4, r or 16, dtype or torch.bfloat16
        starts = equal_vocab_starts(K)
        shares = None
        if dist != "uniform":
            shares = SHARES[dist]
            if len(shares) != K:
                raise ValueError(f"dist {dist} needs K = {len(shares)}")
        tok = _tokens_in_ranges(g, modality_runs(g, N, K, shares=shares), starts)
        x = _randn(g, (N, d_in), 1.0, dt)
        A, B = _adapters(g, K, d_in, d_out, r, dt)
        y0 = _randn(g, (N, d_out), 1.0, torch.float32)
        return Workload(name, N, d_in, d_out, K, r, 1, dt, scale, x, A, B, y0, tok=tok, starts=starts, seed=seed)
    if name == "decode_sweep":
        N, d_in = N or 32, d_in or 4096
        d_out = d_out or d_in
        K, r, dt = K or 4, r or 16, dtype or torch.bfloat16
        starts = equal_vocab_starts(K)
        if dist == "zipf":
            adapter = zipf_choice(g, N, K)
        else:
            adapter = torch.randint(0, K, (N,), generator=g, dtype=torch.int32)
        tok = _tokens_in_ranges(g, adapter, starts)
        x = _randn(g, (N, d_in), 1.0, dt)
        A, B = _adapters(g, K, d_in, d_out, r, dt)
        y0 = _randn(g, (N, d_out), 1.0, torch.float32)
        return Workload(name, N, d_in, d_out, K, r, 1, dt, scale, x, A, B, y0, tok=tok, starts=starts, seed=seed)
    if name in ("topk_mlp", "topk_scaling"):
        if name == "topk_mlp":
            N, d_in, d_out = N or 4096, d_in or 2048, d_out or 6144
            K, r, k = K or 4, r or 16, k or 2
        else:
            N, d_in = N or 8192, d_in or 4096
            d_out = d_out or d_in
            K, r, k = K or 8, r or 64, k or 1
        dt = dtype or torch.bfloat16
        x = _randn(g, (N, d_in), 1.0, dt)
        W1 = _randn(g, (d_in, ROUTER_HIDDEN), 1.0 / math.sqrt(d_in), dt)
        W2 = _randn(g, (ROUTER_HIDDEN, K), 1.0 / math.sqrt(ROUTER_HIDDEN), dt)
        A, B = _adapters(g, K, d_in, d_out, r, dt)
        y0 = _randn(g, (N, d_out), 1.0, torch.float32)
        return Workload(name, N, d_in, d_out, K, r, k, dt, scale, x, A, B, y0, W1=W1, W2=W2, seed=seed)
    raise ValueError(name)
