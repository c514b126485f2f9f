"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only names the workloads and
draws their tensors.  Recipe (the same for every workload):

* one ``torch.Generator`` on the target device, seeded with the workload seed;
* draw order Q, K, V, dO, each fp32 N(0, 1) of shape [B, S, heads, D]
  (Q and dO with the query heads, K and V with the key/value heads);
* apply the workload's transform (the GQA workload multiplies K by 2, which
  is exact in bf16);
* cast to the I/O dtype (bf16 casts round to nearest even).

The shapes are those of the DISTFLASHATTN evaluation (Llama-7B attention:
32 heads of dimension 128, sequences of 32K to 512K tokens, a GQA variant);
no dataset or trained weights are involved.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    H_kv: int
    S: int
    D: int
    n_chunks: int
    dtype: torch.dtype
    k_scale: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return self.D ** -0.5

    @property
    def chunk(self) -> int:
        return self.S // self.n_chunks

    def causal_flops(self, fwd: bool = True, bwd: bool = True) -> float:
        """Algorithmic causal FLOPs: pairs = B*H*S(S+1)/2; fwd 4D, bwd 10D per pair."""
        pairs = self.B * self.H * self.S * (self.S + 1) / 2
        return pairs * self.D * ((4 if fwd else 0) + (10 if bwd else 0))


WORKLOADS = {
    w.name: w
    for w in (
        Workload("single_head_s1k_fp32", 1, 1, 1, 1024, 64, 4, torch.float32),
        Workload("llama7b_s32k", 1, 32, 32, 32768, 128, 8, torch.bfloat16),
        Workload("llama7b_gqa8_s64k", 1, 32, 8, 65536, 128, 8, torch.bfloat16, k_scale=2.0),
        Workload("llama7b_s128k", 1, 32, 32, 131072, 128, 16, torch.bfloat16),
        Workload("llama7b_s512k", 1, 32, 32, 524288, 128, 32, torch.bfloat16),
    )
}


def make(B: int, H: int, H_kv: int, S: int, D: int, dtype: torch.dtype, *, seed: int = 0,
         device: str | torch.device = "cpu", k_scale: float = 1.0, S_kv: int | None = None):
    """Draw (q, k, v, dO) following the recipe above."""
    S_kv = S if S_kv is None else S_kv
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn((B, S, H, D), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((B, S_kv, H_kv, D), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((B, S_kv, H_kv, D), generator=g, device=device, dtype=torch.float32)
    do = torch.randn((B, S, H, D), generator=g, device=device, dtype=torch.float32)
    if k_scale != 1.0:
        k.mul_(k_scale)
    return tuple(t.to(dtype) for t in (q, k, v, do))


def make_workload(w: Workload, device="cpu"):
    return make(w.B, w.H, w.H_kv, w.S, w.D, w.dtype, seed=w.seed, device=device, k_scale=w.k_scale)
