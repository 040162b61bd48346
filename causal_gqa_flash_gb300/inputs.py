"""Seeded synthetic inputs for causal grouped-query attention.

This module only draws random numbers; it holds none of the attention
arithmetic, so both the CUDA path and the oracle can be fed from it.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws q, k, v and dO,
in that order, as float32 standard normals; q and k are multiplied by
``qk_std``; every tensor is then rounded to bf16 (round to nearest even).
Layouts are [B, T, H, d] with H = Hq for q/dO and H = Hkv for k/v.

The named workloads are the attention shapes of the PTX trainer ("A
transformer in PTX", §The model: 6 query heads of 64 over 2 kv heads) and
larger causal shapes up to a Llama-8B-style head layout. There is no dataset:
attention inputs are activations, and normal draws stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    qk_std: float = 1.0
    causal: bool = True

    @property
    def seed(self) -> int:
        return 1000 + int(self.name[1:])

    def describe(self) -> str:
        return (f"B={self.B} T={self.T} Hq={self.Hq} Hkv={self.Hkv} d={self.d} "
                f"{'causal' if self.causal else 'full'} q,k~N(0,{self.qk_std**2:g}) v,dO~N(0,1) bf16")


WORKLOADS = {
    "c1": Workload("c1", 1, 128, 6, 2, 64),
    "c2": Workload("c2", 8, 1024, 6, 2, 64),
    "c3": Workload("c3", 4, 4096, 12, 4, 64),
    "c4": Workload("c4", 2, 8192, 32, 8, 128),
    "c5": Workload("c5", 16, 3000, 6, 2, 64, qk_std=2.0),
}


def make_inputs(B: int, T: int, Hq: int, Hkv: int, d: int, seed: int, qk_std: float = 1.0,
                need_grad_out: bool = True):
    """Return bf16 CPU tensors (q, k, v, dO) drawn as described in the module docstring."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, T, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, T, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, T, Hkv, d), generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        q.mul_(qk_std)
        k.mul_(qk_std)
    dout = torch.randn((B, T, Hq, d), generator=g, dtype=torch.float32) if need_grad_out else None
    to_bf16 = lambda x: None if x is None else x.to(torch.bfloat16)
    return to_bf16(q), to_bf16(k), to_bf16(v), to_bf16(dout)


def workload_inputs(w: Workload, need_grad_out: bool = True):
    return make_inputs(w.B, w.T, w.Hq, w.Hkv, w.d, w.seed, w.qk_std, need_grad_out)
