"""Seeded synthetic inputs for MLA tree-verify attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the fp64 oracle and the CUDA path are fed from
here, so the two always see bit-identical inputs.  Everything is drawn on the
CPU with torch's CPU generator, which makes the inputs identical on any host.

Workloads follow the serving regime the pages describe (The Milestone Commit,
"Context": page_size=1 latent cache, long contexts; The Commit That Locked In
6x Decode, "NSPLIT=64 for TP8 Occupancy": 8 heads per rank under TP8; The
Checkpoint Report, "Mistakes and Incorrect Assumptions": draft tokens appended
after the prefix).  The pages name no dataset; these draws stand in for it:

  q, KV rows      ~ N(0, 1) in fp32, rounded to bf16 (round-to-nearest-even)
  slot table      a seeded random subset of the pool (page_size=1 scatter),
                  or contiguous per-request ranges ("defragged" layout)
  draft tree      parent[i] ~ Uniform{-1, 0, ..., i-1}  (-1 = hangs off the
                  prefix), or a chain parent[i] = i - 1
  sm_scale        1 / sqrt(192)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

D_QK = 576
D_V = 512
SM_SCALE = 1.0 / math.sqrt(192.0)
BF16_NAN_BITS = 0x7FC0


@dataclass
class Spec:
    """Shape and layout of one verify step."""
    name: str
    B: int
    H: int
    T: int
    prefix: List[int]
    num_slots: int
    tree: str = "random"          # "random" | "chain"
    layout: str = "scattered"     # "scattered" | "contiguous"
    seed: int = 0
    row_stride: int = D_QK
    canary: bool = False          # unreferenced pool rows become bf16 NaN
    sm_scale: float = SM_SCALE

    def n_keys(self) -> List[int]:
        return [p + self.T for p in self.prefix]

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of one step: every key row read once."""
        return sum(self.n_keys()) * D_QK * 2


@dataclass
class Workload:
    spec: Spec
    q: torch.Tensor             # bf16 [B*T, H, 576]
    kv_pool: torch.Tensor       # bf16 [num_slots, row_stride]
    slot_idx: torch.Tensor      # int32 [sum N_b]
    kv_indptr: torch.Tensor     # int32 [B+1]
    prefix_len: torch.Tensor    # int32 [B]
    parents: torch.Tensor       # int32 [B, T]
    kv_start: Optional[torch.Tensor] = None   # int64 [B] when layout == contiguous
    extra: dict = field(default_factory=dict)


# The five step shapes of the target regime plus the two sweeps.
def spec(name: str, **over) -> Spec:
    base = {
        "tiny": Spec("tiny", B=1, H=8, T=4, prefix=[256], num_slots=4096, tree="chain", seed=0),
        "tp8": Spec("tp8", B=1, H=8, T=16, prefix=[4096], num_slots=1 << 20, seed=1),
        "fullh": Spec("fullh", B=1, H=64, T=16, prefix=[65536], num_slots=1 << 20, seed=2),
        "long": Spec("long", B=1, H=8, T=32, prefix=[200000], num_slots=1 << 18, seed=3),
        "batched": Spec("batched", B=8, H=64, T=16, prefix=[], num_slots=1 << 20, seed=4),
    }
    if name not in base:
        raise KeyError(name)
    s = base[name]
    if name == "batched" and "prefix" not in over:
        g = torch.Generator().manual_seed(s.seed + 1000)
        s = replace(s, prefix=[int(x) for x in torch.randint(1024, 65537, (s.B,), generator=g)])
    return replace(s, **over)


def sweep_spec(P: int, H: int = 8, T: int = 16, layout: str = "scattered", seed: int = 5) -> Spec:
    """Sweep points: one request, prefix P, pool large enough to scatter into."""
    slots = 1 << 20
    while slots < 2 * (P + T):
        slots <<= 1
    return Spec(f"sweep_H{H}_T{T}_P{P}_{layout}", B=1, H=H, T=T, prefix=[P], num_slots=slots,
                layout=layout, seed=seed)


def _bf16_normal(shape, g: torch.Generator, chunk_rows: int = 1 << 16) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g).to(torch.bfloat16)
    return out


def make_parents(T: int, tree: str, g: torch.Generator) -> torch.Tensor:
    if tree == "chain":
        return torch.arange(-1, T - 1, dtype=torch.int32)
    if tree == "random":
        par = torch.empty(T, dtype=torch.int32)
        for i in range(T):
            par[i] = int(torch.randint(0, i + 1, (1,), generator=g)) - 1
        return par
    if tree == "flat":
        return torch.full((T,), -1, dtype=torch.int32)
    raise ValueError(tree)


def make(s: Spec) -> Workload:
    """Draw one step's inputs for ``s`` (deterministic in ``s.seed``)."""
    g = torch.Generator().manual_seed(s.seed)
    N = s.n_keys()
    total = sum(N)
    if total > s.num_slots:
        raise ValueError("pool too small for the requested keys")
    q = _bf16_normal((s.B * s.T, s.H, D_QK), g)
    parents = torch.stack([make_parents(s.T, s.tree, g) for _ in range(s.B)]).to(torch.int32)
    indptr = torch.zeros(s.B + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(N, dtype=torch.int64), 0).to(torch.int32)
    kv_start = None
    if s.layout == "scattered":
        slots = torch.randperm(s.num_slots, generator=g)[:total].to(torch.int32)
    elif s.layout == "contiguous":
        # disjoint contiguous ranges at seeded offsets, in request order
        free = s.num_slots - total
        cuts = sorted(int(x) for x in torch.randint(0, free + 1, (s.B,), generator=g))
        starts, pos = [], 0
        for b in range(s.B):
            pos = max(pos, cuts[b])
            starts.append(pos)
            pos += N[b]
        kv_start = torch.tensor(starts, dtype=torch.int64)
        slots = torch.cat([torch.arange(starts[b], starts[b] + N[b], dtype=torch.int32)
                           for b in range(s.B)])
    else:
        raise ValueError(s.layout)
    pool = _bf16_normal((s.num_slots, s.row_stride), g)
    if s.canary:
        used = torch.zeros(s.num_slots, dtype=torch.bool)
        used[slots.long()] = True
        pool.view(torch.int16)[~used] = BF16_NAN_BITS
        # padding columns beyond the 576 used ones are never read either
        if s.row_stride > D_QK:
            pool.view(torch.int16)[:, D_QK:] = BF16_NAN_BITS
    return Workload(spec=s, q=q, kv_pool=pool, slot_idx=slots, kv_indptr=indptr,
                    prefix_len=torch.tensor(s.prefix, dtype=torch.int32), parents=parents,
                    kv_start=kv_start)


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
