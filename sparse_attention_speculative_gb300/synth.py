"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and lays them out; it contains none of the
method's arithmetic (no attention, no scoring, no selection).  It imports neither
the CUDA binding nor the oracle.

Recipe (one sequence b, seed = workload.seq_seed(b)):
  * q (verify rows) ~ N(0,1) [R, Hq, d]; K, V ~ N(0,1) [capacity, Hkv, d];
    draft queries ~ N(0,1) [gamma, Hq, d]; all drawn in fp32 then rounded to bf16.
  * heavy hitters: at each planted prefix position j and every KV head g,
    K[j, g] += 3 * sqrt(d) * u_g where u_g is the unit vector along the sum of the
    group's R * G verify query rows.  This raises those keys' scaled logits by
    about 3 * |sum q| / (R * G) ~ 7 above the N(0,1) background.
  * positions: `planted_count` or round(planted_frac * P_b) distinct positions drawn
    uniformly from [0, P_b), or `bursts` runs of `burst_len` tokens at uniform
    offsets.
  * paging: sequence b owns ceil(capacity / page) pages; the physical block of
    each page is a seeded permutation of all blocks (identity when `contiguous`).
    Unused block-table entries are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional

import torch

from .workloads import Workload


@dataclass
class Batch:
    """One batch of inputs for a single layer, all tensors on one device."""
    w: Workload
    q: torch.Tensor            # bf16 [B, R, Hq, d]
    q_draft: torch.Tensor      # bf16 [gamma, B, Hq, d]
    k_cache: torch.Tensor      # bf16 [NB, Hkv, page, d]
    v_cache: torch.Tensor      # bf16 [NB, Hkv, page, d]
    block_table: torch.Tensor  # int32 [B, max_blocks]
    prefix_len: torch.Tensor   # int32 [B]
    planted: List[torch.Tensor]  # per sequence: int64 planted prefix positions

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _planted_positions(w: Workload, P_b: int, gen: torch.Generator, device) -> torch.Tensor:
    if P_b <= 0:
        return torch.zeros((0,), dtype=torch.int64, device=device)
    if w.bursts > 0:
        span = max(P_b - w.burst_len, 1)
        starts = torch.randint(0, span, (w.bursts,), generator=gen, device=device)
        offs = torch.arange(min(w.burst_len, P_b), device=device)
        pos = (starts[:, None] + offs[None, :]).reshape(-1)
        return torch.unique(pos.clamp_(max=P_b - 1))
    n = w.planted_count if w.planted_count > 0 else int(round(w.planted_frac * P_b))
    n = min(n, P_b)
    if n == 0:
        return torch.zeros((0,), dtype=torch.int64, device=device)
    return torch.sort(torch.randperm(P_b, generator=gen, device=device)[:n]).values


def make_batch(w: Workload, device="cpu", layer: int = 0,
               prefix_lens: Optional[List[int]] = None, extra_capacity: int = 0) -> Batch:
    """Build one layer's seeded inputs for workload `w` on `device`.  Each sequence's
    cache holds `extra_capacity` more tokens than one iteration needs (for loops that
    append the accepted tokens of several iterations)."""
    device = torch.device(device)
    prefix = list(prefix_lens) if prefix_lens is not None else list(w.prefix())
    B, R, Hq, Hkv, d, page = w.B, w.R, w.Hq, w.Hkv, w.d, w.page
    assert len(prefix) == B and Hq % Hkv == 0
    G = Hq // Hkv
    caps = [w.capacity(p) + extra_capacity for p in prefix]
    nblk = [math.ceil(c / page) for c in caps]
    max_blocks = max(nblk)
    NB = sum(nblk)

    tgen = torch.Generator(device=device)
    tgen.manual_seed(w.seed * 7919 + layer * 104729 + 17)
    if w.contiguous:
        perm = torch.arange(NB, device=device)
    else:
        perm = torch.randperm(NB, generator=tgen, device=device)
    block_table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=device)
    k_cache = torch.empty((NB, Hkv, page, d), dtype=torch.bfloat16, device=device)
    v_cache = torch.empty_like(k_cache)
    q = torch.empty((B, R, Hq, d), dtype=torch.bfloat16, device=device)
    q_draft = torch.empty((w.gamma, B, Hq, d), dtype=torch.bfloat16, device=device)
    planted = []
    first = 0
    for b in range(B):
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seq_seed(b) * 131 + layer)
        blocks = perm[first:first + nblk[b]]
        first += nblk[b]
        block_table[b, :nblk[b]] = blocks.to(torch.int32)
        qb = torch.randn((R, Hq, d), generator=gen, device=device)
        kb = torch.randn((nblk[b] * page, Hkv, d), generator=gen, device=device)
        vb = torch.randn((nblk[b] * page, Hkv, d), generator=gen, device=device)
        qd = torch.randn((w.gamma, Hq, d), generator=gen, device=device)
        pos = _planted_positions(w, prefix[b], gen, device)
        if pos.numel() > 0:
            # direction of the group's verify queries, per KV head: [Hkv, d]
            qsum = qb.bfloat16().float().reshape(R, Hkv, G, d).sum(dim=(0, 2))
            u = qsum / qsum.norm(dim=-1, keepdim=True).clamp_min(1e-12)
            kb[pos] += 3.0 * math.sqrt(d) * u[None, :, :]
        q[b] = qb.to(torch.bfloat16)
        q_draft[:, b] = qd.to(torch.bfloat16)
        paged_k = kb.to(torch.bfloat16).reshape(nblk[b], page, Hkv, d).permute(0, 2, 1, 3)
        paged_v = vb.to(torch.bfloat16).reshape(nblk[b], page, Hkv, d).permute(0, 2, 1, 3)
        k_cache[blocks] = paged_k
        v_cache[blocks] = paged_v
        planted.append(pos)
    prefix_len = torch.tensor(prefix, dtype=torch.int32, device=device)
    return Batch(w, q, q_draft, k_cache, v_cache, block_table, prefix_len, planted)


def to_u16(t: torch.Tensor):
    """Raw bit patterns of a bf16 tensor as a host numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def host_arrays(batch: Batch) -> Dict[str, object]:
    """Host copies of a batch in the form the oracle takes."""
    return dict(
        q=to_u16(batch.q),
        q_draft=to_u16(batch.q_draft),
        k_cache=to_u16(batch.k_cache),
        v_cache=to_u16(batch.v_cache),
        block_table=batch.block_table.cpu().numpy(),
        prefix_len=batch.prefix_len.cpu().numpy(),
    )


def seeded_bf16(shape, seed: int, device) -> torch.Tensor:
    """N(0,1) values of `shape` from a generator seeded with `seed`, rounded to bf16."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(shape, generator=gen, device=device).to(torch.bfloat16)


def write_tokens(batch: Batch, b: int, positions: torch.Tensor, k_rows: torch.Tensor,
                 v_rows: torch.Tensor) -> None:
    """Store K/V rows [n, Hkv, d] of sequence b at logical token positions (int64 [n])
    through its block table (the cache append of a decode loop; plain indexing)."""
    page = batch.k_cache.shape[2]
    blocks = batch.block_table[b].to(torch.int64)[positions // page]
    offs = positions % page
    batch.k_cache[blocks, :, offs, :] = k_rows
    batch.v_cache[blocks, :, offs, :] = v_rows
