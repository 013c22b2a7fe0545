"""Workload shapes for the verify / select / sparse-draft path.

Each entry is a synthetic stand-in for one of the workloads the Vegas and Dustin
summaries evaluate on (Qwen3 and Qwen2.5 attention geometry, 32K-128K contexts,
batch 1-16).  No dataset or model weight is involved: q, K and V are seeded
N(0, 1) values rounded to bf16, with planted heavy-hitter keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # sequences in the batch
    P: int                 # prefix length P_b (tokens before the verify block)
    Hq: int                # query heads
    Hkv: int               # KV heads (GQA groups)
    d: int                 # head dimension
    gamma: int             # draft tokens per iteration; the verify block has gamma+1 rows
    k: int                 # selection budget, including the protected tokens
    n_sink: int            # attention-sink prefix tokens always kept
    n_recent: int          # most recent prefix tokens always kept
    page: int = 16         # tokens per KV-cache page
    planted_frac: float = 0.0   # fraction of prefix positions given a heavy-hitter key
    planted_count: int = 0      # or: an exact number of heavy-hitter positions
    bursts: int = 0             # or: this many bursts of burst_len heavy-hitter tokens
    burst_len: int = 64
    contiguous: bool = False    # identity block table instead of a shuffled one
    seed: int = 0
    per_seq_seed_base: Optional[int] = None  # sequence b uses seed base + b
    layers: int = 1
    iterations: int = 1
    prefix_lens: Optional[Tuple[int, ...]] = None  # ragged batch: explicit P_b per sequence

    @property
    def R(self) -> int:
        return self.gamma + 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def prefix(self) -> Tuple[int, ...]:
        if self.prefix_lens is not None:
            return tuple(self.prefix_lens)
        return (self.P,) * self.B

    @property
    def P_max(self) -> int:
        return max(self.prefix())

    def seq_seed(self, b: int) -> int:
        if self.per_seq_seed_base is not None:
            return self.per_seq_seed_base + b
        return self.seed * 1000003 + b

    def capacity(self, P_b: int) -> int:
        """Cache tokens reserved for a sequence: prefix, verify block and a draft tail."""
        return P_b + 2 * self.gamma + 2

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Tiny single layer (oracle-sized): contiguous cache, 8 planted keys.
TINY = Workload("tiny_p512_d64", B=1, P=512, Hq=4, Hkv=1, d=64, gamma=3, k=64, n_sink=4,
                n_recent=16, planted_count=8, contiguous=True, seed=1)

# Qwen3-8B attention geometry, one layer, 32K prefix, shuffled paged cache.
QWEN3_8B_32K = Workload("qwen3_8b_32k", B=1, P=32768, Hq=32, Hkv=8, d=128, gamma=4, k=2048,
                        n_sink=16, n_recent=256, planted_frac=0.01, seed=2)

# Qwen2.5-72B attention geometry, batch 16 at 32K each, per-sequence seeds.
QWEN25_72B_B16_32K = Workload("qwen25_72b_b16_32k", B=16, P=32768, Hq=64, Hkv=8, d=128,
                              gamma=5, k=512, n_sink=4, n_recent=64, planted_frac=0.005,
                              seed=3, per_seq_seed_base=3000)

# 128K context, Qwen3-8B geometry, heavy hitters in 64-token bursts.
LONG_128K = Workload("qwen3_8b_128k_bursts", B=1, P=131072, Hq=32, Hkv=8, d=128, gamma=6,
                     k=8192, n_sink=16, n_recent=512, bursts=20, burst_len=64, seed=4)

# 36-layer attention-only loop in Qwen3-8B geometry (sink/recent as the 32K layer).
LOOP_36L = Workload("qwen3_8b_36layer_loop", B=4, P=65536, Hq=32, Hkv=8, d=128, gamma=5,
                    k=4096, n_sink=16, n_recent=256, planted_frac=0.01, seed=5, layers=36,
                    iterations=50)

# One layer of that loop at its initial prefix (the shape of one verification call of the
# loop; a few GB, small enough for profiler captures).
LOOP_LAYER = Workload("qwen3_8b_loop_layer", B=4, P=65536, Hq=32, Hkv=8, d=128, gamma=5,
                      k=4096, n_sink=16, n_recent=256, planted_frac=0.01, seed=5)

ALL = {w.name: w for w in (TINY, QWEN3_8B_32K, QWEN25_72B_B16_32K, LONG_128K, LOOP_36L,
                           LOOP_LAYER)}
