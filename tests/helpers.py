"""Small structured-input builders for the oracle pins (host numpy only)."""
from __future__ import annotations

import numpy as np


def bf16_bits(x) -> np.ndarray:
    """Bit patterns of values that are exactly representable in bf16."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def bf16_round_bits(x) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (for random test data)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bits_to_float(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def make_table(lengths, page, shuffle_seed=None, extra_blocks=0):
    """Block table for sequences of the given cache lengths (tokens)."""
    nblk = [max(1, -(-L // page)) for L in lengths]
    NB = sum(nblk) + extra_blocks
    ids = np.arange(NB, dtype=np.int32)
    if shuffle_seed is not None:
        ids = np.random.default_rng(shuffle_seed).permutation(NB).astype(np.int32)
    table = np.full((len(lengths), max(nblk)), -1, dtype=np.int32)
    first = 0
    for b, n in enumerate(nblk):
        table[b, :n] = ids[first:first + n]
        first += n
    return table, NB


def paged_cache(logical, table, NB, page, fill=0.0):
    """Scatter per-sequence logical arrays [L_b, Hkv, d] (float) into a paged cache
    [NB, Hkv, page, d] of bf16 bit patterns."""
    Hkv, d = logical[0].shape[1:]
    cache = np.full((NB, Hkv, page, d), fill, dtype=np.float32)
    for b, arr in enumerate(logical):
        for j in range(arr.shape[0]):
            blk = table[b, j // page]
            cache[blk, :, j % page, :] = arr[j]
    return bf16_bits(cache)
