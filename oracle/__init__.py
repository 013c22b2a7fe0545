"""fp64 CPU oracle for verification-guided sparse self-speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path (the CUDA
library and its Python binding) never imports, loads or calls it, and this package
imports nothing from the product path.

The arithmetic lives in ``vsd_oracle.c`` (plain C, double precision, OpenMP over
independent (sequence, row, head) items).  This module compiles it with gcc into
``liboracle.so`` next to the source and wraps each function for numpy arrays.
bf16 tensors are passed as their raw 16-bit patterns (``uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``vsd_oracle.c`` into ``liboracle.so`` (OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_verify.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, I, I, I, D,
                                          P, P, P]
            lib.oracle_verify_all_rows.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, I,
                                                   D, P, P, P]
            lib.oracle_sparse_verify.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P,
                                                 I, D, P]
            lib.oracle_select_hybrid.argtypes = [I, I, P, P, P, I, I, I, I, P, P]
            lib.oracle_partial_masked.argtypes = [I, I, I, I, I, P, P, P, P]
            lib.oracle_score_from_logits.argtypes = [I, I, I, P, P, P]
            lib.oracle_score_from_partials.argtypes = [I, I, I, P, P, P]
            lib.oracle_select.argtypes = [I, I, P, P, I, I, I, P, P]
            lib.oracle_sparse_decode.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, I, P,
                                                 P, D, P]
            lib.oracle_block_topk.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, I, D, P, I,
                                              P]
            for name in ("oracle_verify", "oracle_verify_all_rows", "oracle_score_from_logits",
                         "oracle_score_from_partials", "oracle_select", "oracle_sparse_decode",
                         "oracle_sparse_verify", "oracle_select_hybrid", "oracle_partial_masked",
                         "oracle_block_topk", "oracle_num_threads"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError("%s failed with code %d" % (what, rc))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 tensors are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def verify(q, k_cache, v_cache, block_table, prefix_len, *, scale, P_max,
           row0=0, row1=None, collect=True):
    """Full-attention verification with Collect-2-Query.

    q: uint16 [B, R, Hq, d]; k_cache/v_cache: uint16 [NB, Hkv, page, d];
    block_table: [B, max_blocks]; prefix_len: [B].
    Returns (out [B,R,Hq,d], logits [B,2,Hq,P_max] or None, partial [B,Hkv,P_max] or None)
    as float64; positions j >= P_b of logits/partial are 0.
    """
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    bt = _i32(block_table)
    pl = _i32(prefix_len)
    B, R, Hq, d = q.shape
    NB, Hkv, page, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and bt.shape[0] == B
    if row1 is None:
        row1 = R - 1
    out = np.zeros((B, R, Hq, d), dtype=np.float64)
    logits = np.zeros((B, 2, Hq, P_max), dtype=np.float64) if collect else None
    partial = np.zeros((B, Hkv, P_max), dtype=np.float64) if collect else None
    rc = _load().oracle_verify(B, Hq, Hkv, d, page, bt.shape[1], NB, R, _ptr(q), _ptr(k_cache),
                               _ptr(v_cache), _ptr(bt), _ptr(pl), int(row0), int(row1),
                               int(P_max), float(scale),
                               _ptr(logits) if collect else None,
                               _ptr(partial) if collect else None, _ptr(out))
    _check(rc, "oracle_verify")
    return out, logits, partial


def verify_all_rows(q, k_cache, v_cache, block_table, prefix_len, *, scale, P_max):
    """Full-attention verification collecting every verify row (the selection equation
    as printed).  Returns (out [B,R,Hq,d], logits [B,R,Hq,P_max], partial [B,Hkv,P_max])
    as float64; positions j >= P_b of logits/partial are 0."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    bt = _i32(block_table)
    pl = _i32(prefix_len)
    B, R, Hq, d = q.shape
    NB, Hkv, page, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and bt.shape[0] == B
    out = np.zeros((B, R, Hq, d), dtype=np.float64)
    logits = np.zeros((B, R, Hq, P_max), dtype=np.float64)
    partial = np.zeros((B, Hkv, P_max), dtype=np.float64)
    rc = _load().oracle_verify_all_rows(B, Hq, Hkv, d, page, bt.shape[1], NB, R, _ptr(q),
                                        _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(pl),
                                        int(P_max), float(scale), _ptr(logits), _ptr(partial),
                                        _ptr(out))
    _check(rc, "oracle_verify_all_rows")
    return out, logits, partial


def score_from_logits(logits, prefix_len):
    logits = _f64(logits)
    pl = _i32(prefix_len)
    B, two, Hq, P_max = logits.shape
    assert two == 2
    score = np.zeros((B, P_max), dtype=np.float64)
    _check(_load().oracle_score_from_logits(B, Hq, P_max, _ptr(logits), _ptr(pl), _ptr(score)),
           "oracle_score_from_logits")
    return score


def score_from_partials(partial, prefix_len):
    partial = _f64(partial)
    pl = _i32(prefix_len)
    n_rows, Hkv, P_max = partial.shape
    score = np.zeros((n_rows, P_max), dtype=np.float64)
    _check(_load().oracle_score_from_partials(n_rows, Hkv, P_max, _ptr(partial), _ptr(pl),
                                              _ptr(score)), "oracle_score_from_partials")
    return score


def select(score, prefix_len, *, k, n_sink, n_recent):
    """Protected top-k.  score: [n_rows, P_max].  Returns (idx [n_rows,k] int32, n_sel)."""
    score = _f64(score)
    pl = _i32(prefix_len)
    n_rows, P_max = score.shape
    idx = np.full((n_rows, k), -1, dtype=np.int32)
    n_sel = np.zeros((n_rows,), dtype=np.int32)
    _check(_load().oracle_select(n_rows, P_max, _ptr(score), _ptr(pl), int(k), int(n_sink),
                                 int(n_recent), _ptr(idx), _ptr(n_sel)), "oracle_select")
    return idx, n_sel


def sparse_decode(q, k_cache, v_cache, block_table, idx, n_sel, tail_start, seq_len, *, scale):
    """Sparse draft-step attention.  q: uint16 [B, Hq, d]; idx: [B, k_max]."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    bt = _i32(block_table)
    if idx is None:  # no selected positions: the tail alone
        idx = np.zeros((q.shape[0], 0), dtype=np.int32)
        n_sel = np.zeros((q.shape[0],), dtype=np.int32)
    idx = _i32(idx)
    ns = _i32(n_sel)
    ts = _i32(tail_start)
    sl = _i32(seq_len)
    B, Hq, d = q.shape
    NB, Hkv, page, _ = k_cache.shape
    out = np.zeros((B, Hq, d), dtype=np.float64)
    k_max = idx.shape[1] if idx.ndim == 2 else 0
    _check(_load().oracle_sparse_decode(B, Hq, Hkv, d, page, bt.shape[1], NB, _ptr(q),
                                        _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(idx),
                                        _ptr(ns), k_max, _ptr(ts), _ptr(sl), float(scale),
                                        _ptr(out)), "oracle_sparse_decode")
    return out


def sparse_verify(q, k_cache, v_cache, block_table, prefix_len, idx, n_sel, *, scale):
    """Sparse verification: verify row t of sequence b attends idx[b, :n_sel[b]] and
    the verify block positions P_b .. P_b + t.  q: uint16 [B, R, Hq, d]; idx [B, k_max].
    Returns out [B, R, Hq, d] float64."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    bt = _i32(block_table)
    pl = _i32(prefix_len)
    idx = _i32(idx)
    ns = _i32(n_sel)
    B, R, Hq, d = q.shape
    NB, Hkv, page, _ = k_cache.shape
    out = np.zeros((B, R, Hq, d), dtype=np.float64)
    _check(_load().oracle_sparse_verify(B, Hq, Hkv, d, page, bt.shape[1], NB, R, _ptr(q),
                                        _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(pl),
                                        _ptr(idx), _ptr(ns), idx.shape[1], float(scale),
                                        _ptr(out)), "oracle_sparse_verify")
    return out


def select_hybrid(score_target, score_draft, prefix_len, *, k, m, n_sink, n_recent):
    """Dustin's hybrid budget: protected sinks and recent window, then the top-m by the
    draft signal, then the rest by the target signal.  Returns (idx [n_rows, k], n_sel)."""
    st = _f64(score_target)
    sd = _f64(score_draft)
    pl = _i32(prefix_len)
    n_rows, P_max = st.shape
    assert sd.shape == st.shape
    idx = np.full((n_rows, k), -1, dtype=np.int32)
    n_sel = np.zeros((n_rows,), dtype=np.int32)
    _check(_load().oracle_select_hybrid(n_rows, P_max, _ptr(st), _ptr(sd), _ptr(pl), int(k),
                                        int(m), int(n_sink), int(n_recent), _ptr(idx),
                                        _ptr(n_sel)), "oracle_select_hybrid")
    return idx, n_sel


def partial_masked(logits, prefix_len, head_mask, Hkv):
    """Per-KV-group partial scores over the heads with head_mask[h] != 0.
    logits: [B, C, Hq, P_max] (C collected rows).  Returns [B, Hkv, P_max]."""
    lg = _f64(logits)
    pl = _i32(prefix_len)
    hm = np.ascontiguousarray(np.asarray(head_mask, dtype=np.uint8))
    B, C, Hq, P_max = lg.shape
    partial = np.zeros((B, Hkv, P_max), dtype=np.float64)
    _check(_load().oracle_partial_masked(B, C, Hq, Hkv, P_max, _ptr(lg), _ptr(pl), _ptr(hm),
                                         _ptr(partial)), "oracle_partial_masked")
    return partial


def block_topk(q, k_cache, block_table, prefix_len, *, kb, scale, page_blocks_max=None):
    """Per-query block top-k: block scores r [B, R, Hq, page_blocks_max] (the scaled dot
    product of each query with each prefix page's mean key; 0 past the prefix) and the
    kb best pages of every (b, t, h), ascending, padded with -1: blocks [B, R, Hq, kb]."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    bt = _i32(block_table)
    pl = _i32(prefix_len)
    B, R, Hq, d = q.shape
    NB, Hkv, page, d2 = k_cache.shape
    assert d2 == d and bt.shape[0] == B
    if page_blocks_max is None:
        page_blocks_max = max([(int(p) + page - 1) // page for p in pl] + [1])
    scores = np.zeros((B, R, Hq, page_blocks_max), dtype=np.float64)
    blocks = np.full((B, R, Hq, kb), -1, dtype=np.int32)
    _check(_load().oracle_block_topk(B, Hq, Hkv, d, page, bt.shape[1], NB, R, _ptr(q),
                                     _ptr(k_cache), _ptr(bt), _ptr(pl), int(kb), float(scale),
                                     _ptr(scores), int(page_blocks_max), _ptr(blocks)),
           "oracle_block_topk")
    return scores, blocks
