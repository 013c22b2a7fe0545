"""ctypes binding of libvsd (include/vsd.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  torch supplies device memory and the current stream.  If libvsd.so is
missing the calls raise immediately; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvsd.so")

_lock = threading.Lock()
_lib = None

VSD_OK = 0
STATUS_NAMES = {
    -1: "VSD_ERR_INVALID_ARG",
    -2: "VSD_ERR_UNSUPPORTED",
    -3: "VSD_ERR_CUDA",
    -4: "VSD_ERR_WORKSPACE",
    -5: "VSD_ERR_TIMEOUT",
}
DEV_BAD_BLOCK = 0x1
DEV_BAD_INDEX = 0x2
DEV_BAD_LENGTH = 0x4
DEV_TIMEOUT = 0x8
STEP_RECORD_ROWS = 0x1
STEP_REUSE_ROWS = 0x2
STEP_EARLY_GATHER = 0x4
SPARSE_VERIFY_EARLY_GATHER = 0x4
VERIFY_EARLY_PREFETCH = 0x4


class VsdError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = "%s failed: %s" % (what, STATUS_NAMES.get(status, str(status)))
        if status == -3 and _lib is not None:
            msg += " (cudaError %d)" % _lib.vsd_last_cuda_error()
        super().__init__(msg)


class Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("num_blocks", ctypes.c_int)]


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libvsd.so (built by ``sparse_attention_speculative_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError("libvsd.so is not built (%s); run "
                               "`python -m sparse_attention_speculative_gb300.build`" % path)
        lib = ctypes.CDLL(path)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        GP = ctypes.POINTER(Geom)
        lib.vsd_verify_workspace_size.argtypes = [GP, I, I, ctypes.POINTER(SZ)]
        lib.vsd_verify_attn_collect.argtypes = [GP, I, P, P, P, P, P, I, I, I, F, P, P, P, P, SZ, P]
        lib.vsd_verify_attn_collect_noalloc.argtypes = [GP, I, P, P, P, P, P, I, I, I, F, P, P,
                                                        P, P]
        lib.vsd_verify_attn_collect_all.argtypes = [GP, I, P, P, P, P, P, I, F, P, P, P, P, SZ,
                                                    P]
        lib.vsd_sparse_verify_workspace_size.argtypes = [GP, I, I, ctypes.POINTER(SZ)]
        lib.vsd_sparse_verify_attn.argtypes = [GP, I, P, P, P, P, P, P, P, I, ctypes.c_uint, F, P,
                                                P, SZ, P]
        lib.vsd_verify_attn_collect_srh.argtypes = [GP, I, P, P, P, P, P, I, I, P, I, F, P, P, P,
                                                    P, SZ, P]
        lib.vsd_select_hybrid_workspace_size.argtypes = [I, I, ctypes.POINTER(SZ)]
        lib.vsd_select_topk_hybrid.argtypes = [I, I, P, I, P, P, I, I, I, I, I, P, P, P, SZ, P]
        lib.vsd_select_workspace_size.argtypes = [I, I, I, I, ctypes.POINTER(SZ)]
        lib.vsd_select_topk.argtypes = [I, I, P, P, I, I, I, I, P, P, P, P, SZ, P]
        lib.vsd_sparse_workspace_size.argtypes = [GP, I, I, ctypes.POINTER(SZ)]
        lib.vsd_sparse_decode_attn.argtypes = [GP, P, P, P, P, P, P, I, P, P, I, F, P, P, SZ, P]
        lib.vsd_verify_attn_collect_scored.argtypes = [GP, I, P, P, P, P, P, I, I, I, F, P, P,
                                                       P, P, I, I, ctypes.c_uint, P, P, P, P, SZ,
                                                       P]
        lib.vsd_select_topk_scored.argtypes = [I, P, P, P, I, I, I, I, P, P, P]
        lib.vsd_page_key_means.argtypes = [GP, P, P, P, P, I, P, P]
        lib.vsd_copy.argtypes = [P, P, SZ, P]
        lib.vsd_append_kv.argtypes = [GP, I, P, P, P, P, I, P, P, P]
        lib.vsd_sparse_decode_attn_step.argtypes = [GP, P, P, P, P, P, P, P, P, I, P, P, I, P,
                                                    ctypes.c_uint, F, P, P, SZ, P]
        lib.vsd_advance_lengths.argtypes = [I, I, P, I, P, P, P, I, P, P]
        lib.vsd_block_topk.argtypes = [GP, I, P, P, P, I, I, F, P, P, P]
        lib.vsd_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
        lib.vsd_get_error_string.argtypes = [I]
        lib.vsd_get_error_string.restype = ctypes.c_char_p
        lib.vsd_last_cuda_error.argtypes = []
        for name in ("vsd_verify_workspace_size", "vsd_verify_attn_collect",
                     "vsd_verify_attn_collect_all", "vsd_sparse_verify_workspace_size",
                     "vsd_verify_attn_collect_srh", "vsd_select_hybrid_workspace_size",
                     "vsd_select_topk_hybrid",
                     "vsd_sparse_verify_attn",
                     "vsd_verify_attn_collect_noalloc",
                     "vsd_select_workspace_size", "vsd_select_topk", "vsd_sparse_workspace_size",
                     "vsd_sparse_decode_attn", "vsd_page_key_means", "vsd_block_topk",
                     "vsd_verify_attn_collect_scored", "vsd_select_topk_scored", "vsd_copy",
                     "vsd_append_kv", "vsd_advance_lengths", "vsd_sparse_decode_attn_step",
                     "vsd_read_device_status", "vsd_last_cuda_error"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(rc: int, what: str) -> None:
    if rc != VSD_OK:
        raise VsdError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def geom_for(B: int, Hq: int, k_cache: torch.Tensor, block_table: torch.Tensor) -> Geom:
    NB, Hkv, page, d = k_cache.shape
    return Geom(B, Hq, Hkv, d, page, int(block_table.shape[1]), NB)


_ws_cache = {}


def _workspace(nbytes: int, device, tag: str) -> Optional[torch.Tensor]:
    """Cached device scratch, one buffer per (call kind, device, size), zero-filled
    when allocated as the workspace contract asks (every call leaves it reusable by
    calls of the same kind; the kinds whose counters are laid out per (sequence, KV
    head) carry B * Hkv in their tag)."""
    if nbytes == 0:
        return None
    key = (tag, str(device), nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    off = (-ws.data_ptr()) % 256
    return ws[off:off + nbytes]


def vsd_verify_workspace_size(geom: Geom, R: int, P_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().vsd_verify_workspace_size(ctypes.byref(geom), R, P_max, ctypes.byref(out)),
           "vsd_verify_workspace_size")
    return int(out.value)


def vsd_verify_attn_collect(q, k_cache, v_cache, block_table, prefix_len, *, P_max: int,
                            scale: float, row0: int = 0, row1: Optional[int] = None,
                            logits=None, partial=None, out=None, collect: bool = True,
                            workspace=None, stream=None):
    """Verification attention + Collect-2-Query.  Returns (out, logits, partial)."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_table, torch.int32, "block_table")
    _need(prefix_len, torch.int32, "prefix_len")
    geom = geom_for(B, Hq, k_cache, block_table)
    if row1 is None:
        row1 = R - 1
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if collect:
        if logits is None:
            logits = torch.empty((B, 2, Hq, P_max), dtype=torch.float32, device=dev)
        if partial is None:
            partial = torch.empty((B, geom.Hkv, P_max), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _workspace(vsd_verify_workspace_size(geom, R, P_max), dev, "verify")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_verify_attn_collect(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
                                     int(row0), int(row1), int(P_max), float(scale),
                                     _ptr(logits), _ptr(partial), _ptr(out), _ptr(workspace),
                                     ws_bytes, _stream(stream))
    _check(rc, "vsd_verify_attn_collect")
    return out, logits, partial


def vsd_verify_attn_collect_all(q, k_cache, v_cache, block_table, prefix_len, *, P_max: int,
                                scale: float, logits=None, partial=None, out=None,
                                collect: bool = True, workspace=None, stream=None):
    """Verification collecting every verify row (logits fp32 [B, R, Hq, P_max]; the
    partial scores sum all R rows).  Returns (out, logits, partial)."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_table, torch.int32, "block_table")
    _need(prefix_len, torch.int32, "prefix_len")
    geom = geom_for(B, Hq, k_cache, block_table)
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if collect:
        if logits is None:
            logits = torch.empty((B, R, Hq, P_max), dtype=torch.float32, device=dev)
        if partial is None:
            partial = torch.empty((B, geom.Hkv, P_max), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _workspace(vsd_verify_workspace_size(geom, R, P_max), dev, "verify")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_verify_attn_collect_all(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
                                         int(P_max), float(scale), _ptr(logits), _ptr(partial),
                                         _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vsd_verify_attn_collect_all")
    return out, logits, partial


def vsd_verify_attn_collect_noalloc(q, k_cache, v_cache, block_table, prefix_len, *,
                                    P_max: int, scale: float, row0: int = 0,
                                    row1: Optional[int] = None, logits=None, partial=None,
                                    out=None, collect: bool = True, stream=None):
    """vsd_verify_attn_collect with the library's fixed device scratch instead of a
    workspace (the C call allocates nothing; outputs are allocated here when not
    given).  Returns (out, logits, partial)."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_table, torch.int32, "block_table")
    _need(prefix_len, torch.int32, "prefix_len")
    geom = geom_for(B, Hq, k_cache, block_table)
    if row1 is None:
        row1 = R - 1
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if collect:
        if logits is None:
            logits = torch.empty((B, 2, Hq, P_max), dtype=torch.float32, device=dev)
        if partial is None:
            partial = torch.empty((B, geom.Hkv, P_max), dtype=torch.float32, device=dev)
    rc = lib.vsd_verify_attn_collect_noalloc(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), _ptr(block_table),
                                             _ptr(prefix_len), int(row0), int(row1),
                                             int(P_max), float(scale), _ptr(logits),
                                             _ptr(partial), _ptr(out), _stream(stream))
    _check(rc, "vsd_verify_attn_collect_noalloc")
    return out, logits, partial


def vsd_select_topk(partial, prefix_len, *, k: int, n_sink: int, n_recent: int, idx=None,
                    n_sel=None, scores_out=None, want_scores: bool = False,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor, Optional[torch.Tensor]]:
    """Protected top-k over the aggregated score.  partial: fp32 [n_rows, Hkv, P_max]."""
    lib = load()
    _need(partial, torch.float32, "partial")
    _need(prefix_len, torch.int32, "prefix_len")
    n_rows, Hkv, P_max = partial.shape
    dev = partial.device
    if idx is None:
        idx = torch.empty((n_rows, k), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    if want_scores and scores_out is None:
        scores_out = torch.empty((n_rows, P_max), dtype=torch.float32, device=dev)
    rc = lib.vsd_select_topk(n_rows, Hkv, _ptr(partial), _ptr(prefix_len), P_max, int(k),
                             int(n_sink), int(n_recent), _ptr(idx), _ptr(n_sel),
                             _ptr(scores_out), None, 0, _stream(stream))
    _check(rc, "vsd_select_topk")
    return idx, n_sel, scores_out


def vsd_sparse_workspace_size(geom: Geom, k_max: int, max_tail: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().vsd_sparse_workspace_size(ctypes.byref(geom), int(k_max), int(max_tail),
                                            ctypes.byref(out)), "vsd_sparse_workspace_size")
    return int(out.value)


def vsd_sparse_decode_attn(q, k_cache, v_cache, block_table, idx, n_sel, tail_start, seq_len,
                           *, scale: float, max_tail: int, out=None, workspace=None,
                           stream=None):
    """Sparse draft-step attention.  q: bf16 [B, Hq, d]; idx: int32 [B, k_max] or None."""
    lib = load()
    B, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(tail_start, torch.int32, "tail_start")
    _need(seq_len, torch.int32, "seq_len")
    geom = geom_for(B, Hq, k_cache, block_table)
    k_max = 0 if idx is None else int(idx.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = _workspace(vsd_sparse_workspace_size(geom, k_max, max_tail), q.device,
                               "sparse:%d" % (geom.B * geom.Hkv))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_sparse_decode_attn(ctypes.byref(geom), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_table), _ptr(idx), _ptr(n_sel), k_max,
                                    _ptr(tail_start), _ptr(seq_len), int(max_tail), float(scale),
                                    _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vsd_sparse_decode_attn")
    return out


def vsd_read_device_status(stream=None) -> int:
    flags = ctypes.c_uint(0)
    _check(load().vsd_read_device_status(_stream(stream), ctypes.byref(flags)),
           "vsd_read_device_status")
    return int(flags.value)


def vsd_sparse_verify_workspace_size(geom: Geom, R: int, k_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().vsd_sparse_verify_workspace_size(ctypes.byref(geom), int(R), int(k_max),
                                                   ctypes.byref(out)),
           "vsd_sparse_verify_workspace_size")
    return int(out.value)


def vsd_sparse_verify_attn(q, k_cache, v_cache, block_table, prefix_len, idx, n_sel, *,
                           scale: float, flags: int = 0, out=None, workspace=None, stream=None):
    """Sparse verification: verify row t attends idx[b, :n_sel[b]] and the verify block
    positions P_b .. P_b + t.  q: bf16 [B, R, Hq, d]; idx: int32 [B, k_max].  flags: 0 or
    SPARSE_VERIFY_EARLY_GATHER.  Returns out."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(prefix_len, torch.int32, "prefix_len")
    _need(idx, torch.int32, "idx")
    _need(n_sel, torch.int32, "n_sel")
    geom = geom_for(B, Hq, k_cache, block_table)
    k_max = int(idx.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = _workspace(vsd_sparse_verify_workspace_size(geom, R, k_max), q.device,
                               "sparse_verify")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_sparse_verify_attn(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_table), _ptr(prefix_len), _ptr(idx), _ptr(n_sel),
                                    k_max, int(flags), float(scale), _ptr(out), _ptr(workspace),
                                    ws_bytes, _stream(stream))
    _check(rc, "vsd_sparse_verify_attn")
    return out


def vsd_verify_attn_collect_srh(q, k_cache, v_cache, block_table, prefix_len, head_mask, *,
                                P_max: int, scale: float, row0: int = 0,
                                row1: Optional[int] = None, logits=None, partial=None,
                                out=None, workspace=None, stream=None):
    """Verification with the collected logits and partial scores restricted to the query
    heads with head_mask[h] != 0 (uint8 [Hq] on the device).  Returns (out, logits,
    partial); the logits of the other heads are left untouched."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(head_mask, torch.uint8, "head_mask")
    geom = geom_for(B, Hq, k_cache, block_table)
    if row1 is None:
        row1 = R - 1
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if logits is None:
        logits = torch.zeros((B, 2, Hq, P_max), dtype=torch.float32, device=dev)
    if partial is None:
        partial = torch.empty((B, geom.Hkv, P_max), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _workspace(vsd_verify_workspace_size(geom, R, P_max), dev, "verify")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_verify_attn_collect_srh(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
                                         int(row0), int(row1), _ptr(head_mask), int(P_max),
                                         float(scale), _ptr(logits), _ptr(partial), _ptr(out),
                                         _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vsd_verify_attn_collect_srh")
    return out, logits, partial


def vsd_select_topk_hybrid(partial_target, partial_draft, prefix_len, *, k: int, m: int,
                           n_sink: int, n_recent: int, idx=None, n_sel=None, workspace=None,
                           stream=None):
    """Dustin's hybrid budget: protected sinks and recent window, then the top-m by the
    draft score, then the rest by the target score.  partial_*: fp32 [n_rows, Hkv*, P_max]."""
    lib = load()
    _need(partial_target, torch.float32, "partial_target")
    _need(partial_draft, torch.float32, "partial_draft")
    _need(prefix_len, torch.int32, "prefix_len")
    n_rows, Hkv_t, P_max = partial_target.shape
    Hkv_d = int(partial_draft.shape[1])
    assert partial_draft.shape[0] == n_rows and partial_draft.shape[2] == P_max
    dev = partial_target.device
    if idx is None:
        idx = torch.empty((n_rows, k), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    if workspace is None:
        nb = ctypes.c_size_t(0)
        _check(lib.vsd_select_hybrid_workspace_size(n_rows, P_max, ctypes.byref(nb)),
               "vsd_select_hybrid_workspace_size")
        workspace = _workspace(int(nb.value), dev, "select_hybrid")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_select_topk_hybrid(n_rows, Hkv_t, _ptr(partial_target), Hkv_d,
                                    _ptr(partial_draft), _ptr(prefix_len), P_max, int(k), int(m),
                                    int(n_sink), int(n_recent), _ptr(idx), _ptr(n_sel),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vsd_select_topk_hybrid")
    return idx, n_sel


def page_blocks(P_max: int) -> int:
    """Pages of 16 tokens covering a prefix of P_max tokens."""
    return (int(P_max) + 15) // 16


def vsd_page_key_means(k_cache, block_table, prefix_len, *, B: int, page_blocks_max: int,
                       page_begin=None, page_means=None, stream=None):
    """Mean key of every prefix page: fp32 [B, Hkv, page_blocks_max, d] (pages from
    page_begin[b], default 0, to ceil(P_b / 16) are written).  Returns page_means."""
    lib = load()
    _need(prefix_len, torch.int32, "prefix_len")
    if page_begin is not None:
        _need(page_begin, torch.int32, "page_begin")
    Hkv, d = int(k_cache.shape[1]), int(k_cache.shape[3])
    geom = geom_for(B, Hkv, k_cache, block_table)
    if page_means is None:
        page_means = torch.zeros((B, Hkv, page_blocks_max, d), dtype=torch.float32,
                                 device=k_cache.device)
    rc = lib.vsd_page_key_means(ctypes.byref(geom), _ptr(k_cache), _ptr(block_table),
                                _ptr(prefix_len), _ptr(page_begin), int(page_blocks_max),
                                _ptr(page_means), _stream(stream))
    _check(rc, "vsd_page_key_means")
    return page_means


def vsd_block_topk(q, page_means, prefix_len, *, kb: int, scale: float, k_cache=None,
                   block_table=None, scores=None, blocks=None, stream=None):
    """Per-query page scores fp32 [B, R, Hq, page_blocks_max] and the kb best pages of
    every (b, t, h), ascending and padded with -1: int32 [B, R, Hq, kb].  q: bf16
    [B, R, Hq, d]; page_means from vsd_page_key_means.  Returns (scores, blocks)."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(page_means, torch.float32, "page_means")
    _need(prefix_len, torch.int32, "prefix_len")
    Hkv, nblk = int(page_means.shape[1]), int(page_means.shape[2])
    geom = Geom(B, Hq, Hkv, d, 16, 1, 1)
    if k_cache is not None:
        geom = geom_for(B, Hq, k_cache, block_table)
    dev = q.device
    if scores is None:
        scores = torch.zeros((B, R, Hq, nblk), dtype=torch.float32, device=dev)
    if blocks is None:
        blocks = torch.empty((B, R, Hq, kb), dtype=torch.int32, device=dev)
    rc = lib.vsd_block_topk(ctypes.byref(geom), R, _ptr(q), _ptr(page_means), _ptr(prefix_len),
                            nblk, int(kb), float(scale), _ptr(scores), _ptr(blocks),
                            _stream(stream))
    _check(rc, "vsd_block_topk")
    return scores, blocks


HIST_BINS = 4096


def vsd_verify_attn_collect_scored(q, k_cache, v_cache, block_table, prefix_len, *, P_max: int,
                                   scale: float, row0: int = 0, row1: Optional[int] = None,
                                   logits=None, partial=None, score=None, score_hist=None,
                                   n_sink: int = 0, n_recent: int = 0, flags: int = 0,
                                   k_new=None, v_new=None, out=None, workspace=None, stream=None):
    """Verification with Collect-2-Query that also sums the partial scores over the KV
    groups (score fp32 [B, P_max]) and counts the level-0 histogram (uint32-valued int32
    [B, 4096]) of the selection's candidates (the n_sink first and n_recent last prefix
    positions left out).  flags: 0 or VERIFY_EARLY_PREFETCH.  k_new, v_new: bf16
    [B, R, Hkv, d] or None: the verify block's keys and values, stored into the caches at
    P_b .. P_b + R - 1 by the call itself.  Returns (out, logits, partial, score,
    score_hist)."""
    lib = load()
    B, R, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    for name, x in (("k_new", k_new), ("v_new", v_new)):
        if x is not None:
            _need(x, torch.bfloat16, name)
    geom = geom_for(B, Hq, k_cache, block_table)
    if row1 is None:
        row1 = R - 1
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if partial is None:
        partial = torch.empty((B, geom.Hkv, P_max), dtype=torch.float32, device=dev)
    if score is None:
        score = torch.empty((B, P_max), dtype=torch.float32, device=dev)
    if score_hist is None:
        score_hist = torch.empty((B, HIST_BINS), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _workspace(vsd_verify_workspace_size(geom, R, P_max), dev, "verify")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_verify_attn_collect_scored(ctypes.byref(geom), R, _ptr(q), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
                                            int(row0), int(row1), int(P_max), float(scale),
                                            _ptr(logits), _ptr(partial), _ptr(score),
                                            _ptr(score_hist), int(n_sink), int(n_recent),
                                            int(flags), _ptr(k_new), _ptr(v_new), _ptr(out),
                                            _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "vsd_verify_attn_collect_scored")
    return out, logits, partial, score, score_hist


def vsd_select_topk_scored(score, score_hist, prefix_len, *, k: int, n_sink: int, n_recent: int,
                           idx=None, n_sel=None, stream=None):
    """The protected top-k from an aggregated score [n_rows, P_max] and its histogram
    (from vsd_verify_attn_collect_scored).  Returns (idx [n_rows, k], n_sel)."""
    lib = load()
    _need(score, torch.float32, "score")
    n_rows, P_max = score.shape
    dev = score.device
    if idx is None:
        idx = torch.empty((n_rows, k), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    rc = lib.vsd_select_topk_scored(int(n_rows), _ptr(score), _ptr(score_hist), _ptr(prefix_len),
                                    int(P_max), int(k), int(n_sink), int(n_recent), _ptr(idx),
                                    _ptr(n_sel), _stream(stream))
    _check(rc, "vsd_select_topk_scored")
    return idx, n_sel


def vsd_copy(dst, src, stream=None):
    """dst <- src (same byte size, a multiple of 16) by a kernel; either tensor may be in
    pinned host memory."""
    lib = load()
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("vsd_copy: size mismatch")
    _check(lib.vsd_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "vsd_copy")
    return dst


def vsd_append_kv(k_new, v_new, k_cache, v_cache, block_table, pos_base, *, pos_offset: int = 0,
                  stream=None):
    """Store K/V rows k_new, v_new: bf16 [B, n_new, Hkv, d] at positions
    pos_base[b] + pos_offset + t of each sequence (through the block table)."""
    lib = load()
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(pos_base, torch.int32, "pos_base")
    B, n_new = int(k_new.shape[0]), int(k_new.shape[1])
    if tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new and v_new shapes differ")
    geom = geom_for(B, int(k_cache.shape[1]), k_cache, block_table)
    rc = lib.vsd_append_kv(ctypes.byref(geom), n_new, _ptr(k_new), _ptr(v_new), _ptr(block_table),
                           _ptr(pos_base), int(pos_offset), _ptr(k_cache), _ptr(v_cache),
                           _stream(stream))
    _check(rc, "vsd_append_kv")


def vsd_advance_lengths(accepted, prefix_len, tail_start, seq_len, *, max_prefix: int,
                        prefix_copies=None, stream=None):
    """After a verification that accepted accepted[b] drafts: prefix_len += accepted + 1,
    tail_start = the old prefix, seq_len[i] = old prefix + accepted + 2 + i, and every row
    of prefix_copies ([n_copies, B]) = the new prefix.  All int32 device tensors."""
    lib = load()
    for t, name in ((accepted, "accepted"), (prefix_len, "prefix_len"),
                    (tail_start, "tail_start"), (seq_len, "seq_len")):
        _need(t, torch.int32, name)
    B = int(prefix_len.shape[0])
    gamma = int(seq_len.shape[0])
    n_copies = 0
    if prefix_copies is not None:
        _need(prefix_copies, torch.int32, "prefix_copies")
        n_copies = prefix_copies.numel() // max(B, 1)
    rc = lib.vsd_advance_lengths(B, gamma, _ptr(accepted), int(max_prefix), _ptr(prefix_len),
                                 _ptr(tail_start), _ptr(seq_len), n_copies, _ptr(prefix_copies),
                                 _stream(stream))
    _check(rc, "vsd_advance_lengths")


def vsd_sparse_decode_attn_step(q, k_cache, v_cache, block_table, idx, n_sel, tail_start, seq_len,
                                *, scale: float, max_tail: int, k_new=None, v_new=None,
                                sel_rows=None, flags: int = 0, out=None, workspace=None,
                                stream=None):
    """A draft step of a decode loop: the step's input token (k_new, v_new: bf16
    [B, Hkv, d]) is stored at seq_len - 1 and attended; sel_rows (int32 [B, k_max]) caches
    the selection's cache rows (STEP_RECORD_ROWS writes them, STEP_REUSE_ROWS reads
    them); STEP_EARLY_GATHER gathers before waiting for the preceding kernel (see
    include/vsd.h for what the caller promises with it)."""
    lib = load()
    B, Hq, d = q.shape
    _need(q, torch.bfloat16, "q")
    _need(tail_start, torch.int32, "tail_start")
    _need(seq_len, torch.int32, "seq_len")
    if k_new is not None:
        _need(k_new, torch.bfloat16, "k_new")
        _need(v_new, torch.bfloat16, "v_new")
    if sel_rows is not None:
        _need(sel_rows, torch.int32, "sel_rows")
    geom = geom_for(B, Hq, k_cache, block_table)
    k_max = 0 if idx is None else int(idx.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = _workspace(vsd_sparse_workspace_size(geom, k_max, max_tail), q.device,
                               "sparse:%d" % (geom.B * geom.Hkv))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.vsd_sparse_decode_attn_step(ctypes.byref(geom), _ptr(q), _ptr(k_new), _ptr(v_new),
                                         _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                         _ptr(idx), _ptr(n_sel), k_max, _ptr(tail_start),
                                         _ptr(seq_len), int(max_tail), _ptr(sel_rows),
                                         int(flags), float(scale), _ptr(out), _ptr(workspace),
                                         ws_bytes, _stream(stream))
    _check(rc, "vsd_sparse_decode_attn_step")
    return out
