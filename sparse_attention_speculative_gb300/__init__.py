"""Verification-guided sparse self-speculative decoding kernels for GB300 (sm_103a).

The hot path is three C-ABI calls of ``libvsd.so`` (see ``include/vsd.h``):
verification attention with Collect-2-Query, protected top-k selection over the
aggregated logits, and the sparse draft-step attention.  This package holds the
CUDA sources (``csrc/``), the in-tree build (``build.py``), the ctypes binding
(``_lib.py``), one decode iteration as a CUDA graph (``iteration.py``), decode
iterations over a multi-layer stack with the cache appends and prefix growth on the
device (``decode_loop.py``), the workload
table (``workloads.py``) and the seeded input generators (``synth.py``).
"""
from ._lib import (DEV_BAD_BLOCK, DEV_BAD_INDEX, DEV_BAD_LENGTH, DEV_TIMEOUT, Geom,  # noqa: F401
                   SPARSE_VERIFY_EARLY_GATHER, STEP_EARLY_GATHER, STEP_RECORD_ROWS,
                   VERIFY_EARLY_PREFETCH,
                   STEP_REUSE_ROWS,
                   VsdError, geom_for, load, vsd_read_device_status, vsd_select_topk,
                   vsd_sparse_decode_attn, vsd_sparse_workspace_size, vsd_verify_attn_collect,
                   vsd_select_topk_hybrid, vsd_sparse_verify_attn,
                   vsd_sparse_verify_workspace_size, vsd_verify_attn_collect_srh,
                   vsd_verify_attn_collect_all,
                   vsd_verify_attn_collect_noalloc, vsd_verify_workspace_size,
                   page_blocks, vsd_page_key_means, vsd_block_topk,
                   vsd_verify_attn_collect_scored, vsd_select_topk_scored, HIST_BINS,
                   vsd_copy, vsd_append_kv, vsd_advance_lengths, vsd_sparse_decode_attn_step)
from .decode_loop import DecodeLoop  # noqa: F401
from .iteration import IterationGraph  # noqa: F401
