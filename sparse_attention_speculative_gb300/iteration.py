"""One speculative-decoding iteration as a single CUDA graph.

A decode loop calls the same sequence of kernels every iteration: verification with
Collect-2-Query (which also sums the collected logits over the KV groups and counts
the first histogram level of that score), the protected top-k selection starting from
them, and gamma draft steps over the selection plus the dense tail.  `IterationGraph` records that sequence once -- with
the host-to-device copies of the iteration's inputs and the device-to-host copies of
its results -- and replays it with one launch per iteration.  The kernels inside are
chained by programmatic dependent launch, so each one's launch overlaps the tail of
its predecessor.  The input and result copies are kernels too (`vsd_copy`: the device
addresses pinned host memory directly over the CPU-GPU link), which cost about 1 us
per iteration where DMA copy nodes cost about 8.  All arithmetic runs in libvsd's
kernels; this module only owns buffers and the graph.

The caller fills the pinned host inputs (`h_q`, `h_q_draft`, `h_prefix_len`,
`h_tail_start`, `h_seq_len`), calls `run()`, and reads the pinned host results
(`h_out`, `h_idx`, `h_n_sel`, `h_draft_out`) once `synchronize()` (or `run(sync=True)`)
returns.  The paged caches and the block table stay on the device and are referenced,
not copied: writing new tokens into them between iterations is the caller's business.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


class IterationGraph:
    """verify -> select -> gamma draft steps (+ input/result copies) as one graph.

    Shapes: q bf16 [B, R, Hq, d]; q_draft bf16 [gamma, B, Hq, d]; prefix_len,
    tail_start int32 [B]; seq_len int32 [gamma, B] (one row per draft step);
    out bf16 [B, R, Hq, d]; idx int32 [B, k]; n_sel int32 [B];
    draft_out bf16 [gamma, B, Hq, d].
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_table: torch.Tensor, *, B: int, R: int, Hq: int, gamma: int,
                 P_max: int, k: int, n_sink: int, n_recent: int, max_tail: int,
                 scale: float, row0: int = 0, row1: Optional[int] = None,
                 stream: Optional[torch.cuda.Stream] = None):
        if not k_cache.is_cuda:
            raise ValueError("the caches must be CUDA tensors")
        _lib.load()
        dev = k_cache.device
        d = int(k_cache.shape[3])
        Hkv = int(k_cache.shape[1])
        self.B, self.R, self.Hq, self.gamma, self.d, self.Hkv = B, R, Hq, gamma, d, Hkv
        self.k_cache, self.v_cache, self.block_table = k_cache, v_cache, block_table
        self.P_max, self.k, self.n_sink, self.n_recent = P_max, k, n_sink, n_recent
        self.max_tail, self.scale = max_tail, scale
        self.row0, self.row1 = row0, (R - 1 if row1 is None else row1)
        self.stream = stream if stream is not None else torch.cuda.Stream(device=dev)

        def dbuf(shape, dtype):
            return torch.zeros(shape, dtype=dtype, device=dev)

        bf, i32 = torch.bfloat16, torch.int32
        # Inputs and results each live in one arena (pinned on the host, mirrored on the
        # device), so an iteration moves them with one copy each way.
        in_spec = (("q", (B, R, Hq, d), bf), ("q_draft", (gamma, B, Hq, d), bf),
                   ("prefix_len", (B,), i32), ("tail_start", (B,), i32),
                   ("seq_len", (gamma, B), i32))
        out_spec = (("out", (B, R, Hq, d), bf), ("idx", (B, k), i32), ("n_sel", (B,), i32),
                    ("draft_out", (gamma, B, Hq, d), bf))
        self._h_in, self._d_in = self._arena(in_spec, dev, "h_", "")
        self._h_res, self._d_res = self._arena(out_spec, dev, "h_", "")
        # device-only intermediates
        self.logits = dbuf((B, 2, Hq, P_max), torch.float32)
        self.partial = dbuf((B, Hkv, P_max), torch.float32)
        self.score = dbuf((B, P_max), torch.float32)
        self.score_hist = dbuf((B, _lib.HIST_BINS), torch.int32)
        geom = _lib.geom_for(B, Hq, k_cache, block_table)
        nb = _lib.vsd_verify_workspace_size(geom, R, P_max)
        self.verify_ws = dbuf((max(nb, 1),), torch.uint8)[:nb] if nb else None
        nb = _lib.vsd_sparse_workspace_size(geom, k, max_tail)
        self.sparse_ws = dbuf((max(nb, 1),), torch.uint8)[:nb] if nb else None
        self.graph = torch.cuda.CUDAGraph()
        # warm the library on this stream (per-device setup happens outside capture)
        with torch.cuda.stream(self.stream):
            self._record()
        self.stream.synchronize()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._record()
        self.stream.synchronize()

    def _arena(self, spec, dev, host_prefix, dev_prefix):
        """One pinned host buffer and one device buffer holding every tensor of `spec`
        (256-byte aligned views), exposed as attributes host_prefix+name / name."""
        offs, total = [], 0
        for name, shape, dtype in spec:
            n = 1
            for x in shape:
                n *= x
            nbytes = n * torch.tensor([], dtype=dtype).element_size()
            offs.append((name, shape, dtype, total, nbytes))
            total += (nbytes + 255) // 256 * 256
        h = torch.zeros(total, dtype=torch.uint8).pin_memory()
        dbuf = torch.zeros(total, dtype=torch.uint8, device=dev)
        for name, shape, dtype, off, nbytes in offs:
            setattr(self, host_prefix + name, h[off:off + nbytes].view(dtype).view(shape))
            setattr(self, dev_prefix + name, dbuf[off:off + nbytes].view(dtype).view(shape))
        return h, dbuf

    def _record(self):
        s = self.stream
        _lib.vsd_copy(self._d_in, self._h_in, stream=s)
        _lib.vsd_verify_attn_collect_scored(self.q, self.k_cache, self.v_cache, self.block_table,
                                            self.prefix_len, P_max=self.P_max, scale=self.scale,
                                            row0=self.row0, row1=self.row1, logits=self.logits,
                                            partial=self.partial, score=self.score,
                                            score_hist=self.score_hist, n_sink=self.n_sink,
                                            n_recent=self.n_recent, out=self.out,
                                            workspace=self.verify_ws, stream=s)
        _lib.vsd_select_topk_scored(self.score, self.score_hist, self.prefix_len, k=self.k,
                                    n_sink=self.n_sink, n_recent=self.n_recent, idx=self.idx,
                                    n_sel=self.n_sel, stream=s)
        for i in range(self.gamma):
            _lib.vsd_sparse_decode_attn(self.q_draft[i], self.k_cache, self.v_cache,
                                        self.block_table, self.idx, self.n_sel, self.tail_start,
                                        self.seq_len[i], scale=self.scale,
                                        max_tail=self.max_tail, out=self.draft_out[i],
                                        workspace=self.sparse_ws, stream=s)
        _lib.vsd_copy(self._h_res, self._d_res, stream=s)

    @property
    def h2d_bytes(self) -> int:
        return self._h_in.numel()

    @property
    def d2h_bytes(self) -> int:
        return self._h_res.numel()

    def run(self, sync: bool = False) -> None:
        """Replay the iteration on the graph's stream (after the current stream's work)."""
        self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        if sync:
            self.stream.synchronize()

    def reset_workspaces(self) -> None:
        """Zero the draft step's workspace (its per-pair counters): needed after a call
        whose status word showed VSD_DEV_TIMEOUT, which may leave counters behind."""
        if self.sparse_ws is not None:
            with torch.cuda.stream(self.stream):
                self.sparse_ws.zero_()

    def synchronize(self) -> None:
        self.stream.synchronize()
