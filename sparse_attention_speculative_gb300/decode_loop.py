"""Vegas decode iterations over a multi-layer attention stack, one CUDA graph each.

One iteration of verification-guided sparse self-speculative decoding (Vegas summary,
sec. 2 core mechanism: verification phase -> KV selection -> drafting phase) over L
layers, every kernel libvsd's:

  for every layer l:   verification with Collect-2-Query and the fused aggregation
                       -> this layer's score rows and histograms; the same call
                       stores the verify block's keys/values into layer l's cache at
                       [P_b, P_b + R) before it reads them
                                                     (vsd_verify_attn_collect_scored)
  once:                the protected top-k of every (layer, sequence) row
                                                             (vsd_select_topk_scored)
                       the accepted counts move every prefix     (vsd_advance_lengths)
  for draft step i:    for every layer l: the sparse draft attention over the selection
                       plus the dense tail, which also stores the step's input token
                       keys/values at seq_len_i - 1; the first step records the
                       selection's cache rows for the later ones
                                                        (vsd_sparse_decode_attn_step)

The prefix lengths, the draft tails and the per-row prefixes of the selection live on
the device and advance inside the graph, so consecutive replays are consecutive decode
iterations; `reset()` puts the prefixes back.  The iteration's inputs (queries, the new
keys and values, the accepted counts) come from one input arena and its results (every
verification and draft output, the selections) go to one result arena.  `run()` replays
the variant that also copies the inputs in from a pinned host arena and the results
back to a pinned host arena (both copies are `vsd_copy` kernels that address the pinned
memory directly); `replay_device()` replays the one without host copies.  This module
owns buffers and graphs only; all arithmetic runs in libvsd's kernels.
"""
from __future__ import annotations

from typing import Callable, Dict, Optional, Sequence

import torch

from . import _lib


class DecodeLoop:
    """Shapes (L layers, B sequences, R = gamma + 1 verify rows):
      inputs   q bf16 [L, B, R, Hq, d]; q_draft bf16 [L, gamma, B, Hq, d];
               k_verify, v_verify bf16 [L, B, R, Hkv, d]; k_draft, v_draft bf16
               [L, gamma, B, Hkv, d]; accepted int32 [B] (drafts accepted by this
               iteration's verification, 0 .. gamma)
      results  out bf16 [L, B, R, Hq, d]; draft_out bf16 [gamma, L, B, Hq, d];
               idx int32 [L * B, k]; n_sel int32 [L * B]; and, after the iteration,
               the loop state: prefix_len, tail_start int32 [B], seq_len int32
               [gamma, B] (host views h_prefix_len_out, h_tail_start_out, h_seq_len_out)
    Host mirrors of both arenas carry the prefix ``h_`` (pinned).
    """

    def __init__(self, k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
                 block_tables: Sequence[torch.Tensor], prefix_len0, *, Hq: int, gamma: int,
                 k: int, n_sink: int, n_recent: int, P_max: int, scale: float,
                 collect_logits: bool = True, stream: Optional[torch.cuda.Stream] = None):
        _lib.load()
        L = len(k_caches)
        if L == 0 or len(v_caches) != L or len(block_tables) != L:
            raise ValueError("one K cache, V cache and block table per layer")
        kc0 = k_caches[0]
        if not kc0.is_cuda:
            raise ValueError("the caches must be CUDA tensors")
        dev = kc0.device
        self.L, self.gamma, self.R, self.Hq = L, gamma, gamma + 1, Hq
        self.Hkv, self.d = int(kc0.shape[1]), int(kc0.shape[3])
        pl0 = torch.as_tensor(prefix_len0, dtype=torch.int32).flatten()
        self.B = B = int(pl0.numel())
        self.k, self.n_sink, self.n_recent = k, n_sink, n_recent
        self.P_max, self.scale = P_max, scale
        self.max_tail = 2 * gamma + 1
        for kc, vc, bt in zip(k_caches, v_caches, block_tables):
            if tuple(kc.shape) != tuple(kc0.shape) or tuple(vc.shape) != tuple(kc0.shape):
                raise ValueError("every layer's caches must have one shape")
            if int(bt.shape[0]) != B:
                raise ValueError("block tables need one row per sequence")
            # the longest prefix, its verify block and the last draft token must fit
            if int(bt.shape[1]) * 16 < P_max + self.R + gamma:
                raise ValueError("block table too short for prefixes up to P_max")
        if int(pl0.max()) > P_max:
            raise ValueError("an initial prefix exceeds P_max")
        self.k_caches, self.v_caches = list(k_caches), list(v_caches)
        self.block_tables = list(block_tables)
        self.stream = stream if stream is not None else torch.cuda.Stream(device=dev)
        R, Hkv, d = self.R, self.Hkv, self.d
        bf, i32 = torch.bfloat16, torch.int32
        in_spec = (("q", (L, B, R, Hq, d), bf), ("q_draft", (L, gamma, B, Hq, d), bf),
                   ("k_verify", (L, B, R, Hkv, d), bf), ("v_verify", (L, B, R, Hkv, d), bf),
                   ("k_draft", (L, gamma, B, Hkv, d), bf), ("v_draft", (L, gamma, B, Hkv, d), bf),
                   ("accepted", (B,), i32))
        # row stride of the logits, partial-score and score buffers: a multiple of 32
        # positions, so every row starts on a 128-byte boundary (the verification writes
        # 32 consecutive positions per warp store; rows that start inside a 32-byte
        # sector leave partly written sectors that cost DRAM read-modify-writes)
        self.row_stride = (P_max + 31) // 32 * 32
        self._h_in, self._d_in = _arena(self, in_spec, dev)

        def dbuf(shape, dtype):
            return torch.zeros(shape, dtype=dtype, device=dev)

        # device state of the decode loop, and its initial value (copied in by reset())
        st_spec = (("prefix_len", (B,), i32), ("rows_prefix", (L * B,), i32),
                   ("tail_start", (B,), i32), ("seq_len", (gamma, B), i32))
        self._h_state0, self._d_state = _arena(self, st_spec, dev, host_prefix="_init_")
        self._state_views = {name: (getattr(self, name).data_ptr() - self._d_state.data_ptr(),
                                    getattr(self, name)) for name, _, _ in st_spec}
        self._init_prefix_len.copy_(pl0)
        self._init_rows_prefix.copy_(pl0.repeat(L))
        self._init_tail_start.copy_(pl0)
        self._d_state0 = self._h_state0.to(dev)
        res_spec = (("out", (L, B, R, Hq, d), bf), ("draft_out", (gamma, L, B, Hq, d), bf),
                    ("idx", (L * B, k), i32), ("n_sel", (L * B,), i32),
                    ("state_out", (self._h_state0.numel(),), torch.uint8))
        self._h_res, self._d_res = _arena(self, res_spec, dev)
        # host views of the loop state after the iteration (the state arena's layout)
        base = self.h_state_out
        for name, (t0, n) in self._state_views.items():
            setattr(self, "h_%s_out" % name, base[t0:t0 + n.numel() * 4].view(torch.int32)
                    .view(n.shape))
        # device-only intermediates, shared by the layers
        rs = self.row_stride
        self.logits = dbuf((B, 2, Hq, rs), torch.float32) if collect_logits else None
        self.partial = dbuf((B, Hkv, rs), torch.float32)
        self.score = dbuf((L * B, rs), torch.float32)
        self.score_hist = dbuf((L * B, _lib.HIST_BINS), torch.int32)
        self.sel_rows = dbuf((L * B, k), torch.int32)  # the selection's cache rows
        geom = _lib.geom_for(B, Hq, kc0, self.block_tables[0])
        nb = _lib.vsd_verify_workspace_size(geom, R, self.row_stride)
        self.verify_ws = _aligned(dbuf((nb + 256,), torch.uint8), nb) if nb else None
        nb = _lib.vsd_sparse_workspace_size(geom, k, self.max_tail)
        self.sparse_ws = _aligned(dbuf((nb + 256,), torch.uint8), nb) if nb else None
        # warm the library on this stream (per-device setup happens outside capture),
        # then capture both variants and put the state back
        self.reset()
        with torch.cuda.stream(self.stream):
            self._record(host_io=True)
        self.stream.synchronize()
        self.graph_io = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_io, stream=self.stream):
            self._record(host_io=True)
        self.graph_dev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_dev, stream=self.stream):
            self._record(host_io=False)
        self.stream.synchronize()
        self.reset()
        self.stream.synchronize()

    # ------------------------------------------------------------------ recording
    def _record(self, host_io: bool, marks: Optional[Dict[str, Callable]] = None,
                accepted: Optional[torch.Tensor] = None):
        """Enqueue one iteration on self.stream.  `marks` (optional) maps phase names
        ("verified", "selected", "drafted") to callables run after that phase;
        `accepted` (optional, int32 [B] on the device) replaces the input arena's
        accepted counts."""
        s = self.stream
        L, B, gamma = self.L, self.B, self.gamma
        if host_io:
            _lib.vsd_copy(self._d_in, self._h_in, stream=s)
        for l in range(L):
            kc, vc, bt = self.k_caches[l], self.v_caches[l], self.block_tables[l]
            rows = slice(l * B, (l + 1) * B)
            # the call stores the verify block's rows itself (at the prefix length and
            # beyond); its predecessor (the previous layer's verification, the previous
            # iteration's last draft step or the input copy, which writes neither the
            # lengths nor the cache below them) lets the prefix's first tiles be
            # fetched before the wait for it
            _lib.vsd_verify_attn_collect_scored(
                self.q[l], kc, vc, bt, self.prefix_len, P_max=self.row_stride, scale=self.scale,
                row0=0, row1=self.R - 1, logits=self.logits, partial=self.partial,
                score=self.score[rows], score_hist=self.score_hist[rows], n_sink=self.n_sink,
                n_recent=self.n_recent, flags=_lib.VERIFY_EARLY_PREFETCH,
                k_new=self.k_verify[l], v_new=self.v_verify[l], out=self.out[l],
                workspace=self.verify_ws, stream=s)
        if marks and "verified" in marks:
            marks["verified"]()
        _lib.vsd_select_topk_scored(self.score, self.score_hist, self.rows_prefix, k=self.k,
                                    n_sink=self.n_sink, n_recent=self.n_recent, idx=self.idx,
                                    n_sel=self.n_sel, stream=s)
        _lib.vsd_advance_lengths(self.accepted if accepted is None else accepted,
                                 self.prefix_len, self.tail_start, self.seq_len,
                                 max_prefix=self.P_max, prefix_copies=self.rows_prefix,
                                 stream=s)
        if marks and "selected" in marks:
            marks["selected"]()
        for i in range(gamma):
            for l in range(L):
                kc, vc, bt = self.k_caches[l], self.v_caches[l], self.block_tables[l]
                rows = slice(l * B, (l + 1) * B)
                # the step's input token joins the cache inside the draft call; the first
                # step records the selection's cache rows, the later steps reuse them.  A
                # call whose predecessor is the draft call of another layer (which writes
                # none of the inputs this one gathers from) gathers before waiting for it;
                # the first call after the advance (which writes the tails), and with one
                # layer every call (its predecessor wrote this layer's previous token and
                # recorded rows), wait first
                flags = _lib.STEP_RECORD_ROWS if i == 0 else _lib.STEP_REUSE_ROWS
                if l > 0 or (i > 0 and L > 1):
                    flags |= _lib.STEP_EARLY_GATHER
                _lib.vsd_sparse_decode_attn_step(
                    self.q_draft[l, i], kc, vc, bt, self.idx[rows], self.n_sel[rows],
                    self.tail_start, self.seq_len[i], scale=self.scale, max_tail=self.max_tail,
                    k_new=self.k_draft[l, i], v_new=self.v_draft[l, i],
                    sel_rows=self.sel_rows[rows], flags=flags, out=self.draft_out[i, l],
                    workspace=self.sparse_ws, stream=s)
        if marks and "drafted" in marks:
            marks["drafted"]()
        _lib.vsd_copy(self.state_out, self._d_state, stream=s)
        if host_io:
            _lib.vsd_copy(self._h_res, self._d_res, stream=s)

    # ------------------------------------------------------------------ use
    @property
    def launches_per_iteration(self) -> int:
        """libvsd kernel launches of one device iteration (no host copies): per layer the
        verification (which stores the verify block's K/V itself) and its merge kernel;
        the selection and the advance; per draft step and layer the draft kernel (it
        stores its input token's K/V itself); the state copy."""
        return self.L * 2 + 2 + self.gamma * self.L + 1

    @property
    def h2d_bytes(self) -> int:
        return self._h_in.numel()

    @property
    def d2h_bytes(self) -> int:
        return self._h_res.numel()

    def reset(self) -> None:
        """Put the prefixes and draft tails back to their initial values (on the
        loop's stream; no host synchronisation)."""
        _lib.vsd_copy(self._d_state, self._d_state0, stream=self.stream)

    def run(self, sync: bool = False) -> None:
        """One iteration with its host copies: inputs from the pinned host arena,
        results to the pinned result arena (valid after synchronize())."""
        self.stream.wait_stream(torch.cuda.current_stream(self.stream.device))
        with torch.cuda.stream(self.stream):
            self.graph_io.replay()
        if sync:
            self.stream.synchronize()

    def replay_device(self) -> None:
        """One iteration on the device arenas only (no host copies)."""
        with torch.cuda.stream(self.stream):
            self.graph_dev.replay()

    def record_marked(self, marks: Dict[str, Callable],
                      first: Optional[Callable] = None) -> torch.cuda.CUDAGraph:
        """A graph of one device iteration with `marks` (e.g. external event records)
        at its phase boundaries and `first` before it, for a per-phase breakdown."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            if first is not None:
                first()
            self._record(host_io=False, marks=marks)
        self.stream.synchronize()
        return g

    def record_run(self, accepted_rows: torch.Tensor) -> torch.cuda.CUDAGraph:
        """A graph of a whole decode run on the device arenas: reset(), then one
        iteration per row of `accepted_rows` (int32 [n, B] on the device: the drafts
        each iteration's verification accepts)."""
        if accepted_rows.dtype != torch.int32 or accepted_rows.dim() != 2 or \
                int(accepted_rows.shape[1]) != self.B or not accepted_rows.is_cuda:
            raise ValueError("accepted_rows must be an int32 CUDA tensor [n, B]")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.reset()
            for i in range(int(accepted_rows.shape[0])):
                self._record(host_io=False, accepted=accepted_rows[i])
        self.stream.synchronize()
        return g

    def reset_workspaces(self) -> None:
        """Zero the draft step's workspace (its per-pair counters): needed after a call
        whose status word showed VSD_DEV_TIMEOUT, which may leave counters behind."""
        if self.sparse_ws is not None:
            with torch.cuda.stream(self.stream):
                self.sparse_ws.zero_()

    def synchronize(self) -> None:
        self.stream.synchronize()


def _aligned(buf: torch.Tensor, nbytes: int) -> torch.Tensor:
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def _arena(obj, spec, dev, host_prefix: str = "h_"):
    """One pinned host buffer and one device buffer holding every tensor of `spec`
    (256-byte aligned views), exposed on `obj` as host_prefix + name and name."""
    offs, total = [], 0
    for name, shape, dtype in spec:
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        offs.append((name, shape, dtype, total, nbytes))
        total += (nbytes + 255) // 256 * 256
    h = torch.zeros(total, dtype=torch.uint8).pin_memory()
    d = torch.zeros(total + 256, dtype=torch.uint8, device=dev)
    d = _aligned(d, total)
    for name, shape, dtype, off, nbytes in offs:
        setattr(obj, host_prefix + name, h[off:off + nbytes].view(dtype).view(shape))
        setattr(obj, name, d[off:off + nbytes].view(dtype).view(shape))
    return h, d
