"""Benchmark of one Vegas iteration on GB300: verify + Collect-2-Query, top-k
selection, and gamma sparse draft steps, through the libvsd C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line.  `value` is the algorithmic bytes of the whole iteration
(KV read by verify, logits and partial scores written, partial scores read by the
select, gathered KV of every draft step, queries and outputs) divided by the device
time of the iteration, summed over ranks.  L2 is flushed before every timed
iteration (512 MB write then 512 MB read, untimed); each iteration is enqueued
behind a GPU sleep so host launch latency never shows in the device timestamps.
`--impl reference` times the fp64 CPU oracle on the same workload instead (a
deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20  # > 129 MB of L2
B2B_CALLS = 20
METRIC = ("KV-read GB/s of one Vegas iteration (verify+collect2, top-k select, "
          "gamma sparse draft steps)")


def flush_l2(buf_w, buf_r):
    """Evict L2 before a timed iteration: write a buffer larger than L2, then read
    another one, so the lines left behind are clean and their eviction costs the
    timed kernels no DRAM write-back."""
    buf_w.zero_()
    buf_r.sum(dtype=torch.int64)


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank-space runs (string literals are
    kept as they are), so that edits to comments leave the digest alone."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def verify_sources_digest():
    """Digest of the code (comments left out) the verification kernels compile from: their
    own files, the PTX and common helpers, the public header and the verification part of
    the internal launch interface."""
    csrc = os.path.join(ROOT, "sparse_attention_speculative_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("verify_attn.cuh", "verify_attn.cu", "verify_attn_d128.cu", "verify_attn_d64.cu",
                 "ptx.cuh", "common.cuh"):
        h.update(_code_only(open(os.path.join(csrc, name)).read()).encode())
    h.update(_code_only(open(os.path.join(ROOT, "include", "vsd.h")).read()).encode())
    launch = open(os.path.join(csrc, "launch.h")).read()
    i = launch.index("// " + "-" * 64 + " verify")
    j = launch.index("// " + "-" * 64, i + 10)
    h.update(_code_only(launch[i:j]).encode())
    return h.hexdigest()[:16]


def profile_traffic(workload: str, bytes_per_call: float):
    """DRAM bytes per launch of the verification call, from the committed ncu record
    (profiles/verify_traffic.json: read + write bytes of the main and merge kernels of one
    call on a captured workload, with that call's algorithmic bytes), scaled to a call of
    `bytes_per_call` algorithmic bytes; None when the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "verify_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if rec.get("sources_digest") != verify_sources_digest():
        return None
    return rec["dram_bytes_per_call"] * bytes_per_call / rec["algorithmic_bytes_per_call"]


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ workload bytes

def sparse_verify_bytes(w, n_sel):
    """Algorithmic bytes of one sparse verification: K and V of the selected positions
    and the verify block, q in and out."""
    kv_row = w.d * 2
    return sum(2 * w.Hkv * (n + w.R) * kv_row + 2 * w.R * w.Hq * w.d * 2 for n in n_sel)


def iteration_bytes(w, prefix, n_sel, tail_lens):
    """Algorithmic bytes of one iteration (per kernel), from the shapes."""
    d, Hq, Hkv, R = w.d, w.Hq, w.Hkv, w.R
    kv_row = d * 2  # bytes of one (token, head) K or V row
    verify = 0
    for P in prefix:
        verify += 2 * Hkv * (P + R) * kv_row          # K and V of every attended key
        verify += 2 * R * Hq * d * 2                  # q in, out
        verify += 2 * Hq * P * 4 + Hkv * P * 4        # logits and partial scores written
    select = sum(Hkv * P * 4 for P in prefix) + sum(4 * min(w.k, P) for P in prefix)
    sparse = []
    for tl in tail_lens:
        s = 0
        for b, P in enumerate(prefix):
            s += 2 * Hkv * (n_sel[b] + tl[b]) * kv_row + 2 * Hq * d * 2
        sparse.append(s)
    return verify, select, sparse


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, world, rank, local):
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build as pkg_build
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import ALL

    if rank == 0 or not pkg_build.up_to_date():
        pkg_build.build()
    if world > 1:
        torch.distributed.barrier()
    vsd.load()
    w = ALL[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    batch = make_batch(w, dev)
    B, R, Hq, d, gamma = w.B, w.R, w.Hq, w.d, w.gamma
    prefix = list(w.prefix())
    P_max = w.P_max
    geom = vsd.geom_for(B, Hq, batch.k_cache, batch.block_table)
    ws_bytes = vsd.vsd_verify_workspace_size(geom, R, P_max)
    workspace = torch.zeros(max(ws_bytes, 1) + 256, dtype=torch.uint8, device=dev)
    off = (-workspace.data_ptr()) % 256
    workspace = workspace[off:off + ws_bytes] if ws_bytes else None
    out = torch.empty_like(batch.q)
    logits = torch.empty((B, 2, Hq, P_max), dtype=torch.float32, device=dev)
    partial = torch.empty((B, w.Hkv, P_max), dtype=torch.float32, device=dev)
    score = torch.empty((B, P_max), dtype=torch.float32, device=dev)
    score_hist = torch.empty((B, vsd.HIST_BINS), dtype=torch.int32, device=dev)
    idx = torch.empty((B, w.k), dtype=torch.int32, device=dev)
    n_sel = torch.empty((B,), dtype=torch.int32, device=dev)
    d_out = torch.empty((gamma, B, Hq, d), dtype=torch.bfloat16, device=dev)
    tail_start = batch.prefix_len.clone()
    seq_len = torch.empty((gamma, B), dtype=torch.int32, device=dev)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(w.seed + 77)
    max_tail = 2 * gamma + 1

    def draw_seq_len():
        a = rng.integers(0, gamma + 1, size=B)  # accepted drafts this iteration
        return np.array([[prefix[b] + a[b] + 2 + i for b in range(B)] for i in range(gamma)],
                        dtype=np.int32)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 + gamma)]

    def step(events=True):
        # verification with Collect-2-Query and the fused aggregation (the score summed
        # over the KV groups and its first histogram level), then the selection from them
        vsd.vsd_verify_attn_collect_scored(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, P_max=P_max,
                                           scale=w.scale, row0=0, row1=R - 1, logits=logits,
                                           partial=partial, score=score, score_hist=score_hist,
                                           n_sink=w.n_sink, n_recent=w.n_recent, out=out,
                                           workspace=workspace)
        if events:
            ev[1].record(stream)
        vsd.vsd_select_topk_scored(score, score_hist, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                   n_recent=w.n_recent, idx=idx, n_sel=n_sel)
        if events:
            ev[2].record(stream)
        for i in range(gamma):
            vsd.vsd_sparse_decode_attn(batch.q_draft[i], batch.k_cache, batch.v_cache,
                                       batch.block_table, idx, n_sel, tail_start, seq_len[i],
                                       scale=w.scale, max_tail=max_tail, out=d_out[i])
            if events:
                ev[3 + i].record(stream)

    # this library's kernel launches per step: verification and its merge + aggregation
    # kernel, selection, and one kernel per draft step (the draft step merges its splits
    # inside the kernel)
    launches_per_verify = 2
    launches_per_step = launches_per_verify + 1 + gamma
    enqueue_s = []
    sleep_cycles = 8_000_000  # ~4 ms: the whole step is enqueued before the GPU gets to it

    def timed_step(sl):
        seq_len.copy_(torch.from_numpy(sl))
        flush_l2(flush_w, flush_r)
        torch.cuda.synchronize()
        torch.cuda._sleep(sleep_cycles)  # keep the GPU busy while the host enqueues the step
        t_host = time.perf_counter()
        ev[0].record(stream)
        step()
        enqueue_s.append(time.perf_counter() - t_host)

    for _ in range(args.warmup):
        timed_step(draw_seq_len())
    torch.cuda.synchronize()
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x during warm-up" % status)

    # the whole iteration as one CUDA graph: the kernels are chained by programmatic
    # dependent launch, so each one's launch overlaps the tail of its predecessor
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(events=False)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def graph_step(sl):
        seq_len.copy_(torch.from_numpy(sl))
        flush_l2(flush_w, flush_r)
        torch.cuda.synchronize()
        torch.cuda._sleep(sleep_cycles)
        g0.record(stream)
        graph.replay()
        g1.record(stream)

    for _ in range(args.warmup):
        graph_step(draw_seq_len())
    torch.cuda.synchronize()

    per = {"verify": [], "select": [], "sparse": [], "step": [], "graph": []}
    tails_seen = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for _ in range(args.steps):
            sl = draw_seq_len()
            tails_seen.append([[int(sl[i, b] - prefix[b]) for b in range(B)]
                               for i in range(gamma)])
            graph_step(sl)
            torch.cuda.synchronize()
            per["graph"].append(g0.elapsed_time(g1) * 1e-3)
        # per-kernel breakdown: the same iteration launched eagerly, events between kernels
        for _ in range(args.steps):
            timed_step(draw_seq_len())
            torch.cuda.synchronize()
            per["verify"].append(ev[0].elapsed_time(ev[1]) * 1e-3)
            per["select"].append(ev[1].elapsed_time(ev[2]) * 1e-3)
            per["sparse"].append([ev[2 + i].elapsed_time(ev[3 + i]) * 1e-3 for i in range(gamma)])
            per["step"].append(ev[0].elapsed_time(ev[2 + gamma]) * 1e-3)
        # the verification call alone, back to back: K and V (>= 134 MB at these sizes)
        # exceed L2, so every call streams them from HBM; per-call time = span / calls
        per["verify_b2b"] = []
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_verify_attn_collect(batch.q, batch.k_cache, batch.v_cache,
                                            batch.block_table, batch.prefix_len, P_max=P_max,
                                            scale=w.scale, row0=0, row1=R - 1, logits=logits,
                                            partial=partial, out=out, workspace=workspace)
            v1.record(stream)
            torch.cuda.synchronize()
            per["verify_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        # the same with the fused aggregation (what the iteration runs)
        per["verify_scored_b2b"] = []
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_verify_attn_collect_scored(
                    batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
                    P_max=P_max, scale=w.scale, row0=0, row1=R - 1, logits=logits,
                    partial=partial, score=score, score_hist=score_hist, n_sink=w.n_sink,
                    n_recent=w.n_recent, flags=vsd.VERIFY_EARLY_PREFETCH, out=out,
                    workspace=workspace)
            v1.record(stream)
            torch.cuda.synchronize()
            per["verify_scored_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        # sparse verification (Dustin) over this iteration's selection, back to back
        per["sparse_verify_b2b"] = []
        sv_out = torch.empty_like(batch.q)
        sv_geom = vsd.geom_for(B, Hq, batch.k_cache, batch.block_table)
        sv_ws = torch.zeros(vsd.vsd_sparse_verify_workspace_size(sv_geom, R, w.k) + 256,
                            dtype=torch.uint8, device=dev)
        sv_ws = sv_ws[(-sv_ws.data_ptr()) % 256:]
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, idx, n_sel,
                                           scale=w.scale, flags=vsd.SPARSE_VERIFY_EARLY_GATHER,
                                           out=sv_out, workspace=sv_ws)
            v1.record(stream)
            torch.cuda.synchronize()
            per["sparse_verify_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        # Dustin's hybrid budget (a synthetic draft-lookahead signal, m = k / 4) and the
        # collect restricted to a quarter of the query heads (semantic retrieval heads)
        per["hybrid_b2b"], per["srh_b2b"], per["select_b2b"] = [], [], []
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                    n_recent=w.n_recent, idx=idx, n_sel=n_sel)
            v1.record(stream)
            torch.cuda.synchronize()
            per["select_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        per["select_scored_b2b"] = []
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_select_topk_scored(score, score_hist, batch.prefix_len, k=w.k,
                                           n_sink=w.n_sink, n_recent=w.n_recent, idx=idx,
                                           n_sel=n_sel)
            v1.record(stream)
            torch.cuda.synchronize()
            per["select_scored_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        g_d = torch.Generator(device=dev)
        g_d.manual_seed(w.seed + 5)
        partial_draft = torch.randn((B, 2, P_max), generator=g_d, device=dev)
        idx_h = torch.empty_like(idx)
        nsel_h = torch.empty_like(n_sel)
        head_mask = torch.tensor([1 if h % 4 == 0 else 0 for h in range(Hq)], dtype=torch.uint8,
                                 device=dev)
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_select_topk_hybrid(partial, partial_draft, batch.prefix_len, k=w.k,
                                           m=w.k // 4, n_sink=w.n_sink, n_recent=w.n_recent,
                                           idx=idx_h, n_sel=nsel_h)
            v1.record(stream)
            torch.cuda.synchronize()
            per["hybrid_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_verify_attn_collect_srh(batch.q, batch.k_cache, batch.v_cache,
                                                batch.block_table, batch.prefix_len, head_mask,
                                                P_max=P_max, scale=w.scale, logits=logits,
                                                partial=partial, out=out, workspace=workspace)
            v1.record(stream)
            torch.cuda.synchronize()
            per["srh_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        # the contrasting per-query block top-k (page mean keys, then per-(t, h) page
        # scores and top kb = k / 16 pages: the same token budget per query)
        per["page_means_b2b"], per["block_topk_b2b"] = [], []
        nblk_max = vsd.page_blocks(P_max)
        kb = max(1, w.k // 16)
        means = torch.zeros((B, w.Hkv, nblk_max, d), dtype=torch.float32, device=dev)
        bscores = torch.zeros((B, R, Hq, nblk_max), dtype=torch.float32, device=dev)
        bblocks = torch.empty((B, R, Hq, kb), dtype=torch.int32, device=dev)
        for _ in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_page_key_means(batch.k_cache, batch.block_table, batch.prefix_len, B=B,
                                       page_blocks_max=nblk_max, page_means=means)
            v1.record(stream)
            torch.cuda.synchronize()
            per["page_means_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
            torch.cuda._sleep(sleep_cycles)
            v0.record(stream)
            for _ in range(B2B_CALLS):
                vsd.vsd_block_topk(batch.q, means, batch.prefix_len, kb=kb, scale=w.scale,
                                   scores=bscores, blocks=bblocks)
            v1.record(stream)
            torch.cuda.synchronize()
            per["block_topk_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
        # the same, collecting every verify row (the selection equation as printed):
        # what Collect-2-Query saves
        per["verify_all_b2b"] = []
        if R * (Hq // w.Hkv) <= 48:
            logits_all = torch.empty((B, R, Hq, P_max), dtype=torch.float32, device=dev)
            for _ in range(3):
                torch.cuda.synchronize()
                torch.cuda._sleep(sleep_cycles)
                v0.record(stream)
                for _ in range(B2B_CALLS):
                    vsd.vsd_verify_attn_collect_all(batch.q, batch.k_cache, batch.v_cache,
                                                    batch.block_table, batch.prefix_len,
                                                    P_max=P_max, scale=w.scale, logits=logits_all,
                                                    partial=partial, out=out, workspace=workspace)
                v1.record(stream)
                torch.cuda.synchronize()
                per["verify_all_b2b"].append(v0.elapsed_time(v1) * 1e-3 / B2B_CALLS)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x in the timed region" % status)
    n_sel_host = n_sel.cpu().tolist()

    # algorithmic bytes (the draft tails vary with the drawn accept counts)
    mean_tails = [[statistics.mean(t[i][b] for t in tails_seen) for b in range(B)]
                  for i in range(gamma)]
    vb, sb, spb = iteration_bytes(w, prefix, n_sel_host, mean_tails)
    total_bytes = vb + sb + sum(spb)
    t_step = sum(per["graph"])
    t_tensor = torch.tensor([t_step], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_tensor, op=torch.distributed.ReduceOp.MAX)
    t_max = float(t_tensor.item())
    value = world * total_bytes * args.steps / t_max / 1e9
    peak, peak_kind = measured_peaks()
    # per-kernel figures: medians over the timed iterations (L2 flushed before each)
    t_verify = statistics.median(per["verify"])
    t_select = statistics.median(per["select"])
    t_sparse = statistics.median([x for s in per["sparse"] for x in s])
    nominal = NOMINAL_HBM_GBS
    kernels = {
        "verify_collect": {"us": t_verify * 1e6, "bytes": vb, "GB_s": vb / t_verify / 1e9,
                           "frac_of_%s_hbm" % peak_kind: vb / t_verify / 1e9 / peak,
                           "frac_of_nominal_8tbs": vb / t_verify / 1e9 / nominal},
        "select_topk": {"us": t_select * 1e6, "bytes": sb, "GB_s": sb / t_select / 1e9,
                        "frac_of_%s_hbm" % peak_kind: sb / t_select / 1e9 / peak,
                        "frac_of_nominal_8tbs": sb / t_select / 1e9 / nominal},
        "sparse_draft_step": {"us": t_sparse * 1e6, "bytes": statistics.mean(spb),
                              "GB_s": statistics.mean(spb) / t_sparse / 1e9,
                              "frac_of_%s_hbm" % peak_kind:
                                  statistics.mean(spb) / t_sparse / 1e9 / peak,
                              "frac_of_nominal_8tbs":
                                  statistics.mean(spb) / t_sparse / 1e9 / nominal},
    }
    t_verify_b2b = statistics.median(per["verify_b2b"])
    achieved = vb / t_verify_b2b / 1e9
    clk = clocks.summary()
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_max / args.steps * 1e3,
        "us_per_iter": t_max / args.steps * 1e6,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": B, "P": w.P, "Hq": Hq, "Hkv": w.Hkv, "d": d,
                   "gamma": gamma, "k": w.k, "n_sink": w.n_sink, "n_recent": w.n_recent,
                   "page": w.page,
                   "l2": "flushed before every timed iteration (512 MB write, then 512 MB "
                         "read so no dirty lines remain)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "timing": "value: one CUDA-graph replay of the iteration per step (device events "
                  "around the replay); kernels: medians over the timed iterations of the "
                  "same iteration launched eagerly with events between kernels, so each "
                  "figure includes its launch gap",
        "us_per_iter_eager": statistics.mean(per["step"]) * 1e6,
        "kernels": kernels,
        "select_over_verify": t_select / t_verify,
        "fused_aggregation": {
            "verify_scored_us": statistics.median(per["verify_scored_b2b"]) * 1e6,
            "select_scored_us": statistics.median(per["select_scored_b2b"]) * 1e6,
            "verify_plain_us": t_verify_b2b * 1e6,
            "select_plain_us": statistics.median(per["select_b2b"]) * 1e6,
            "select_over_verify": statistics.median(per["select_scored_b2b"]) /
                                  statistics.median(per["verify_scored_b2b"]),
            "note": "back-to-back calls; scored = the verification call also sums the "
                    "per-group partials into the score and counts its first histogram "
                    "level, and the selection starts from them (what the iteration runs)"},
        "verify_back_to_back_us": t_verify_b2b * 1e6,
        "sparse_verify": {
            "us": statistics.median(per["sparse_verify_b2b"]) * 1e6,
            "full_verify_us": t_verify_b2b * 1e6,
            "attended_keys_per_head": [int(n) + R for n in n_sel_host],
            "note": "verify rows attend the selection plus the verify block (a compressed "
                    "cache gathered into the workspace, then the verification kernel); "
                    "back-to-back calls"},
        "hybrid_select_us": statistics.median(per["hybrid_b2b"]) * 1e6,
        "select_back_to_back_us": statistics.median(per["select_b2b"]) * 1e6,
        "srh_verify_us": statistics.median(per["srh_b2b"]) * 1e6,
        "block_topk": {
            "kb_pages": kb,
            "page_means_us": statistics.median(per["page_means_b2b"]) * 1e6,
            "page_means_gbs": sum(P * w.Hkv * d * 2 + ((P + 15) // 16) * w.Hkv * d * 4
                                  for P in prefix) / statistics.median(per["page_means_b2b"])
                              * 1e-9,
            "scores_and_topk_us": statistics.median(per["block_topk_b2b"]) * 1e6,
            "note": "per-query block-sparse top-k: mean key of every 16-token page (a full "
                    "recompute; a decode loop refreshes only the last page), then every "
                    "(verify row, head) scores the pages and keeps its kb best; back-to-back "
                    "calls"},
        "collect2_vs_all_rows": None if not per["verify_all_b2b"] else {
            "collect2_us": t_verify_b2b * 1e6,
            "all_rows_us": statistics.median(per["verify_all_b2b"]) * 1e6,
            "logits_bytes_collect2": sum(2 * Hq * P * 4 for P in prefix),
            "logits_bytes_all_rows": sum(R * Hq * P * 4 for P in prefix),
            "note": "back-to-back calls; all rows = every verify row's logits written and "
                    "summed (the selection equation as printed)"},
        "roofline": {"bound": "hbm", "kernel": "vsd_verify_attn_collect",
                     "timing": "%d verification calls back to back between two events on "
                               "the launching stream (K/V larger than L2), per-call mean; "
                               "bytes = algorithmic bytes of one call" % B2B_CALLS,
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profile_traffic(w.name, vb)},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_all_timed_loops": (2 * launches_per_step * args.steps +
                                         (6 if per["verify_all_b2b"] else 3) * B2B_CALLS *
                                         launches_per_verify + 3 * B2B_CALLS * 3 +
                                         3 * B2B_CALLS * (3 + launches_per_verify)),
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
        # the device timestamps only measure kernels if the host finished enqueueing a
        # step while the GPU was still asleep
        "host_enqueue_us_median": statistics.median(enqueue_s) * 1e6,
        "gpu_sleep_us": sleep_cycles / (clk.get("sm_max_mhz") or 2070.0),
    }
    if args.e2e:
        result["e2e"] = run_e2e(args, w, batch, vsd, dev, stream, workspace, prefix, total_bytes)
    return result, batch


def run_e2e(args, w, batch, vsd, dev, stream, workspace, prefix, total_bytes):
    """The same iteration through the package's public iteration object: every step
    copies the step's inputs from pinned host memory, runs verify -> select -> gamma
    draft steps, and copies every result back to pinned host memory -- all recorded
    once as a CUDA graph and replayed with one launch per step."""
    B, R, Hq, d, gamma = w.B, w.R, w.Hq, w.d, w.gamma
    it = vsd.IterationGraph(batch.k_cache, batch.v_cache, batch.block_table, B=B, R=R, Hq=Hq,
                            gamma=gamma, P_max=w.P_max, k=w.k, n_sink=w.n_sink,
                            n_recent=w.n_recent, max_tail=2 * gamma + 1, scale=w.scale)
    it.h_q.copy_(batch.q.cpu())
    it.h_q_draft.copy_(batch.q_draft.cpu())
    it.h_prefix_len.copy_(batch.prefix_len.cpu())
    it.h_tail_start.copy_(batch.prefix_len.cpu())
    rng = np.random.default_rng(w.seed + 91)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for step in range(args.warmup + args.steps):
        a = rng.integers(0, gamma + 1, size=B)
        it.h_seq_len.copy_(torch.tensor([[prefix[b] + a[b] + 2 + i for b in range(B)]
                                         for i in range(gamma)], dtype=torch.int32))
        flush_l2(flush_w, flush_r)
        torch.cuda.synchronize()
        with torch.cuda.stream(it.stream):
            torch.cuda._sleep(2_000_000)  # the replay is queued before the GPU gets to it
            e0.record(it.stream)
            it.graph.replay()
            e1.record(it.stream)
        it.synchronize()
        if step >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.mean(times)
    return {"value": total_bytes / t / 1e9, "unit": "GB/s", "us_per_iter": t * 1e6,
            "h2d_bytes_per_step": it.h2d_bytes, "d2h_bytes_per_step": it.d2h_bytes,
            "path": "IterationGraph: pinned host inputs -> verify -> select -> %d draft steps "
                    "-> pinned host results, one CUDA-graph replay per step" % gamma}


# ------------------------------------------------------------------ multi-layer loop

def append_bytes(w):
    """Algorithmic bytes of one iteration's cache appends for one layer: the R verify
    rows and the gamma draft-step rows of every sequence and KV head, K and V, read from
    the input arena and written into the cache."""
    return 2 * 2 * w.B * (w.R + w.gamma) * w.Hkv * w.d * 2


def loop_run_bytes(w, accepted):
    """Algorithmic bytes of a decode run (one entry per iteration: verification,
    selection, draft steps and appends over every layer) for the accepted counts
    `accepted` [iterations][B]; the prefixes grow by accepted + 1 per iteration."""
    prefix = list(w.prefix())
    per_iter = []
    for acc in accepted:
        n_sel = [min(w.k, P) for P in prefix]
        tails = [[int(acc[b]) + 2 + i for b in range(w.B)] for i in range(w.gamma)]
        vb, sb, spb = iteration_bytes(w, prefix, n_sel, tails)
        per_iter.append({"verify": w.layers * vb, "select": w.layers * sb,
                         "sparse": w.layers * sum(spb), "append": w.layers * append_bytes(w),
                         "prefix": list(prefix)})
        prefix = [P + int(a) + 1 for P, a in zip(prefix, acc)]
    return per_iter


def run_gpu_loop(args, world, rank, local):
    """Decode runs of a multi-layer model's attention (`DecodeLoop`): every iteration
    runs each layer's scored verification, which first stores that layer's verify-block
    K/V into its cache, one selection over all layers x sequences, advances the prefixes
    by the accepted counts, and runs gamma draft steps over every layer, each storing its
    input token's K/V first.  One step = one run of `w.iterations` iterations from the initial prefix
    (one CUDA-graph replay); the caches (tens of GB) exceed L2, so no flush is needed."""
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build as pkg_build
    from sparse_attention_speculative_gb300.synth import make_batch, seeded_bf16
    from sparse_attention_speculative_gb300.workloads import ALL

    if rank == 0 or not pkg_build.up_to_date():
        pkg_build.build()
    if world > 1:
        torch.distributed.barrier()
    vsd.load()
    w = ALL[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    NL, B, R, Hq, Hkv, d, gamma = w.layers, w.B, w.R, w.Hq, w.Hkv, w.d, w.gamma
    iters = w.iterations
    P_max = max(w.prefix()) + iters * R  # the longest prefix of a run
    batches = [make_batch(w, dev, layer=l, extra_capacity=iters * R + 2 * R)
               for l in range(NL)]
    loop = vsd.DecodeLoop([bt.k_cache for bt in batches], [bt.v_cache for bt in batches],
                          [bt.block_table for bt in batches], list(w.prefix()), Hq=Hq,
                          gamma=gamma, k=w.k, n_sink=w.n_sink, n_recent=w.n_recent,
                          P_max=P_max, scale=w.scale)
    # the iteration's inputs: each layer's seeded queries and the seeded K/V of the new
    # tokens (the same every iteration; the positions they go to move with the prefix)
    for l, bt in enumerate(batches):
        loop.q[l].copy_(bt.q)
        loop.q_draft[l].copy_(bt.q_draft)
    loop.k_verify.copy_(seeded_bf16((NL, B, R, Hkv, d), w.seed * 31 + 1, dev))
    loop.v_verify.copy_(seeded_bf16((NL, B, R, Hkv, d), w.seed * 31 + 2, dev))
    loop.k_draft.copy_(seeded_bf16((NL, gamma, B, Hkv, d), w.seed * 31 + 3, dev))
    loop.v_draft.copy_(seeded_bf16((NL, gamma, B, Hkv, d), w.seed * 31 + 4, dev))
    rng = np.random.default_rng(w.seed + 77)
    n_runs = args.warmup + args.steps
    acc_all = rng.integers(0, gamma + 1, size=(n_runs, iters, B)).astype(np.int32)
    acc_dev = torch.from_numpy(acc_all).to(dev)
    stream = loop.stream
    # one graph of a whole run; each run's accepted draws are copied into its input rows
    # just before its replay (800 bytes, stream-ordered)
    acc_rows = torch.empty((iters, B), dtype=torch.int32, device=dev)
    acc_rows.copy_(acc_dev[0])
    t_cap = time.perf_counter()
    run_graph = loop.record_run(acc_rows)
    t_cap = time.perf_counter() - t_cap
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x after capture" % status)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for r in range(args.warmup):
            acc_rows.copy_(acc_dev[r])
            run_graph.replay()
    stream.synchronize()
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x during warm-up" % status)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(8_000_000)  # the first replays are queued before the GPU gets to them
            e0.record(stream)
            for r in range(args.warmup, n_runs):
                acc_rows.copy_(acc_dev[r])
                run_graph.replay()
            e1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    t_total = e0.elapsed_time(e1) * 1e-3
    if world > 1:
        torch.distributed.barrier()
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x in the timed region" % status)
    del run_graph
    run_bytes = [loop_run_bytes(w, acc_all[r]) for r in range(args.warmup, n_runs)]
    total_bytes = sum(sum(it["verify"] + it["select"] + it["sparse"] + it["append"]
                          for it in rb) for rb in run_bytes)
    t_tensor = torch.tensor([t_total], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_tensor, op=torch.distributed.ReduceOp.MAX)
    t_max = float(t_tensor.item())
    value = world * total_bytes / t_max / 1e9
    peak, peak_kind = measured_peaks()
    clk = clocks.summary()

    # per-phase breakdown: one run of iterations from a graph with external event
    # records at the phase boundaries (verify = the layers' verifications, each storing
    # its verify block's K/V; select = the selection + the advance; draft = the draft
    # steps, each storing its input token's K/V)
    marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    g_marked = loop.record_marked({"verified": lambda: marks[1].record(stream),
                                   "selected": lambda: marks[2].record(stream),
                                   "drafted": lambda: marks[3].record(stream)},
                                  first=lambda: marks[0].record(stream))
    phase = {"verify": [], "select": [], "sparse": []}
    acc_ph = acc_all[args.warmup]
    with torch.cuda.stream(stream):
        loop.reset()
        for it in range(iters):
            loop.accepted.copy_(acc_dev[args.warmup, it])
            g_marked.replay()
            stream.synchronize()
            phase["verify"].append(marks[0].elapsed_time(marks[1]) * 1e-3)
            phase["select"].append(marks[1].elapsed_time(marks[2]) * 1e-3)
            phase["sparse"].append(marks[2].elapsed_time(marks[3]) * 1e-3)
    del g_marked
    ph_bytes = loop_run_bytes(w, acc_ph)
    t_v, t_s, t_sp = (statistics.mean(phase[k]) for k in ("verify", "select", "sparse"))
    b_v = statistics.mean(it["verify"] + it["append"] * R / (R + gamma) for it in ph_bytes)
    b_s = statistics.mean(it["select"] for it in ph_bytes)
    b_sp = statistics.mean(it["sparse"] + it["append"] * gamma / (R + gamma) for it in ph_bytes)
    nominal = NOMINAL_HBM_GBS

    def entry(t, nbytes, calls):
        return {"us": t * 1e6, "calls": calls, "us_per_call": t * 1e6 / calls, "bytes": nbytes,
                "GB_s": nbytes / t / 1e9, "frac_of_%s_hbm" % peak_kind: nbytes / t / 1e9 / peak,
                "frac_of_nominal_8tbs": nbytes / t / 1e9 / nominal}

    # the dominant kernel: the layers' verification calls inside the iteration (their
    # phase between two event records in the graph, the calls' verify-block stores
    # included), algorithmic bytes of the calls / phase time
    verify_call_bytes = statistics.mean(it["verify"] for it in ph_bytes) / NL
    achieved = statistics.mean(it["verify"] for it in ph_bytes) / t_v / 1e9
    us_iter = t_max / (args.steps * iters) * 1e6
    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
        "us_per_iter": us_iter, "iterations_per_step": iters,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": NL, "B": B, "P": w.P, "Hq": Hq, "Hkv": Hkv,
                   "d": d, "gamma": gamma, "k": w.k, "n_sink": w.n_sink,
                   "n_recent": w.n_recent, "page": w.page, "iterations": iters,
                   "prefix": "starts at P and grows by accepted + 1 every iteration "
                             "(accepted ~ uniform{0..gamma}, seeded); the verify block's "
                             "and every draft token's K/V are appended inside the graph",
                   "l2": "no flush: every iteration streams %.1f GB from %.1f GB of caches "
                         "(far larger than the 126 MB L2)"
                         % (total_bytes / (args.steps * iters) / 1e9,
                            2 * NL * batches[0].k_cache.numel() * 2 / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "timing": "value: %d runs of %d iterations, each run one CUDA-graph replay (%d libvsd "
                  "kernels per iteration), device events around all runs; phases: one run "
                  "from a graph with event records at the phase boundaries"
                  % (args.steps, iters, loop.launches_per_iteration),
        "graph_capture_s": t_cap,
        "phases": {"verify_collect": entry(t_v, b_v, NL),
                   "select_topk": entry(t_s, b_s, 1),
                   "sparse_draft_steps": entry(t_sp, b_sp, gamma * NL)},
        "select_over_verify_call": t_s / (t_v / NL),
        "roofline": {"bound": "hbm", "kernel": "vsd_verify_attn_collect_scored",
                     "timing": "the %d layers' verification calls inside the iteration (their "
                               "phase between event records in the iteration graph, each call "
                               "storing its verify block's K/V), per call; bytes = "
                               "algorithmic bytes of one call at the run's prefixes" % NL,
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak,
                     "bytes_per_call": verify_call_bytes,
                     "traffic": profile_traffic("qwen3_8b_loop_layer", verify_call_bytes)},
        "gpu_launches": loop.launches_per_iteration * iters * args.steps + args.steps,
        "gpu_launches_per_iteration": loop.launches_per_iteration,
        "clocks": clk,
    }
    if args.e2e:
        # the same runs through the public API as a caller drives it: per iteration the
        # host fills the pinned input arena (its accepted counts), DecodeLoop.run(sync=True)
        # copies the inputs in, runs the iteration and copies every result back, and the
        # host waits for it; host wall clock around every call, no GPU sleep in front
        for name in ("q", "q_draft", "k_verify", "v_verify", "k_draft", "v_draft"):
            getattr(loop, "h_" + name).copy_(getattr(loop, name))
        walls = []
        for r in range(n_runs):
            loop.reset()
            loop.synchronize()
            for it in range(iters):
                loop.h_accepted.copy_(torch.from_numpy(acc_all[r, it]))
                t0 = time.perf_counter()
                loop.run(sync=True)
                t1 = time.perf_counter()
                if r >= args.warmup:
                    walls.append(t1 - t0)
        status = vsd.vsd_read_device_status()
        if status:
            raise RuntimeError("device status 0x%x in the end-to-end runs" % status)
        t_wall = sum(walls)
        result["e2e"] = {"value": total_bytes / t_wall / 1e9, "unit": "GB/s",
                         "wall_us_per_iter": t_wall / len(walls) * 1e6,
                         "h2d_bytes_per_step": loop.h2d_bytes * iters,
                         "d2h_bytes_per_step": loop.d2h_bytes * iters,
                         "path": "DecodeLoop.run(sync=True) per iteration (host wall clock): "
                                 "pinned host inputs (queries, new K/V, accepted counts) -> "
                                 "the iteration -> every output, selection and the loop "
                                 "state back to pinned host memory; %d iterations per step"
                                 % iters}
    if rank == 0 and args.cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline_loop(w, batches)
    if args.configs and rank == 0:
        # the single-layer configurations' per-call figures, from the same run
        del loop, batches
        torch.cuda.empty_cache()
        result["configs"] = {}
        for name in ("qwen3_8b_32k", "qwen25_72b_b16_32k", "qwen3_8b_128k_bursts"):
            result["configs"][name] = layer_figures(ALL[name], dev, peak, peak_kind)
    return result


def layer_figures(w, dev, peak, peak_kind, reps=10, chain=20):
    """Per-call figures of one single-layer configuration, three ways, each from CUDA
    graphs replayed with L2 flushed before every replay (512 MB written, then 512 MB
    read) and a GPU sleep in front so the replay is queued before the GPU reaches it:
      iteration   verify (main + merge/aggregation kernel) -> select -> gamma draft
                  steps, device events around the replay;
      in_iteration the same graph with external event records between the calls: each
                  call's share of it (the verification's share includes the start of the
                  replay, the other calls lose their overlap with their predecessor);
      chained     `chain` calls of one kind back to back in one graph (each a
                  programmatic dependent of the previous one), time / chain."""
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300.synth import make_batch
    batch = make_batch(w, dev)
    B, R, Hq, d, gamma = w.B, w.R, w.Hq, w.d, w.gamma
    P_max = w.P_max
    prefix = list(w.prefix())
    stream = torch.cuda.current_stream()
    geom = vsd.geom_for(B, Hq, batch.k_cache, batch.block_table)
    nb = vsd.vsd_verify_workspace_size(geom, R, P_max)
    ws = torch.zeros(nb + 256, dtype=torch.uint8, device=dev)
    ws = ws[(-ws.data_ptr()) % 256:][:nb] if nb else None
    max_tail = 2 * gamma + 1
    nb = vsd.vsd_sparse_workspace_size(geom, w.k, max_tail)
    sws = torch.zeros(nb + 256, dtype=torch.uint8, device=dev)
    sws = sws[(-sws.data_ptr()) % 256:][:nb] if nb else None
    out = torch.empty_like(batch.q)
    logits = torch.empty((B, 2, Hq, P_max), dtype=torch.float32, device=dev)
    partial = torch.empty((B, w.Hkv, P_max), dtype=torch.float32, device=dev)
    score = torch.empty((B, P_max), dtype=torch.float32, device=dev)
    hist = torch.empty((B, vsd.HIST_BINS), dtype=torch.int32, device=dev)
    idx = torch.empty((B, w.k), dtype=torch.int32, device=dev)
    n_sel = torch.empty((B,), dtype=torch.int32, device=dev)
    d_out = torch.empty((gamma, B, Hq, d), dtype=torch.bfloat16, device=dev)
    tail_start = batch.prefix_len.clone()
    a = np.random.default_rng(w.seed + 77).integers(0, gamma + 1, size=B)
    seq_len = torch.tensor([[prefix[b] + int(a[b]) + 2 + i for b in range(B)]
                            for i in range(gamma)], dtype=torch.int32, device=dev)

    def verify():
        # (its predecessor in every graph below writes neither the cache below the
        # prefix nor the lengths or block table: the first tiles are fetched before the
        # dependency wait)
        vsd.vsd_verify_attn_collect_scored(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, P_max=P_max,
                                           scale=w.scale, row0=0, row1=R - 1, logits=logits,
                                           partial=partial, score=score, score_hist=hist,
                                           n_sink=w.n_sink, n_recent=w.n_recent,
                                           flags=vsd.VERIFY_EARLY_PREFETCH, out=out,
                                           workspace=ws)

    def select():
        vsd.vsd_select_topk_scored(score, hist, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                   n_recent=w.n_recent, idx=idx, n_sel=n_sel)

    # the draft steps run as a decode loop runs them: the first step after the
    # selection records the selected positions' cache rows, the later ones reuse them,
    # and those whose inputs were all written two or more launches back gather before
    # waiting for their predecessor
    rows = torch.zeros((B, w.k), dtype=torch.int32, device=dev)

    def draft(i, flags=None):
        if flags is None:
            flags = (vsd.STEP_RECORD_ROWS if i == 0 else
                     vsd.STEP_REUSE_ROWS | (vsd.STEP_EARLY_GATHER if i >= 2 else 0))
        vsd.vsd_sparse_decode_attn_step(batch.q_draft[i], batch.k_cache, batch.v_cache,
                                        batch.block_table, idx, n_sel, tail_start, seq_len[i],
                                        scale=w.scale, max_tail=max_tail, sel_rows=rows,
                                        flags=flags, out=d_out[i], workspace=sws)

    # Dustin's sparse verification over the selection (the fused kernel where R * G <= 32)
    sv_geom = vsd.geom_for(B, Hq, batch.k_cache, batch.block_table)
    nb = vsd.vsd_sparse_verify_workspace_size(sv_geom, R, w.k)
    sv_ws = torch.zeros(nb + 256, dtype=torch.uint8, device=dev)
    sv_ws = sv_ws[(-sv_ws.data_ptr()) % 256:][:nb]
    sv_out = torch.empty_like(batch.q)

    def sparse_verify(flags=0):
        vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                   batch.prefix_len, idx, n_sel, scale=w.scale, flags=flags,
                                   out=sv_out, workspace=sv_ws)

    marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3 + gamma)]

    def iteration(marked=False):
        cur = torch.cuda.current_stream()  # the capturing stream inside a capture
        if marked:
            marks[0].record(cur)
        verify()
        if marked:
            marks[1].record(cur)
        select()
        if marked:
            marks[2].record(cur)
        for i in range(gamma):
            draft(i)
            if marked:
                marks[3 + i].record(cur)

    iteration()
    torch.cuda.synchronize()
    graphs = {}
    for name, fn in (("iteration", iteration), ("in_iteration", lambda: iteration(True)),
                     ("verify", lambda: [verify() for _ in range(chain)]),
                     ("select", lambda: [select() for _ in range(chain)]),
                     ("draft", lambda: [draft(i % gamma, vsd.STEP_REUSE_ROWS |
                                              vsd.STEP_EARLY_GATHER) for i in range(chain)]),
                     # (back-to-back calls write nothing another call reads: the
                     # selected rows are gathered before the dependency wait)
                     ("sparse_verify", lambda: [sparse_verify(vsd.SPARSE_VERIFY_EARLY_GATHER)
                                                for _ in range(chain)])):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = {k: [] for k in graphs}
    phases = []
    for rep in range(reps + 2):
        for name, g in graphs.items():
            flush_l2(flush_w, flush_r)
            torch.cuda.synchronize()
            torch.cuda._sleep(2_000_000)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            if rep >= 2:
                times[name].append(e0.elapsed_time(e1) * 1e-3)
                if name == "in_iteration":
                    phases.append([marks[i].elapsed_time(marks[i + 1]) * 1e-3
                                   for i in range(2 + gamma)])
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x in the per-call figures of %s" % (status, w.name))
    n_sel_host = n_sel.cpu().tolist()
    tails = [[int(a[b]) + 2 + i for b in range(B)] for i in range(gamma)]
    vb, sb, spb = iteration_bytes(w, prefix, n_sel_host, tails)
    t = {k: statistics.median(v) for k, v in times.items()}
    ph = [statistics.median(p[i] for p in phases) for i in range(2 + gamma)]

    def fig(tt, nbytes):
        return {"us": tt * 1e6, "bytes": nbytes, "GB_s": nbytes / tt / 1e9,
                "frac_of_%s_hbm" % peak_kind: nbytes / tt / 1e9 / peak}

    res = {"iteration": fig(t["iteration"], vb + sb + sum(spb)),
           "in_iteration": {"verify_collect_scored": fig(ph[0], vb),
                            "select_topk_scored_us": ph[1] * 1e6,
                            "select_over_verify": ph[1] / ph[0],
                            "draft_steps": [fig(ph[2 + i], spb[i]) for i in range(gamma)]},
           "chained": {"verify_collect_scored": fig(t["verify"] / chain, vb),
                       "select_topk_scored_us": t["select"] / chain * 1e6,
                       "select_over_verify": t["select"] / t["verify"],
                       "sparse_draft_step": fig(t["draft"] / chain, statistics.mean(spb)),
                       "sparse_verify": fig(t["sparse_verify"] / chain,
                                            sparse_verify_bytes(w, n_sel_host))},
           "timing": "CUDA graphs, L2 flushed before every replay, medians of %d replays; "
                     "in_iteration: event records between the calls of the iteration graph; "
                     "chained: %d calls of one kind in one graph" % (reps, chain),
           "draft_calls": "vsd_sparse_decode_attn_step as a decode loop calls it: step 0 "
                          "records the selection's cache rows, later steps reuse them, steps "
                          ">= 2 (chained: every call) gather before waiting for their "
                          "predecessor",
           "shape": {"B": B, "P": w.P, "Hq": Hq, "Hkv": w.Hkv, "d": d, "gamma": gamma,
                     "k": w.k}}
    del graphs
    return res


def run_cpu_baseline_loop(w, batches, layers_sample=4):
    """The fp64 oracle on a sample of the loop's layers (one iteration each), the time
    scaled to all layers."""
    import oracle
    from sparse_attention_speculative_gb300.synth import host_arrays
    oracle.build()
    prefix = list(w.prefix())
    n = min(layers_sample, w.layers)
    hs = [host_arrays(batches[l]) for l in range(n)]
    t0 = time.perf_counter()
    vb = sb = 0
    spb_total = 0
    for l in range(n):
        n_sel, tails = cpu_oracle_iteration(w, hs[l], prefix, 1234 + l)
        v_l, s_l, sp_l = iteration_bytes(w, prefix, n_sel, tails)
        vb, sb, spb_total = vb + v_l, sb + s_l, spb_total + sum(sp_l)
    dt = time.perf_counter() - t0
    return {"value": (vb + sb + spb_total) / dt / 1e9, "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "seconds_per_iter": dt * w.layers / n,
            "sample": "%d of the %d layers of one iteration of %s (each: verify+collect2, "
                      "select, %d draft steps), fp64 C oracle; seconds_per_iter scales the "
                      "sample to all layers" % (n, w.layers, w.name, w.gamma)}


# ------------------------------------------------------------------ oracle (CPU) arm

def cpu_oracle_iteration(w, h, prefix, steps_seed):
    """One iteration of the fp64 oracle on the host: verify, select, gamma drafts."""
    import oracle
    out, logits, partial = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                         h["prefix_len"], scale=w.scale, P_max=w.P_max)
    score = oracle.score_from_logits(logits, h["prefix_len"])
    idx, n_sel = oracle.select(score, h["prefix_len"], k=w.k, n_sink=w.n_sink,
                               n_recent=w.n_recent)
    rng = np.random.default_rng(steps_seed)
    a = rng.integers(0, w.gamma + 1, size=w.B)
    tails = []
    for i in range(w.gamma):
        sl = np.array([prefix[b] + a[b] + 2 + i for b in range(w.B)], np.int32)
        oracle.sparse_decode(h["q_draft"][i], h["k_cache"], h["v_cache"], h["block_table"], idx,
                             n_sel, h["prefix_len"], sl, scale=w.scale)
        tails.append([int(sl[b] - prefix[b]) for b in range(w.B)])
    return n_sel.tolist(), tails


def run_cpu_baseline(w, batch, iters=3):
    import oracle
    from sparse_attention_speculative_gb300.synth import host_arrays
    oracle.build()
    h = host_arrays(batch)
    prefix = list(w.prefix())
    t0 = time.perf_counter()
    for i in range(iters):
        n_sel, tails = cpu_oracle_iteration(w, h, prefix, 1234 + i)
    dt = (time.perf_counter() - t0) / iters
    vb, sb, spb = iteration_bytes(w, prefix, n_sel, tails)
    total = vb + sb + sum(spb)
    return {"value": total / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds_per_iter": dt,
            "sample": "%d full iteration(s) of %s (verify+collect2, select, %d draft steps), "
                      "fp64 C oracle" % (iters, w.name, w.gamma)}


def run_reference(args, world, rank):
    """The oracle as the reference arm: same workload, metric and unit."""
    if rank != 0:
        return None
    import oracle
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import ALL
    oracle.build()
    w = ALL[args.workload]
    batch = make_batch(w, "cpu")
    h = host_arrays(batch)
    prefix = list(w.prefix())
    for i in range(min(args.warmup, 1)):
        cpu_oracle_iteration(w, h, prefix, 99 + i)
    times = []
    n_sel, tails = None, None
    for i in range(args.steps):
        t0 = time.perf_counter()
        n_sel, tails = cpu_oracle_iteration(w, h, prefix, 1000 + i)
        times.append(time.perf_counter() - t0)
    vb, sb, spb = iteration_bytes(w, prefix, n_sel, tails)
    total = vb + sb + sum(spb)
    t = sum(times)
    value = total * args.steps / t / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "gamma": w.gamma, "k": w.k, "n_sink": w.n_sink, "n_recent": w.n_recent},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": ("each step one full iteration of %s on the host" % w.name
                                    if w.layers == 1 else
                                    "each step one layer (of %d, the rate is the same for "
                                    "every layer) of one iteration of %s on the host"
                                    % (w.layers, w.name))},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def profile_call(args):
    """One libvsd call of a single-layer workload, --warmup untimed then --steps more
    times, nothing else: the command an ncu capture runs (few launches, few GB)."""
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build as pkg_build
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import ALL
    pkg_build.build()
    vsd.load()
    w = ALL[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    batch = make_batch(w, dev)
    B, R, gamma = w.B, w.R, w.gamma
    out, logits, partial, score, hist = vsd.vsd_verify_attn_collect_scored(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale, n_sink=w.n_sink, n_recent=w.n_recent)
    idx, n_sel = vsd.vsd_select_topk_scored(score, hist, batch.prefix_len, k=w.k,
                                            n_sink=w.n_sink, n_recent=w.n_recent)
    seq_len = batch.prefix_len + R
    for _ in range(args.warmup + args.steps):
        if args.profile_call == "verify":
            vsd.vsd_verify_attn_collect_scored(batch.q, batch.k_cache, batch.v_cache,
                                               batch.block_table, batch.prefix_len,
                                               P_max=w.P_max, scale=w.scale, logits=logits,
                                               partial=partial, score=score, score_hist=hist,
                                               n_sink=w.n_sink, n_recent=w.n_recent, out=out)
        elif args.profile_call == "select":
            vsd.vsd_select_topk_scored(score, hist, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                       n_recent=w.n_recent, idx=idx, n_sel=n_sel)
        elif args.profile_call == "sparse_verify":
            vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                       batch.prefix_len, idx, n_sel, scale=w.scale)
        else:
            vsd.vsd_sparse_decode_attn(batch.q_draft[0], batch.k_cache, batch.v_cache,
                                       batch.block_table, idx, n_sel, batch.prefix_len,
                                       seq_len, scale=w.scale, max_tail=2 * gamma + 1)
    torch.cuda.synchronize()
    status = vsd.vsd_read_device_status()
    if status:
        raise RuntimeError("device status 0x%x" % status)
    print("profile-call %s on %s: %d calls" % (args.profile_call, w.name,
                                               args.warmup + args.steps))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="qwen3_8b_36layer_loop")
    ap.add_argument("--impl", default="vsd", choices=["vsd", "reference"])
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--profile-call", choices=["verify", "select", "draft", "sparse_verify"],
                    default=None,
                    help="run one call of the workload --steps times and exit (for ncu)")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the single-layer configurations' per-call figures (loop only)")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.profile_call:
        profile_call(args)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    from sparse_attention_speculative_gb300.workloads import ALL
    w = ALL[args.workload]
    if w.layers > 1:
        res = run_gpu_loop(args, world, rank, local)
    else:
        res, batch = run_gpu(args, world, rank, local)
        if rank == 0 and args.cpu_baseline:
            res["cpu_baseline"] = run_cpu_baseline(w, batch)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
