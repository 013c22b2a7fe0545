"""GPU parity: every kernel of the hot path, called through the C ABI, against the
fp64 oracle on the same seeded inputs (comparison rules in parity_utils)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import (assert_attn_close, assert_index_sets, assert_rel_close,
                                fp32_row_sum)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_speculative_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)
    yield


def _vsd():
    import sparse_attention_speculative_gb300 as vsd
    return vsd


def run_verify(batch, w, row0=0, row1=None):
    vsd = _vsd()
    out, logits, partial = vsd.vsd_verify_attn_collect(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale, row0=row0, row1=row1)
    torch.cuda.synchronize()
    return out, logits, partial


def check_verify(batch, w, row0=0, row1=None, status_ok=True):
    from sparse_attention_speculative_gb300.synth import host_arrays
    vsd = _vsd()
    out, logits, partial = run_verify(batch, w, row0, row1)
    status = vsd.vsd_read_device_status()
    if status_ok:
        assert status == 0, "device status 0x%x" % status
    h = host_arrays(batch)
    o_ref, l_ref, p_ref = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                        h["prefix_len"], scale=w.scale, P_max=w.P_max,
                                        row0=row0, row1=row1)
    assert_attn_close(out.float().cpu().numpy(), o_ref, "verify output")
    lg = logits.cpu().numpy()
    pa = partial.cpu().numpy()
    for b, P in enumerate(h["prefix_len"].tolist()):
        assert_rel_close(lg[b, :, :, :P], l_ref[b, :, :, :P], "collected logits")
        assert_rel_close(pa[b, :, :P], p_ref[b, :, :P], "partial scores")
    return out, logits, partial, (o_ref, l_ref, p_ref), h


def check_select(partial, prefix_len, w, s_ref_fp64=None):
    vsd = _vsd()
    idx, n_sel, scores = vsd.vsd_select_topk(partial, prefix_len, k=w.k, n_sink=w.n_sink,
                                             n_recent=w.n_recent, want_scores=True)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    pl = prefix_len.cpu().numpy()
    pa = partial.cpu().numpy()
    # 1) same input, decision in the kernel's precision (fp32 sum in group order): exact
    s32 = fp32_row_sum(pa)
    i32, n32 = oracle.select(s32, pl, k=w.k, n_sink=w.n_sink, n_recent=w.n_recent)
    gi, gn = idx.cpu().numpy(), n_sel.cpu().numpy()
    for r, P in enumerate(pl.tolist()):
        assert gn[r] == n32[r]
        np.testing.assert_array_equal(gi[r, :gn[r]], i32[r, :n32[r]])
        assert np.all(gi[r, gn[r]:] == -1)
    # 2) the aggregated score itself against the oracle's fp64 aggregation
    s64 = oracle.score_from_partials(pa, pl)
    sc = scores.cpu().numpy()
    for r, P in enumerate(pl.tolist()):
        assert_rel_close(sc[r, :P], s64[r, :P], "aggregated score")
    # 3) against the oracle's end-to-end fp64 selection, under the tolerance rule
    if s_ref_fp64 is not None:
        i64, n64 = oracle.select(s_ref_fp64, pl, k=w.k, n_sink=w.n_sink, n_recent=w.n_recent)
        assert_index_sets(gi, gn, i64, n64, s_ref_fp64, pl, w.k, w.n_sink, w.n_recent)
    return idx, n_sel


def check_sparse(batch, w, idx, n_sel, tail_start, seq_len, q=None, max_tail=None):
    from sparse_attention_speculative_gb300.synth import host_arrays, to_u16
    vsd = _vsd()
    q = batch.q_draft[0] if q is None else q
    if max_tail is None:
        max_tail = int((seq_len - tail_start).max().item())
    out = vsd.vsd_sparse_decode_attn(q, batch.k_cache, batch.v_cache, batch.block_table, idx,
                                     n_sel, tail_start, seq_len, scale=w.scale,
                                     max_tail=max_tail)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    h = host_arrays(batch)
    ref = oracle.sparse_decode(to_u16(q), h["k_cache"], h["v_cache"], h["block_table"],
                               None if idx is None else idx.cpu().numpy(),
                               None if n_sel is None else n_sel.cpu().numpy(),
                               tail_start.cpu().numpy(), seq_len.cpu().numpy(), scale=w.scale)
    assert_attn_close(out.float().cpu().numpy(), ref, "sparse draft output")
    return out


def full_path(w, device="cuda"):
    from sparse_attention_speculative_gb300.synth import make_batch
    batch = make_batch(w, device)
    out, logits, partial, refs, h = check_verify(batch, w)
    s_ref = oracle.score_from_logits(refs[1], h["prefix_len"])
    idx, n_sel = check_select(partial, batch.prefix_len, w, s_ref)
    # every planted heavy hitter is selected, by the kernel and by the oracle's fp64
    # selection alike (the workloads plant fewer than k keys, boosted well clear of the rest)
    i64, n64 = oracle.select(s_ref, h["prefix_len"], k=w.k, n_sink=w.n_sink,
                             n_recent=w.n_recent)
    for b, pos in enumerate(batch.planted):
        planted = set(pos.cpu().tolist())
        sel = set(idx[b, :int(n_sel[b])].cpu().tolist())
        assert not planted - sel, "planted keys not selected: %d" % len(planted - sel)
        assert not planted - set(i64[b, :int(n64[b])].tolist()), "oracle misses planted keys"
    # draft steps: idx plus a dense tail after the verify block start
    tail = batch.prefix_len.clone()
    for step in range(min(w.gamma, 2)):
        seq_len = batch.prefix_len + 2 + step
        check_sparse(batch, w, idx, n_sel, tail, seq_len, q=batch.q_draft[step])
    return batch


def test_tiny_full_path():
    from sparse_attention_speculative_gb300.workloads import TINY
    full_path(TINY)


def test_qwen3_8b_32k_full_path():
    from sparse_attention_speculative_gb300.workloads import QWEN3_8B_32K
    full_path(QWEN3_8B_32K)


@pytest.mark.slow
def test_qwen25_72b_b16_full_path():
    from sparse_attention_speculative_gb300.workloads import QWEN25_72B_B16_32K
    full_path(QWEN25_72B_B16_32K)


@pytest.mark.slow
def test_long_128k_full_path():
    from sparse_attention_speculative_gb300.workloads import LONG_128K
    full_path(LONG_128K)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("d,Hq,Hkv,gamma", [(128, 32, 8, 4), (64, 4, 1, 3), (128, 8, 8, 0),
                                            (64, 16, 2, 7), (128, 64, 8, 5), (128, 16, 16, 6)])
def test_verify_ragged_geometries(d, Hq, Hkv, gamma):
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    prefix = (0, 1, 127, 128, 129, 1000, 3001)
    w = Workload("ragged", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma,
                 k=64, n_sink=4, n_recent=16, planted_frac=0.01, seed=9, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    row1 = w.R - 1
    check_verify(batch, w, row0=0, row1=row1)


def test_verify_collect_other_rows():
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("rows", B=2, P=700, Hq=8, Hkv=2, d=128, gamma=5, k=64, n_sink=4, n_recent=16,
                 seed=3, prefix_lens=(700, 333))
    batch = make_batch(w, "cuda")
    check_verify(batch, w, row0=2, row1=2)
    check_verify(batch, w, row0=4, row1=1)


def test_verify_deterministic():
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import QWEN3_8B_32K
    w = QWEN3_8B_32K.with_(P=8000)
    batch = make_batch(w, "cuda")
    a = [t.clone() for t in run_verify(batch, w)]
    b = run_verify(batch, w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_verify_bad_block_is_flagged_not_faulted():
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("bad", B=1, P=500, Hq=8, Hkv=2, d=128, gamma=3, k=64, n_sink=4, n_recent=16,
                 seed=5)
    batch = make_batch(w, "cuda")
    batch.block_table[0, 3] = batch.num_blocks + 7  # out of range entry
    run_verify(batch, w)
    assert vsd.vsd_read_device_status() & vsd.DEV_BAD_BLOCK
    assert vsd.vsd_read_device_status() == 0  # reading clears


def test_select_ties_and_small_prefixes():
    vsd = _vsd()
    rng = np.random.default_rng(0)
    prefix = np.array([0, 1, 5, 20, 64, 65, 300, 4096, 20000], np.int32)
    P_max = int(prefix.max())
    Hkv = 4
    # integer-valued partials: many exact ties in the aggregated score
    partial = rng.integers(-3, 4, size=(len(prefix), Hkv, P_max)).astype(np.float32)
    pt = torch.tensor(partial, device="cuda")
    pl = torch.tensor(prefix, device="cuda")
    from sparse_attention_speculative_gb300.workloads import Workload
    for k, ns, nr in [(64, 4, 16), (20, 20, 0), (300, 16, 256), (1, 0, 1), (5000, 4, 64)]:
        w = Workload("sel", B=len(prefix), P=P_max, Hq=8, Hkv=Hkv, d=128, gamma=1, k=k,
                     n_sink=ns, n_recent=nr)
        check_select(pt, pl, w)


def test_select_rare_paths():
    """Boundary bins the first histogram level cannot split: every score equal (all
    three levels, then the tie rule alone decides by position), and scores packed in a
    narrow range (a second level, then the gathered keys resolve the rest)."""
    rng = np.random.default_rng(7)
    from sparse_attention_speculative_gb300.workloads import Workload
    for n_rows in (1, 9):
        P_max, Hkv = 32768, 2
        prefix = np.full(n_rows, P_max, np.int32)
        prefix[1:] = rng.integers(20000, P_max + 1, size=n_rows - 1)
        equal = np.zeros((n_rows, Hkv, P_max), np.float32)
        narrow = (50.0 + rng.uniform(0.0, 0.01, size=(n_rows, Hkv, P_max))).astype(np.float32)
        mixed = np.where(rng.random((n_rows, 1, P_max)) < 0.5, 0.0,
                         rng.normal(size=(n_rows, Hkv, P_max))).astype(np.float32)
        for partial in (equal, narrow, mixed):
            w = Workload("rare", B=n_rows, P=P_max, Hq=8, Hkv=Hkv, d=128, gamma=1, k=2048,
                         n_sink=16, n_recent=256)
            check_select(torch.tensor(partial, device="cuda"), torch.tensor(prefix, device="cuda"),
                         w)


def test_select_many_rows_one_launch():
    rng = np.random.default_rng(1)
    n_rows, Hkv, P_max = 40, 8, 65536
    prefix = rng.integers(1000, P_max + 1, size=n_rows).astype(np.int32)
    partial = rng.normal(size=(n_rows, Hkv, P_max)).astype(np.float32)
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("rows", B=n_rows, P=P_max, Hq=32, Hkv=Hkv, d=128, gamma=5, k=4096, n_sink=16,
                 n_recent=256)
    check_select(torch.tensor(partial, device="cuda"), torch.tensor(prefix, device="cuda"), w)


def test_sparse_edge_cases():
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("sp", B=4, P=3000, Hq=16, Hkv=4, d=128, gamma=3, k=256, n_sink=4, n_recent=16,
                 seed=4, prefix_lens=(3000, 17, 0, 1200))
    batch = make_batch(w, "cuda")
    dev = "cuda"
    k_max = 256
    idx = torch.full((w.B, k_max), -1, dtype=torch.int32, device=dev)
    n_sel = torch.zeros((w.B,), dtype=torch.int32, device=dev)
    g = torch.Generator(device="cpu").manual_seed(0)
    for b, P in enumerate(w.prefix()):
        n = min(P, 200)
        if n:
            sel = torch.sort(torch.randperm(P, generator=g)[:n]).values
            idx[b, :n] = sel.to(torch.int32).to(dev)
            n_sel[b] = n
    tail = batch.prefix_len.clone()
    seq_len = batch.prefix_len + torch.tensor([3, 1, 2, 0], dtype=torch.int32, device=dev)
    check_sparse(batch, w, idx, n_sel, tail, seq_len)
    # dense decode: no indices, the whole cache as the tail
    zero = torch.zeros_like(tail)
    check_sparse(batch, w, None, None, zero, batch.prefix_len + 2)
    # duplicates are attended twice
    idx2 = idx.clone()
    idx2[0, 1] = idx2[0, 0]
    check_sparse(batch, w, idx2, n_sel, tail, seq_len)


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (128, 64, 8), (128, 8, 8), (64, 16, 8)])
def test_sparse_many_splits_one_launch(d, Hq, Hkv):
    """More splits than one wave of the one-split kernel holds (8 sequences x 8 KV heads x
    33 splits), with lists of every shape in the same launch: long (many splits, merged),
    one batch and just over it, a single short split (direct output), the tail alone, and
    an empty list."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    prefix = (6000, 5000, 4500, 300, 129, 128, 17, 0)
    w = Workload("spws", B=8, P=6000, Hq=Hq, Hkv=Hkv, d=d, gamma=3, k=4096, n_sink=0,
                 n_recent=0, seed=12, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    dev = "cuda"
    n_per = [4096, 2000, 129, 128, 100, 0, 5, 0]
    idx = torch.full((w.B, 4096), -1, dtype=torch.int32, device=dev)
    n_sel = torch.tensor(n_per, dtype=torch.int32, device=dev)
    g = torch.Generator(device="cpu").manual_seed(1)
    for b, (P, n) in enumerate(zip(prefix, n_per)):
        if n:
            idx[b, :n] = torch.sort(torch.randperm(P, generator=g)[:n]).values.to(torch.int32).to(dev)
    tail = batch.prefix_len.clone()
    seq_len = batch.prefix_len + torch.tensor([3, 1, 2, 0, 4, 2, 1, 3], dtype=torch.int32,
                                              device=dev)
    check_sparse(batch, w, idx, n_sel, tail, seq_len, max_tail=4)


def test_sparse_bad_index_is_flagged():
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("spbad", B=1, P=100, Hq=8, Hkv=2, d=128, gamma=1, k=8, n_sink=0, n_recent=0,
                 seed=1)
    batch = make_batch(w, "cuda")
    idx = torch.tensor([[0, 5, 999999]], dtype=torch.int32, device="cuda")
    n_sel = torch.tensor([3], dtype=torch.int32, device="cuda")
    tail = batch.prefix_len.clone()
    vsd.vsd_sparse_decode_attn(batch.q_draft[0], batch.k_cache, batch.v_cache, batch.block_table,
                               idx, n_sel, tail, batch.prefix_len + 1, scale=w.scale, max_tail=1)
    assert vsd.vsd_read_device_status() & vsd.DEV_BAD_INDEX


def test_sparse_tail_beyond_the_plan_is_refused():
    """A tail longer than the launch was planned for (k_max + max_tail) must not be
    partly attended: the sequence is flagged and gets a zero output."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("sptail", B=2, P=600, Hq=8, Hkv=2, d=128, gamma=1, k=8, n_sink=0, n_recent=0,
                 seed=3)
    batch = make_batch(w, "cuda")
    tail_start = torch.tensor([0, 590], dtype=torch.int32, device="cuda")
    seq_len = torch.tensor([300, 592], dtype=torch.int32, device="cuda")  # 300 > 1 split
    out = vsd.vsd_sparse_decode_attn(batch.q_draft[0], batch.k_cache, batch.v_cache,
                                     batch.block_table, None, None, tail_start, seq_len,
                                     scale=w.scale, max_tail=2)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() & vsd.DEV_BAD_LENGTH
    assert torch.count_nonzero(out[0]) == 0
    # the other sequence is unaffected
    from sparse_attention_speculative_gb300.synth import host_arrays, to_u16
    h = host_arrays(batch)
    ref = oracle.sparse_decode(to_u16(batch.q_draft[0]), h["k_cache"], h["v_cache"],
                               h["block_table"], None, None, tail_start.cpu().numpy(),
                               seq_len.cpu().numpy(), scale=w.scale)
    assert_attn_close(out[1:].float().cpu().numpy(), ref[1:], "sparse output, valid sequence")


def test_sparse_all_prefix_equals_verify_row():
    """k = P (all indices) sparse draft equals the full verify row it mirrors."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("eq", B=2, P=5000, Hq=32, Hkv=8, d=128, gamma=4, k=5000, n_sink=0, n_recent=0,
                 seed=8, prefix_lens=(5000, 4321))
    batch = make_batch(w, "cuda")
    out, _, _ = run_verify(batch, w)
    t = 2
    idx = torch.arange(w.P_max, dtype=torch.int32, device="cuda").repeat(w.B, 1)
    n_sel = batch.prefix_len.clone()
    seq_len = batch.prefix_len + t + 1
    d_out = vsd.vsd_sparse_decode_attn(batch.q[:, t].contiguous(), batch.k_cache, batch.v_cache,
                                       batch.block_table, idx, n_sel, batch.prefix_len.clone(),
                                       seq_len, scale=w.scale, max_tail=t + 1)
    torch.cuda.synchronize()
    diff = (d_out.float() - out[:, t].float()).abs().max().item()
    assert diff <= 2e-2


def test_workspaces_are_left_ready_for_the_next_call():
    """The sparse step's split partials are combined by the last CTA of each
    (sequence, KV head) pair, found through counters at the start of its workspace;
    every call must leave them at zero so the next call starts clean.  Repeated
    calls on one workspace give identical results (verification included)."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("ws", B=2, P=6000, Hq=16, Hkv=4, d=128, gamma=3, k=256, n_sink=4,
                 n_recent=32, seed=21, prefix_lens=(6000, 2500))
    batch = make_batch(w, "cuda")
    geom = vsd.geom_for(w.B, w.Hq, batch.k_cache, batch.block_table)
    nb = vsd.vsd_verify_workspace_size(geom, w.R, w.P_max)
    assert nb > 0, "this geometry must split pairs across CTAs"
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    counter_bytes = ((w.B * w.Hkv * 4 + 255) // 256) * 256
    for rep in range(3):
        out, logits, partial = vsd.vsd_verify_attn_collect(
            batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
            P_max=w.P_max, scale=w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        if rep == 0:
            first = out.clone()
        else:
            assert torch.equal(out, first)
    idx, n_sel, _ = vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                        n_recent=w.n_recent)
    tail = batch.prefix_len.clone()
    seq_len = batch.prefix_len + 3
    sb = vsd.vsd_sparse_workspace_size(geom, w.k, 3)
    assert sb > 0
    sws = torch.zeros(sb, dtype=torch.uint8, device="cuda")
    outs = []
    for rep in range(3):
        o = vsd.vsd_sparse_decode_attn(batch.q_draft[0], batch.k_cache, batch.v_cache,
                                       batch.block_table, idx, n_sel, tail, seq_len,
                                       scale=w.scale, max_tail=3, workspace=sws)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert int(sws[:counter_bytes].count_nonzero()) == 0, "sparse counters not reset"
        outs.append(o.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    check_sparse(batch, w, idx, n_sel, tail, seq_len, max_tail=3)


def test_iteration_graph_matches_eager_calls():
    """The graph-recorded iteration (H2D copies, verify, select, draft steps, D2H copies)
    gives bit-identical results to the same calls made one by one, twice in a row."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("graph", B=2, P=7000, Hq=32, Hkv=8, d=128, gamma=4, k=512, n_sink=16,
                 n_recent=64, planted_frac=0.01, seed=31, prefix_lens=(7000, 4321))
    batch = make_batch(w, "cuda")
    it = vsd.IterationGraph(batch.k_cache, batch.v_cache, batch.block_table, B=w.B, R=w.R,
                            Hq=w.Hq, gamma=w.gamma, P_max=w.P_max, k=w.k, n_sink=w.n_sink,
                            n_recent=w.n_recent, max_tail=2 * w.gamma + 1, scale=w.scale)
    it.h_q.copy_(batch.q.cpu())
    it.h_q_draft.copy_(batch.q_draft.cpu())
    it.h_prefix_len.copy_(batch.prefix_len.cpu())
    it.h_tail_start.copy_(batch.prefix_len.cpu())
    for rep, acc in enumerate(([1, 3], [4, 0])):
        seq = torch.tensor([[P + a + 2 + i for P, a in zip(w.prefix(), acc)]
                            for i in range(w.gamma)], dtype=torch.int32)
        it.h_seq_len.copy_(seq)
        it.run(sync=True)
        assert vsd.vsd_read_device_status() == 0
        out, _, partial = vsd.vsd_verify_attn_collect(
            batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
            P_max=w.P_max, scale=w.scale)
        idx, n_sel, _ = vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                            n_recent=w.n_recent)
        seq_d = seq.cuda()
        drafts = [vsd.vsd_sparse_decode_attn(batch.q_draft[i], batch.k_cache, batch.v_cache,
                                             batch.block_table, idx, n_sel, batch.prefix_len,
                                             seq_d[i], scale=w.scale, max_tail=2 * w.gamma + 1)
                  for i in range(w.gamma)]
        torch.cuda.synchronize()
        assert torch.equal(it.h_out, out.cpu())
        assert torch.equal(it.h_idx, idx.cpu()) and torch.equal(it.h_n_sel, n_sel.cpu())
        for i in range(w.gamma):
            assert torch.equal(it.h_draft_out[i], drafts[i].cpu()), "draft step %d" % i


@pytest.mark.parametrize("d,Hq,Hkv,gamma,prefix", [
    (128, 32, 8, 4, (4000, 129, 0)),     # Qwen3-8B geometry: R*G = 20
    (128, 16, 2, 5, (3001, 1000, 128)),  # R*G = 48, the largest supported
    (64, 8, 8, 3, (127, 2049, 777)),     # G = 1
])
def test_verify_collect_all_rows(d, Hq, Hkv, gamma, prefix):
    """Every verify row collected and the partial score summed over all rows (the
    selection equation as printed), against the all-rows oracle; the attention output
    is the same as with Collect-2-Query."""
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("all", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma, k=64,
                 n_sink=4, n_recent=16, seed=41, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    out, logits, partial = vsd.vsd_verify_attn_collect_all(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale)
    out2, _, _ = vsd.vsd_verify_attn_collect(batch.q, batch.k_cache, batch.v_cache,
                                             batch.block_table, batch.prefix_len, P_max=w.P_max,
                                             scale=w.scale)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(out, out2)
    h = host_arrays(batch)
    o_ref, l_ref, p_ref = oracle.verify_all_rows(h["q"], h["k_cache"], h["v_cache"],
                                                 h["block_table"], h["prefix_len"],
                                                 scale=w.scale, P_max=w.P_max)
    assert_attn_close(out.float().cpu().numpy(), o_ref, "all-rows verify output")
    lg, pa = logits.cpu().numpy(), partial.cpu().numpy()
    for b, P in enumerate(prefix):
        assert_rel_close(lg[b, :, :, :P], l_ref[b, :, :, :P], "all-rows logits")
        assert_rel_close(pa[b, :, :P], p_ref[b, :, :P], "all-rows partial scores")



def test_results_do_not_depend_on_the_split():
    """The split of the work is not part of the result: a sequence verified alone and
    inside a batch (different CTA ranges and split-K merges) agree within the attention
    tolerance with identical collected logits; a draft step planned for a longer tail
    (more, emptier splits) gives the same output bit for bit while the same one-split
    kernel runs, and within the attention tolerance once the plan moves to the
    persistent kernel (which folds each consumer's run of splits into one partial, so
    its additions come in another order)."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("split", B=3, P=9000, Hq=32, Hkv=8, d=128, gamma=4, k=512, n_sink=16,
                 n_recent=64, seed=51, prefix_lens=(9000, 2500, 6000))
    batch = make_batch(w, "cuda")
    out, logits, partial = run_verify(batch, w)
    for b in range(w.B):
        one = type(batch)(w, batch.q[b:b + 1].contiguous(), batch.q_draft[:, b:b + 1].contiguous(),
                          batch.k_cache, batch.v_cache, batch.block_table[b:b + 1].contiguous(),
                          batch.prefix_len[b:b + 1].contiguous(), [batch.planted[b]])
        o1, l1, p1 = run_verify(one, w)
        assert vsd.vsd_read_device_status() == 0
        diff = (o1[0].float() - out[b].float()).abs().max().item()
        assert diff <= 2e-2, diff
        P = int(batch.prefix_len[b])
        assert torch.equal(l1[0, :, :, :P], logits[b, :, :, :P])
        assert torch.equal(p1[0, :, :P], partial[b, :, :P])
    idx, n_sel, _ = vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                        n_recent=w.n_recent)
    tail = batch.prefix_len.clone()
    seq_len = batch.prefix_len + 3
    outs = [vsd.vsd_sparse_decode_attn(batch.q_draft[0], batch.k_cache, batch.v_cache,
                                       batch.block_table, idx, n_sel, tail, seq_len,
                                       scale=w.scale, max_tail=mt) for mt in (3, 200, 2000)]
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(outs[1], outs[0])  # 5 and 6 splits per pair: one split per CTA
    assert_attn_close(outs[2].float().cpu().numpy(), outs[0].float().cpu().numpy(),
                      "draft output, persistent plan")  # 20 splits per pair x 24 pairs


@pytest.mark.parametrize("d,Hq,Hkv,gamma,prefix,k", [
    (128, 32, 8, 4, (6000, 1500, 300), 512),   # Qwen3-8B geometry, ragged: fused, 20 rows
    (128, 64, 8, 5, (4096, 2049), 256),        # Qwen2.5-72B geometry (48 rows): gathered
    (128, 64, 8, 5, (3000, 2000, 2500, 1800), 512),  # the same, four sequences: gathered
    (64, 8, 1, 3, (132000,), 131500),          # a list beyond 1024 batches (32 rows): gathered
    (64, 8, 2, 3, (777, 31), 64),              # head_dim 64, a prefix shorter than k: fused
    (128, 16, 16, 7, (3000, 5000), 2048),      # one head per group, 8 rows, 17 splits
    (128, 32, 4, 3, (9000,), 4096),            # 8 heads per group, 32 rows, 33 splits
    (128, 32, 8, 4, (32768,), 2048),           # the Qwen3-8B 32K layer: one wave
])
def test_sparse_verify(d, Hq, Hkv, gamma, prefix, k):
    """Dustin's sparse verification: each verify row attends the selected set plus the
    verify block up to itself, against the oracle; selecting the whole prefix gives
    full verification."""
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("spv", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma, k=k,
                 n_sink=4, n_recent=32, planted_frac=0.01, seed=61, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    _, _, partial = run_verify(batch, w)
    idx, n_sel, _ = vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                        n_recent=w.n_recent)
    out = vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                     batch.prefix_len, idx, n_sel, scale=w.scale)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    h = host_arrays(batch)
    ref = oracle.sparse_verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                               h["prefix_len"], idx.cpu().numpy(), n_sel.cpu().numpy(),
                               scale=w.scale)
    assert_attn_close(out.float().cpu().numpy(), ref, "sparse verify output")
    # the early-gather form: the same rows, gathered before the dependency wait
    out_early = vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, idx, n_sel,
                                           scale=w.scale, flags=vsd.SPARSE_VERIFY_EARLY_GATHER)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(out_early, out)
    # a workspace of the caller's, reused: calls repeat bit for bit
    geom = vsd.geom_for(w.B, Hq, batch.k_cache, batch.block_table)
    nb = vsd.vsd_sparse_verify_workspace_size(geom, w.R, k)
    ws = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    ws = ws[(-ws.data_ptr()) % 256:][:nb]
    for flags in (0, vsd.SPARSE_VERIFY_EARLY_GATHER, 0):
        again = vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, idx, n_sel,
                                           scale=w.scale, flags=flags, workspace=ws)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert torch.equal(again, out)
    # every prefix position selected: the same as full verification
    full = torch.full((w.B, w.P_max), -1, dtype=torch.int32, device="cuda")
    for b, P in enumerate(prefix):
        full[b, :P] = torch.arange(P, dtype=torch.int32, device="cuda")
    out_all = vsd.vsd_sparse_verify_attn(batch.q, batch.k_cache, batch.v_cache,
                                         batch.block_table, batch.prefix_len, full,
                                         batch.prefix_len.clone(), scale=w.scale)
    out_dense, _, _ = run_verify(batch, w)
    assert vsd.vsd_read_device_status() == 0
    diff = (out_all.float() - out_dense.float()).abs().max().item()
    assert diff <= 2e-2, diff


@pytest.mark.parametrize("n_rows,P_max", [(3, 20000), (9, 9000)])
def test_select_hybrid(n_rows, P_max):
    """Dustin's hybrid budget: the draft signal picks up to m, the target signal fills
    the rest; exact against the oracle fed the same fp32 sums the kernel decides on."""
    vsd = _vsd()
    rng = np.random.default_rng(n_rows)
    prefix = rng.integers(0, P_max + 1, size=n_rows).astype(np.int32)
    prefix[0] = P_max
    pt = rng.integers(-4, 5, size=(n_rows, 4, P_max)).astype(np.float32)  # ties
    pd = rng.normal(size=(n_rows, 2, P_max)).astype(np.float32)
    tpt, tpd = torch.tensor(pt, device="cuda"), torch.tensor(pd, device="cuda")
    tpl = torch.tensor(prefix, device="cuda")
    st, sd = fp32_row_sum(pt), fp32_row_sum(pd)
    for k, m, ns, nr in [(512, 0, 4, 64), (512, 100, 4, 64), (300, 1000, 16, 32), (64, 5, 0, 0)]:
        idx, n_sel = vsd.vsd_select_topk_hybrid(tpt, tpd, tpl, k=k, m=m, n_sink=ns, n_recent=nr)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        ri, rn = oracle.select_hybrid(st, sd, prefix, k=k, m=m, n_sink=ns, n_recent=nr)
        gi, gn = idx.cpu().numpy(), n_sel.cpu().numpy()
        for r in range(n_rows):
            assert gn[r] == rn[r], (k, m, r)
            np.testing.assert_array_equal(gi[r, :gn[r]], ri[r, :rn[r]])
            assert np.all(gi[r, gn[r]:] == -1)


def test_verify_collect_srh_head_mask():
    """Collected importance restricted to a set of query heads (semantic retrieval
    heads): masked-in logits and the masked partial sums against the oracle; the
    masked-out heads' logits are not written."""
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    for Hq, Hkv, gamma in ((32, 8, 4), (64, 8, 5)):
        w = Workload("srh", B=2, P=5000, Hq=Hq, Hkv=Hkv, d=128, gamma=gamma, k=256, n_sink=4,
                     n_recent=32, seed=71, prefix_lens=(5000, 1234))
        batch = make_batch(w, "cuda")
        mask = np.array([1 if (h * 7) % 5 < 2 else 0 for h in range(Hq)], np.uint8)
        out, logits, partial = vsd.vsd_verify_attn_collect_srh(
            batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
            torch.tensor(mask, device="cuda"), P_max=w.P_max, scale=w.scale)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        h = host_arrays(batch)
        o_ref, l_ref, _ = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                        h["prefix_len"], scale=w.scale, P_max=w.P_max)
        p_ref = oracle.partial_masked(l_ref, h["prefix_len"], mask, Hkv)
        assert_attn_close(out.float().cpu().numpy(), o_ref, "srh verify output")
        lg, pa = logits.cpu().numpy(), partial.cpu().numpy()
        for b, P in enumerate(w.prefix()):
            assert_rel_close(pa[b, :, :P], p_ref[b, :, :P], "srh partial scores")
            on = np.nonzero(mask)[0]
            off = np.nonzero(mask == 0)[0]
            assert_rel_close(lg[b][:, on, :P], l_ref[b][:, on, :P], "srh logits")
            assert np.all(lg[b][:, off, :] == 0)


def test_sparse_long_list_cuda_core_step():
    """A selection longer than 1024 batches of 128 positions runs on the CUDA-core draft
    kernel (splits of several batches); against the oracle."""
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    P, k = 200000, 140000
    w = Workload("sparse_long", B=1, P=P, Hq=2, Hkv=1, d=64, gamma=2, k=k, n_sink=4,
                 n_recent=64, seed=91, prefix_lens=(P,))
    batch = make_batch(w, "cuda")
    rng = np.random.default_rng(91)
    sel = np.sort(rng.choice(P, size=k, replace=False)).astype(np.int32)
    idx = torch.tensor(sel[None, :], device="cuda")
    n_sel = torch.tensor([k], dtype=torch.int32, device="cuda")
    tail_start = batch.prefix_len.clone()
    seq_len = batch.prefix_len + w.R
    check_sparse(batch, w, idx, n_sel, tail_start, seq_len, max_tail=w.R)


def test_vsd_copy_host_device():
    """The kernel copy between pinned host memory and the device, both directions,
    bit for bit; sizes that are not a multiple of 16 bytes are refused."""
    vsd = _vsd()
    rng = np.random.default_rng(3)
    src = torch.tensor(rng.integers(0, 256, size=4096 * 3 + 48, dtype=np.uint8)).pin_memory()
    dev = torch.empty(src.numel(), dtype=torch.uint8, device="cuda")
    back = torch.zeros(src.numel(), dtype=torch.uint8).pin_memory()
    vsd.vsd_copy(dev, src)
    vsd.vsd_copy(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(back, src) and torch.equal(dev.cpu(), src)
    with pytest.raises(vsd.VsdError):
        vsd.vsd_copy(dev[:20], src[:20])
