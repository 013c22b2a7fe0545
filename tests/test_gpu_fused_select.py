"""GPU checks of the fused aggregation: the verification call that also writes the
aggregated score and its level-0 histogram, and the selection that starts from them
(Vegas summary sec. 2.A: the objective sums the collected logits over every head)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import assert_rel_close, fp32_row_sum

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


def _keys(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


@pytest.mark.parametrize("d,Hq,Hkv,gamma,prefix", [
    (128, 32, 8, 4, (32768,)),                  # Qwen3-8B 32K layer
    (128, 32, 8, 4, (6001, 0, 1, 511, 4096)),   # ragged, an empty prefix, P_max % 4 != 0
    (128, 64, 8, 5, (3000, 2049)),              # Qwen2.5-72B geometry
    (64, 8, 2, 3, (777, 31)),                   # head_dim 64
])
def test_fused_score_and_histogram(d, Hq, Hkv, gamma, prefix):
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("fused", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma, k=256,
                 n_sink=4, n_recent=32, planted_frac=0.01, seed=81, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    hist0 = torch.full((w.B, vsd.HIST_BINS), 12345, dtype=torch.int32, device="cuda")  # stale
    out_f, lg_f, pa_f, score, hist = vsd.vsd_verify_attn_collect_scored(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale,
        logits=torch.zeros((w.B, 2, Hq, w.P_max), dtype=torch.float32, device="cuda"),
        score_hist=hist0)
    out, lg, pa = vsd.vsd_verify_attn_collect(batch.q, batch.k_cache, batch.v_cache,
                                              batch.block_table, batch.prefix_len, P_max=w.P_max,
                                              scale=w.scale)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(out_f, out)
    for b, P in enumerate(prefix):  # entries at or past P_b are not written
        assert torch.equal(pa_f[b, :, :P], pa[b, :, :P])
    pa_h = pa.cpu().numpy()
    sc = score.cpu().numpy()
    hs = hist.cpu().numpy().view(np.uint32)
    want = fp32_row_sum(pa_h)
    h = host_arrays(batch)
    _, l_ref, _ = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                h["prefix_len"], scale=w.scale, P_max=w.P_max)
    s_ref = oracle.score_from_logits(l_ref, h["prefix_len"])
    for b, P in enumerate(prefix):
        np.testing.assert_array_equal(sc[b, :P], want[b, :P].astype(np.float32))
        assert_rel_close(sc[b, :P], s_ref[b, :P], "aggregated score")
        np.testing.assert_array_equal(hs[b], np.bincount(_keys(sc[b, :P]) >> 20,
                                                         minlength=vsd.HIST_BINS))
    # the early-prefetch form (first prefix tiles fetched before the dependency wait):
    # the same results, bit for bit
    out_e, _, pa_e, score_e, hist_e = vsd.vsd_verify_attn_collect_scored(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale, flags=vsd.VERIFY_EARLY_PREFETCH)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(out_e, out)
    for b, P in enumerate(prefix):
        assert torch.equal(pa_e[b, :, :P], pa[b, :, :P])
        assert torch.equal(score_e[b, :P], score[b, :P])
    assert torch.equal(hist_e, hist)


def test_scored_select_matches_plain_select():
    """Same index sets, bit for bit, as the selection that aggregates itself: ties,
    prefixes shorter than the budget, an empty prefix, every budget mix."""
    vsd = _vsd()
    rng = np.random.default_rng(5)
    B, Hkv, P_max = 6, 4, 20000
    prefix = np.array([20000, 3, 0, 1500, 19999, 8192], np.int32)
    part = rng.integers(-3, 4, size=(B, Hkv, P_max)).astype(np.float32)   # many ties
    part[3:] = rng.normal(size=(3, Hkv, P_max)).astype(np.float32)
    tp = torch.tensor(part, device="cuda")
    tl = torch.tensor(prefix, device="cuda")
    s = fp32_row_sum(part).astype(np.float32)
    score = torch.tensor(s, device="cuda")
    hist = np.zeros((B, vsd.HIST_BINS), np.uint32)
    for b in range(B):
        hist[b] = np.bincount(_keys(s[b, :prefix[b]]) >> 20, minlength=vsd.HIST_BINS)
    th = torch.tensor(hist.view(np.int32), device="cuda")
    for k, ns, nr in [(2048, 16, 256), (512, 0, 0), (64, 4, 60), (1, 0, 0), (9000, 100, 900)]:
        i1, n1 = vsd.vsd_select_topk(tp, tl, k=k, n_sink=ns, n_recent=nr)[:2]
        i2, n2 = vsd.vsd_select_topk_scored(score, th, tl, k=k, n_sink=ns, n_recent=nr)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert torch.equal(i1, i2) and torch.equal(n1, n2), (k, ns, nr)


def test_fused_path_end_to_end():
    """verify (scored) -> select (scored) selects what verify -> select selects, with the
    histogram of the candidates (the verification told the protected budget) and with
    the histogram of every prefix position (the selection takes the protected ones out)."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import QWEN3_8B_32K as w
    vsd = _vsd()
    batch = make_batch(w, "cuda")
    i1 = n1 = None
    for ns, nr in ((w.n_sink, w.n_recent), (0, 0)):
        _, _, partial, score, hist = vsd.vsd_verify_attn_collect_scored(
            batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
            P_max=w.P_max, scale=w.scale, n_sink=ns, n_recent=nr)
        if i1 is None:
            i1, n1 = vsd.vsd_select_topk(partial, batch.prefix_len, k=w.k, n_sink=w.n_sink,
                                         n_recent=w.n_recent)[:2]
        i2, n2 = vsd.vsd_select_topk_scored(score, hist, batch.prefix_len, k=w.k,
                                            n_sink=w.n_sink, n_recent=w.n_recent)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert torch.equal(i1, i2) and torch.equal(n1, n2), (ns, nr)


@pytest.mark.parametrize("ns,nr", [(4, 32), (0, 100), (7000, 0), (16, 9000)])
def test_candidate_histogram(ns, nr):
    """With a protected budget the verification counts only the selection's candidates
    [min(n_sink, P), max(P - n_recent, that)): an exact bincount of those keys, and the
    scored selection from it equals the oracle's, on ragged prefixes (one shorter than
    the sinks, one covered by the recent window)."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    prefix = (6001, 0, 1, 511, 40000)
    w = Workload("cand", B=len(prefix), P=max(prefix), Hq=32, Hkv=8, d=128, gamma=4, k=10000,
                 n_sink=ns, n_recent=nr, planted_frac=0.01, seed=83, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    score = torch.zeros((w.B, w.P_max), dtype=torch.float32, device="cuda")  # past P_b: 0
    _, _, _, score, hist = vsd.vsd_verify_attn_collect_scored(
        batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.prefix_len,
        P_max=w.P_max, scale=w.scale, score=score, n_sink=ns, n_recent=nr)
    idx, n_sel = vsd.vsd_select_topk_scored(score, hist, batch.prefix_len, k=w.k, n_sink=ns,
                                            n_recent=nr)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    sc = score.cpu().numpy()
    hs = hist.cpu().numpy().view(np.uint32)
    for b, P in enumerate(prefix):
        lo = min(ns, P)
        hi = max(P - nr, lo)
        np.testing.assert_array_equal(hs[b], np.bincount(_keys(sc[b, lo:hi]) >> 20,
                                                         minlength=vsd.HIST_BINS))
    want_i, want_n = oracle.select(sc, np.array(prefix, np.int32), k=w.k, n_sink=ns, n_recent=nr)
    np.testing.assert_array_equal(n_sel.cpu().numpy(), want_n)
    np.testing.assert_array_equal(idx.cpu().numpy(), want_i)


def test_scored_select_flags_a_foreign_histogram():
    vsd = _vsd()
    score = torch.randn((1, 5000), device="cuda")
    tl = torch.tensor([5000], dtype=torch.int32, device="cuda")
    zero = torch.zeros((1, vsd.HIST_BINS), dtype=torch.int32, device="cuda")
    idx, n_sel = vsd.vsd_select_topk_scored(score, zero, tl, k=100, n_sink=4, n_recent=8)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_LENGTH
    assert int(n_sel[0]) == 100  # the selection itself is unspecified


@pytest.mark.parametrize("P_max,prefix,k,ns,nr,ties", [
    (5000, (5000, 4999, 17, 0, 300), 512, 4, 64, True),        # 8K slices, one CTA a row
    (12001, (12001, 9000, 12000), 1024, 16, 256, False),       # 16K slices, P_max % 4 != 0
    (32768, (32768, 32767, 2049), 2048, 16, 256, True),        # one full 32K slice
    (70001, (70001, 65536, 32769, 100), 4096, 16, 256, True),  # 3-CTA clusters
    (131072, (131072,), 8192, 16, 512, False),                 # 4-CTA cluster
    (300000, (300000, 200001), 8192, 4, 64, True),             # 10-CTA clusters (beyond 8)
])
def test_scored_select_against_oracle(P_max, prefix, k, ns, nr, ties):
    """The scored selection at every slice size and cluster width, ragged prefixes,
    scores with many exact ties (small integers) or none, against the oracle's selection
    on the same fp32 scores: identical index rows."""
    vsd = _vsd()
    rng = np.random.default_rng(P_max)
    B = len(prefix)
    if ties:
        s = rng.integers(-20, 21, size=(B, P_max)).astype(np.float32)
    else:
        s = rng.normal(size=(B, P_max)).astype(np.float32)
    pl = np.array(prefix, np.int32)
    hist = np.zeros((B, vsd.HIST_BINS), np.uint32)
    for b in range(B):
        hist[b] = np.bincount(_keys(s[b, :pl[b]]) >> 20, minlength=vsd.HIST_BINS)
    score = torch.tensor(s, device="cuda")
    idx, n_sel = vsd.vsd_select_topk_scored(score, torch.tensor(hist.view(np.int32), device="cuda"),
                                            torch.tensor(pl, device="cuda"), k=k, n_sink=ns,
                                            n_recent=nr)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    want_i, want_n = oracle.select(s, pl, k=k, n_sink=ns, n_recent=nr)
    np.testing.assert_array_equal(n_sel.cpu().numpy(), want_n)
    np.testing.assert_array_equal(idx.cpu().numpy(), want_i)


def test_scored_select_many_rows_and_a_bad_prefix():
    """144 rows of a 64K prefix (one launch of 2-CTA clusters, as a 36-layer loop selects);
    a row whose prefix length is past P_max is flagged and left empty."""
    vsd = _vsd()
    rng = np.random.default_rng(144)
    n_rows, P_max = 144, 65600
    pl = rng.integers(60000, P_max + 1, size=n_rows).astype(np.int32)
    s = rng.normal(size=(n_rows, P_max)).astype(np.float32)
    hist = np.zeros((n_rows, vsd.HIST_BINS), np.uint32)
    for b in range(n_rows):
        hist[b] = np.bincount(_keys(s[b, :pl[b]]) >> 20, minlength=vsd.HIST_BINS)
    score = torch.tensor(s, device="cuda")
    th = torch.tensor(hist.view(np.int32), device="cuda")
    idx, n_sel = vsd.vsd_select_topk_scored(score, th, torch.tensor(pl, device="cuda"), k=4096,
                                            n_sink=16, n_recent=256)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    want_i, want_n = oracle.select(s, pl, k=4096, n_sink=16, n_recent=256)
    np.testing.assert_array_equal(idx.cpu().numpy(), want_i)
    np.testing.assert_array_equal(n_sel.cpu().numpy(), want_n)
    bad = pl.copy()
    bad[3] = P_max + 1
    idx, n_sel = vsd.vsd_select_topk_scored(score, th, torch.tensor(bad, device="cuda"), k=4096,
                                            n_sink=16, n_recent=256)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_LENGTH
    assert int(n_sel[3]) == 0 and bool((idx[3] == -1).all())
    np.testing.assert_array_equal(idx.cpu().numpy()[4:], want_i[4:])


def test_scored_select_boundary_bin_held_by_one_slice():
    """A boundary bin of 3000 near-equal scores all in the first slice of a 32K row (more
    than that slice's share of the exchanged list): the other route to the cut, same
    rows as the oracle; and a bin of exactly equal scores there (ties by position)."""
    vsd = _vsd()
    rng = np.random.default_rng(77)
    P = 32768
    for equal in (False, True):
        s = rng.uniform(-4.0, 4.0, size=(1, P)).astype(np.float32)
        s[0, 16:3016] = 5.0 if equal else 5.0 + np.arange(3000, dtype=np.float32) * 1e-6
        pl = np.array([P], np.int32)
        hist = np.bincount(_keys(s[0]) >> 20, minlength=vsd.HIST_BINS).astype(np.uint32)[None]
        idx, n_sel = vsd.vsd_select_topk_scored(torch.tensor(s, device="cuda"),
                                                torch.tensor(hist.view(np.int32), device="cuda"),
                                                torch.tensor(pl, device="cuda"), k=2048,
                                                n_sink=16, n_recent=256)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        want_i, want_n = oracle.select(s, pl, k=2048, n_sink=16, n_recent=256)
        np.testing.assert_array_equal(idx.cpu().numpy(), want_i)
        np.testing.assert_array_equal(n_sel.cpu().numpy(), want_n)


@pytest.mark.parametrize("d,Hq,Hkv,gamma,prefix", [
    (128, 32, 8, 4, (6001, 0, 1, 511, 4096)),   # ragged; the block crosses a tile at 511
    (64, 8, 2, 3, (127, 30)),                   # head_dim 64; the block ends a tile
])
def test_scored_verify_stores_the_verify_block(d, Hq, Hkv, gamma, prefix):
    """The scored verification given the verify block's K/V stores them into the caches
    itself: the same caches, outputs, scores and histogram, bit for bit, as the append
    kernel followed by the call, in either dependency mode."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("vstore", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma,
                 k=64, n_sink=4, n_recent=16, planted_frac=0.01, seed=91, prefix_lens=prefix)
    batch = make_batch(w, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    kn = torch.randn((w.B, w.R, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn((w.B, w.R, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    kc_a, vc_a = batch.k_cache.clone(), batch.v_cache.clone()
    vsd.vsd_append_kv(kn, vn, kc_a, vc_a, batch.block_table, batch.prefix_len, pos_offset=0)
    ref = vsd.vsd_verify_attn_collect_scored(batch.q, kc_a, vc_a, batch.block_table,
                                             batch.prefix_len, P_max=w.P_max, scale=w.scale,
                                             n_sink=w.n_sink, n_recent=w.n_recent)
    torch.cuda.synchronize()
    for flags in (0, vsd.VERIFY_EARLY_PREFETCH):
        kc_b, vc_b = batch.k_cache.clone(), batch.v_cache.clone()
        got = vsd.vsd_verify_attn_collect_scored(batch.q, kc_b, vc_b, batch.block_table,
                                                 batch.prefix_len, P_max=w.P_max,
                                                 scale=w.scale, n_sink=w.n_sink,
                                                 n_recent=w.n_recent, flags=flags, k_new=kn,
                                                 v_new=vn)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert torch.equal(kc_b, kc_a) and torch.equal(vc_b, vc_a)
        assert torch.equal(got[0], ref[0])
        for b, P in enumerate(prefix):
            assert torch.equal(got[2][b, :, :P], ref[2][b, :, :P])
            assert torch.equal(got[3][b, :P], ref[3][b, :P])
        assert torch.equal(got[4], ref[4])
