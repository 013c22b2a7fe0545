"""GPU parity of the per-query block top-k (the sparse-verification summary's
attention sparsity: each query keeps its top-k pages by a cheap relevance score),
through the C ABI, against the fp64 oracle (comparison rules in parity_utils)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import REL_TOL, assert_rel_close

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


def _run(batch, w, kb, nblk_max=None):
    vsd = _vsd()
    nblk_max = nblk_max or vsd.page_blocks(w.P_max)
    means = vsd.vsd_page_key_means(batch.k_cache, batch.block_table, batch.prefix_len, B=w.B,
                                   page_blocks_max=nblk_max)
    scores, blocks = vsd.vsd_block_topk(batch.q, means, batch.prefix_len, kb=kb, scale=w.scale,
                                        k_cache=batch.k_cache, block_table=batch.block_table)
    torch.cuda.synchronize()
    return means, scores, blocks


def _check(batch, w, kb, nblk_max=None):
    """Scores against the fp64 oracle; the kept pages exactly against the oracle's
    selection fed the kernel's own fp32 scores (the decision in the kernel's precision),
    and under the index-set rule against the fp64 oracle end to end."""
    from sparse_attention_speculative_gb300.synth import host_arrays
    vsd = _vsd()
    means, scores, blocks = _run(batch, w, kb, nblk_max)
    assert vsd.vsd_read_device_status() == 0
    nblk_max = scores.shape[3]
    h = host_arrays(batch)
    s_ref, b_ref = oracle.block_topk(h["q"], h["k_cache"], h["block_table"], h["prefix_len"],
                                     kb=kb, scale=w.scale, page_blocks_max=nblk_max)
    sc = scores.cpu().numpy().astype(np.float64)
    got = blocks.cpu().numpy()
    B, R, Hq, _ = sc.shape
    nblk = [(int(P) + 15) // 16 for P in h["prefix_len"]]
    for b in range(B):
        assert_rel_close(sc[b, :, :, :nblk[b]], s_ref[b, :, :, :nblk[b]], "page scores")
    rows_nblk = np.repeat(np.array(nblk, np.int32), R * Hq)
    flat_sc = sc.reshape(B * R * Hq, nblk_max)
    flat_got = got.reshape(B * R * Hq, kb)
    want_idx, want_n = oracle.select(flat_sc, rows_nblk, k=kb, n_sink=0, n_recent=0)
    np.testing.assert_array_equal(flat_got, want_idx)
    # against the fp64 oracle: equal sets, or swaps within the tolerance of the k-th score
    flat_ref = b_ref.reshape(B * R * Hq, kb)
    flat_sref = s_ref.reshape(B * R * Hq, nblk_max)
    swaps = 0
    for r in range(B * R * Hq):
        n = min(kb, int(rows_nblk[r]))
        a, e = set(flat_got[r, :n].tolist()), set(flat_ref[r, :n].tolist())
        if a == e:
            continue
        kth = min(flat_sref[r, j] for j in e)
        for j in a ^ e:
            assert abs(flat_sref[r, j] - kth) <= REL_TOL * max(1.0, abs(kth)), (r, j)
        swaps += len(a ^ e) // 2
    return means, scores, blocks, swaps


@pytest.mark.parametrize("d,Hq,Hkv,gamma,prefix,kb", [
    (128, 32, 8, 4, (6000, 1500, 17, 0), 64),    # Qwen3-8B geometry, ragged, an empty prefix
    (128, 64, 8, 5, (4096, 2049), 32),           # Qwen2.5-72B geometry (R * G = 48)
    (64, 8, 2, 3, (777, 31), 8),                 # head_dim 64; a prefix with fewer pages than kb
    (128, 32, 8, 7, (32768,), 128),              # a full 32K prefix, R * G = 32
])
def test_block_topk(d, Hq, Hkv, gamma, prefix, kb):
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("btk", B=len(prefix), P=max(prefix), Hq=Hq, Hkv=Hkv, d=d, gamma=gamma, k=kb,
                 n_sink=0, n_recent=0, planted_frac=0.01, seed=71, prefix_lens=prefix)
    _check(make_batch(w, "cuda"), w, kb)


def test_block_topk_maximum_pages():
    """16384 pages (a 262144-token prefix, the largest supported), one KV head."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("btk_max", B=2, P=262144, Hq=2, Hkv=1, d=64, gamma=1, k=1000, n_sink=0,
                 n_recent=0, planted_frac=0.001, seed=72, prefix_lens=(262144, 262131))
    _check(make_batch(w, "cuda"), w, 1000)


def test_block_topk_ties_and_padding():
    """All keys equal: every page of a row scores the same, the lowest kb pages are kept;
    a row with fewer pages than kb is padded with -1."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("btk_tie", B=2, P=5000, Hq=8, Hkv=2, d=128, gamma=2, k=16, n_sink=0,
                 n_recent=0, seed=73, prefix_lens=(5000, 100))
    batch = make_batch(w, "cuda")
    batch.k_cache.copy_(batch.k_cache[:1, :, :1, :].expand_as(batch.k_cache))
    _, scores, blocks = _run(batch, w, 16)
    assert vsd.vsd_read_device_status() == 0
    got = blocks.cpu().numpy()
    assert np.all(got[0] == np.arange(16))
    assert np.all(got[1, :, :, :7] == np.arange(7))
    assert np.all(got[1, :, :, 7:] == -1)


def test_page_means_incremental_and_bad_block():
    """page_begin refreshes only the pages from it on (the others keep their contents,
    bit for bit equal to a full pass where rewritten); a bad block-table entry is
    flagged and its page written as zeros."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    vsd = _vsd()
    w = Workload("btk_inc", B=3, P=3000, Hq=16, Hkv=4, d=64, gamma=3, k=8, n_sink=0,
                 n_recent=0, seed=74, prefix_lens=(3000, 1234, 40))
    batch = make_batch(w, "cuda")
    nblk_max = vsd.page_blocks(w.P_max)
    full = vsd.vsd_page_key_means(batch.k_cache, batch.block_table, batch.prefix_len, B=w.B,
                                  page_blocks_max=nblk_max)
    first = torch.tensor([150, 0, 2], dtype=torch.int32, device="cuda")
    part = torch.full_like(full, 7.0)
    vsd.vsd_page_key_means(batch.k_cache, batch.block_table, batch.prefix_len, B=w.B,
                           page_blocks_max=nblk_max, page_begin=first, page_means=part)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    for b, P in enumerate([3000, 1234, 40]):
        nb, f = (P + 15) // 16, int(first[b])
        assert torch.equal(part[b, :, f:nb], full[b, :, f:nb])
        assert bool((part[b, :, :f] == 7.0).all()) and bool((part[b, :, nb:] == 7.0).all())
    bt = batch.block_table.clone()
    bt[1, 3] = -5
    bad = vsd.vsd_page_key_means(batch.k_cache, bt, batch.prefix_len, B=w.B,
                                 page_blocks_max=nblk_max)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_BLOCK
    assert bool((bad[1, :, 3] == 0).all())
    assert torch.equal(bad[0], full[0]) and torch.equal(bad[1, :, 4:], full[1, :, 4:])


@pytest.mark.parametrize("B,Hq,Hkv", [(2, 4, 2), (3, 64, 2)])  # 16 rows / 384 rows
@pytest.mark.parametrize("nblk_max", [4096, 2048])
@pytest.mark.parametrize("kind", ["outlier", "duplicates", "spread", "two_values"])
def test_block_topk_selection_paths(kind, nblk_max, B, Hq, Hkv):
    """Page means written directly, to drive each path of the selection: an outlier page
    (every other page in one value bucket: the exact-key radix), integer duplicates
    (buckets of equal keys: ties to the lower page), a smooth spread (few candidates
    ranked directly), two values.  Exact against the oracle's selection fed the
    kernel's fp32 scores."""
    vsd = _vsd()
    rng = np.random.default_rng(["outlier", "duplicates", "spread", "two_values"].index(kind))
    R, d, kb = 2, 64, 300
    prefix = np.array([nblk_max * 16, (nblk_max * 3 // 4) * 16 - 5, nblk_max * 8][:B], np.int32)
    means = np.zeros((B, Hkv, nblk_max, d), np.float32)
    if kind == "outlier":
        means[..., 0] = rng.normal(size=(B, Hkv, nblk_max)) * 1e-3
        means[:, :, 77, 0] = 1e4
    elif kind == "duplicates":
        means[..., 0] = rng.integers(-3, 4, size=(B, Hkv, nblk_max))
    elif kind == "spread":
        means[..., 0] = rng.normal(size=(B, Hkv, nblk_max))
    else:
        means[..., 0] = np.where(rng.random((B, Hkv, nblk_max)) < 0.5, 1.0, -1.0)
    q = np.zeros((B, R, Hq, d), np.float32)
    q[..., 0] = 1.0
    q[:, 1, :, 0] = -1.0  # row 1 ranks the pages in reverse
    tq = torch.tensor(q, device="cuda").to(torch.bfloat16)
    tm = torch.tensor(means, device="cuda")
    tp = torch.tensor(prefix, device="cuda")
    scores, blocks = vsd.vsd_block_topk(tq, tm, tp, kb=kb, scale=0.5)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    sc = scores.cpu().numpy().astype(np.float64).reshape(B * R * Hq, nblk_max)
    nblk = np.repeat((prefix + 15) // 16, R * Hq).astype(np.int32)
    want, _ = oracle.select(sc, nblk, k=kb, n_sink=0, n_recent=0)
    np.testing.assert_array_equal(blocks.cpu().numpy().reshape(B * R * Hq, kb), want)
