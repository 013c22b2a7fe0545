"""The seeded synthetic input recipe, checked on the host: paging through a permuted
block table, planted heavy hitters (positions and the boost along the group's query
direction), bursts, determinism, and the cache append used by the decode loops."""
import math

import numpy as np
import torch

from sparse_attention_speculative_gb300.synth import make_batch, seeded_bf16, write_tokens
from sparse_attention_speculative_gb300.workloads import TINY, Workload


def _workload(**kw):
    base = dict(B=3, P=700, Hq=8, Hkv=2, d=64, gamma=3, k=64, n_sink=4, n_recent=16,
                planted_frac=0.02, seed=7, prefix_lens=(700, 333, 0))
    base.update(kw)
    return Workload("inputs", **base)


def _key_row(batch, b, j, g):
    """K row of sequence b, token j, KV head g, read through the block table."""
    page = batch.k_cache.shape[2]
    blk = int(batch.block_table[b, j // page])
    return batch.k_cache[blk, g, j % page].float()


def test_block_table_is_a_permutation_of_the_pages():
    w = _workload()
    batch = make_batch(w, "cpu")
    bt = batch.block_table.numpy()
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(batch.num_blocks))
    for b, P in enumerate(w.prefix()):
        n = math.ceil(w.capacity(P) / w.page)
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, n:] == -1)
    # a shuffled table: not the identity
    assert not np.array_equal(used, np.arange(batch.num_blocks))


def test_contiguous_workload_uses_the_identity_table():
    batch = make_batch(TINY, "cpu")
    n = math.ceil(TINY.capacity(TINY.P) / TINY.page)
    assert np.array_equal(batch.block_table[0, :n].numpy(), np.arange(n))


def test_planted_positions_and_their_boost():
    w = _workload()
    batch = make_batch(w, "cpu")
    d, R, Hkv = w.d, w.R, w.Hkv
    G = w.Hq // Hkv
    for b, P in enumerate(w.prefix()):
        pos = batch.planted[b].numpy()
        assert len(pos) == int(round(w.planted_frac * P))
        assert np.all(np.diff(pos) > 0) and (len(pos) == 0 or (pos[0] >= 0 and pos[-1] < P))
        if len(pos) == 0:
            continue
        # the boost: 3 sqrt(d) along the unit sum of the group's verify query rows
        q = batch.q[b].float().reshape(R, Hkv, G, d).sum(dim=(0, 2))
        u = q / q.norm(dim=-1, keepdim=True)
        planted = set(pos.tolist())
        for g in range(Hkv):
            proj_p = [float(_key_row(batch, b, int(j), g) @ u[g]) for j in pos]
            others = [j for j in range(P) if j not in planted][:200]
            proj_o = [float(_key_row(batch, b, j, g) @ u[g]) for j in others]
            # background keys ~ N(0, 1) along a unit direction; planted ones shifted by
            # 3 sqrt(d) (bf16 rounding of the boosted rows moves them by well under 1)
            assert min(proj_p) > 3 * math.sqrt(d) - 5.0
            assert max(abs(x) for x in proj_o) < 5.0


def test_bursts_are_runs_of_consecutive_positions():
    w = _workload(B=1, P=2000, prefix_lens=(2000,), planted_frac=0.0, bursts=3, burst_len=64)
    pos = make_batch(w, "cpu").planted[0].numpy()
    runs = np.split(pos, np.where(np.diff(pos) != 1)[0] + 1)
    assert 1 <= len(runs) <= 3
    assert sum(len(r) for r in runs) <= 3 * 64 and len(pos) >= 64
    assert pos[0] >= 0 and pos[-1] < 2000


def test_seeded_inputs_are_deterministic_per_layer():
    w = _workload()
    a, b = make_batch(w, "cpu"), make_batch(w, "cpu")
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache),
                 (a.block_table, b.block_table), (a.q_draft, b.q_draft)):
        assert torch.equal(x, y)
    c = make_batch(w, "cpu", layer=1)
    assert not torch.equal(a.k_cache, c.k_cache) and not torch.equal(a.q, c.q)


def test_write_tokens_goes_through_the_block_table():
    w = _workload()
    batch = make_batch(w, "cpu")
    b, P = 1, w.prefix()[1]
    pos = torch.arange(P, P + 3)
    k_rows = seeded_bf16((3, w.Hkv, w.d), 11, "cpu")
    v_rows = seeded_bf16((3, w.Hkv, w.d), 12, "cpu")
    before = batch.k_cache.clone()
    write_tokens(batch, b, pos, k_rows, v_rows)
    page = batch.k_cache.shape[2]
    for i, j in enumerate(pos.tolist()):
        blk = int(batch.block_table[b, j // page])
        assert torch.equal(batch.k_cache[blk, :, j % page], k_rows[i])
        assert torch.equal(batch.v_cache[blk, :, j % page], v_rows[i])
    # nothing else changed
    changed = (batch.k_cache != before).any(dim=-1).nonzero().tolist()
    assert len(changed) <= 3 * w.Hkv
