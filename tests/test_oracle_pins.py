"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test feeds the oracle an input whose answer is known without the oracle:
brute-force enumeration, closed forms on structured inputs, special cases that
reduce to a textbook result, and invariants.  Together they are meant to fail on a
dropped scale, a wrong sign, a wrong GQA mapping, a transposed operand, an
off-by-one in the causal window or the tail, a wrong collected row, or a wrong tie
rule.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.helpers import (bf16_bits, bf16_round_bits, bits_to_float, make_table,
                           paged_cache)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------
# selection: Vegas sec. 2.A (argmax of summed logits over |T| = k) with the Dustin
# protected budget (sinks + recent window kept first)
# --------------------------------------------------------------------------------------

def _protected(P, n_sink, n_recent):
    return set(range(min(n_sink, P))) | set(range(max(0, P - n_recent), P))


def _bruteforce(scores, P, k, n_sink, n_recent):
    """All k-subsets of the prefix that contain the protected set; maximise the
    summed score (exact: integer scores); among maximisers take the lexicographically
    smallest sorted tuple (= lower positions win ties)."""
    S = _protected(P, n_sink, n_recent)
    n = min(k, P)
    free = [j for j in range(P) if j not in S]
    best, best_set = None, None
    for extra in itertools.combinations(free, n - len(S)):
        T = tuple(sorted(S | set(extra)))
        total = sum(int(scores[j]) for j in T)
        if best is None or total > best or (total == best and T < best_set):
            best, best_set = total, T
    return list(best_set)


@pytest.mark.parametrize("ties", [False, True])
def test_select_matches_bruteforce(ties):
    rng = np.random.default_rng(11 if ties else 7)
    for trial in range(60):
        P = int(rng.integers(1, 15))
        n_sink = int(rng.integers(0, 4))
        n_recent = int(rng.integers(0, 5))
        k = int(rng.integers(n_sink + n_recent, n_sink + n_recent + 8))
        if ties:
            scores = rng.integers(-2, 3, size=P).astype(np.float64)
        else:
            scores = rng.permutation(np.arange(-50, 50))[:P].astype(np.float64)
        P_max = P + int(rng.integers(0, 3))
        padded = np.full((1, P_max), 99.0)  # beyond P: must be ignored
        padded[0, :P] = scores
        idx, n_sel = oracle.select(padded, [P], k=k, n_sink=n_sink, n_recent=n_recent)
        want = _bruteforce(scores, P, k, n_sink, n_recent)
        assert n_sel[0] == len(want)
        assert idx[0, :n_sel[0]].tolist() == want, (trial, P, k, n_sink, n_recent, scores)


def test_select_streaming_golden():
    with open(os.path.join(GOLDEN, "select_streaming.json")) as f:
        cases = json.load(f)["cases"]
    rng = np.random.default_rng(3)
    for c in cases:
        P = c["P"]
        # scores that favour the unprotected middle as strongly as possible
        s = rng.normal(size=(1, P)) + 100.0 * (np.arange(P) % 2)
        idx, n_sel = oracle.select(s, [P], k=c["k"], n_sink=c["n_sink"], n_recent=c["n_recent"])
        assert idx[0, :n_sel[0]].tolist() == c["expected"]


def test_select_invariants_large():
    rng = np.random.default_rng(5)
    P_max = 3000
    prefix = [3000, 1, 0, 17, 2500, 300]
    score = rng.normal(size=(len(prefix), P_max))
    for k, ns, nr in [(64, 4, 16), (300, 16, 256), (20, 4, 16), (5000, 16, 256)]:
        idx, n_sel = oracle.select(score, prefix, k=k, n_sink=ns, n_recent=nr)
        for r, P in enumerate(prefix):
            n = min(k, P)
            assert n_sel[r] == n
            sel = idx[r, :n]
            assert np.all(np.diff(sel) > 0) and (n == 0 or (sel[0] >= 0 and sel[-1] < P))
            assert _protected(P, ns, nr) <= set(sel.tolist())
            if k >= P:
                assert sel.tolist() == list(range(P))
            else:
                # every unselected unprotected position scores no higher than every
                # selected unprotected one
                S = _protected(P, ns, nr)
                chosen = [j for j in sel.tolist() if j not in S]
                rest = [j for j in range(P) if j not in S and j not in set(sel.tolist())]
                if chosen and rest:
                    assert min(score[r, chosen]) >= max(score[r, rest])


def test_select_rejects_budget_below_protected():
    with pytest.raises(oracle.OracleError):
        oracle.select(np.zeros((1, 10)), [10], k=5, n_sink=4, n_recent=2)


# --------------------------------------------------------------------------------------
# verification attention + Collect-2-Query (Vegas sec. 2 verification phase, sec. 2.B,
# sec. 3 kernel instrumentation)
# --------------------------------------------------------------------------------------

def _structured_verify(B=2, prefix=(37, 50), Hq=8, Hkv=2, d=64, R=3, page=16, seed=1):
    G = Hq // Hkv
    lengths = [p + R for p in prefix]
    table, NB = make_table(lengths, page, shuffle_seed=seed)
    q = np.zeros((B, R, Hq, d), np.float32)
    for b in range(B):
        for t in range(R):
            for h in range(Hq):
                q[b, t, h, 0] = t + 1
                q[b, t, h, 1] = h + 1
                q[b, t, h, 2] = b + 1
    Ks, Vs = [], []
    rng = np.random.default_rng(seed)
    for b in range(B):
        K = np.zeros((lengths[b], Hkv, d), np.float32)
        for j in range(lengths[b]):
            for g in range(Hkv):
                K[j, g, 0] = (j % 7) - 3
                K[j, g, 1] = g + 1
                K[j, g, 2] = 1
        Ks.append(K)
        Vs.append(bits_to_float(bf16_round_bits(rng.normal(size=(lengths[b], Hkv, d))))
                  .astype(np.float32))
    kc = paged_cache(Ks, table, NB, page)
    vc = paged_cache(Vs, table, NB, page)
    return dict(q=bf16_bits(q), k=kc, v=vc, table=table, prefix=np.array(prefix, np.int32),
                G=G, R=R, Hq=Hq, Hkv=Hkv, d=d)


def test_verify_logits_closed_form():
    s = _structured_verify()
    scale = 1.0 / math.sqrt(s["d"])
    P_max = 64
    out, logits, partial = oracle.verify(s["q"], s["k"], s["v"], s["table"], s["prefix"],
                                         scale=scale, P_max=P_max)
    R, Hq, G, Hkv = s["R"], s["Hq"], s["G"], s["Hkv"]
    rows = (0, R - 1)
    for b, P in enumerate(s["prefix"]):
        j = np.arange(P)
        for c, t in enumerate(rows):
            for h in range(Hq):
                want = scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (h // G + 1) + (b + 1))
                np.testing.assert_allclose(logits[b, c, h, :P], want, rtol=0, atol=1e-12)
            assert np.all(logits[b, :, :, P:] == 0)
        for g in range(Hkv):
            want = np.zeros(P)
            for t in rows:
                for h in range(g * G, (g + 1) * G):
                    want += scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (g + 1) + (b + 1))
            np.testing.assert_allclose(partial[b, g, :P], want, rtol=0, atol=1e-10)
        score = oracle.score_from_logits(logits, s["prefix"])
        want_s = np.zeros(P)
        for t in rows:
            for h in range(Hq):
                want_s += scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (h // G + 1) + (b + 1))
        np.testing.assert_allclose(score[b, :P], want_s, rtol=0, atol=1e-9)
        np.testing.assert_allclose(oracle.score_from_partials(partial, s["prefix"])[b, :P],
                                   want_s, rtol=0, atol=1e-9)


def test_verify_all_rows_closed_form():
    """Every verify row collected (the selection equation summed over all gamma+1 rows):
    each row's logits and the per-group sum over all rows against the closed form."""
    s = _structured_verify(R=4)
    scale = 1.0 / math.sqrt(s["d"])
    P_max = 64
    out, logits, partial = oracle.verify_all_rows(s["q"], s["k"], s["v"], s["table"],
                                                  s["prefix"], scale=scale, P_max=P_max)
    R, Hq, G, Hkv = s["R"], s["Hq"], s["G"], s["Hkv"]
    assert logits.shape == (2, R, Hq, P_max)
    for b, P in enumerate(s["prefix"]):
        j = np.arange(P)
        for t in range(R):
            for h in range(Hq):
                want = scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (h // G + 1) + (b + 1))
                np.testing.assert_allclose(logits[b, t, h, :P], want, rtol=0, atol=1e-12)
        assert np.all(logits[b, :, :, P:] == 0)
        for g in range(Hkv):
            want = np.zeros(P)
            for t in range(R):
                for h in range(g * G, (g + 1) * G):
                    want += scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (g + 1) + (b + 1))
            np.testing.assert_allclose(partial[b, g, :P], want, rtol=0, atol=1e-10)
    # the attention output does not depend on what is collected
    out2, _, _ = oracle.verify(s["q"], s["k"], s["v"], s["table"], s["prefix"], scale=scale,
                               P_max=P_max)
    np.testing.assert_array_equal(out, out2)


def test_verify_collects_requested_rows():
    s = _structured_verify(R=4)
    scale = 1.0 / math.sqrt(s["d"])
    _, logits, _ = oracle.verify(s["q"], s["k"], s["v"], s["table"], s["prefix"], scale=scale,
                                 P_max=64, row0=1, row1=2)
    G = s["G"]
    for b, P in enumerate(s["prefix"]):
        j = np.arange(P)
        for c, t in enumerate((1, 2)):
            for h in range(s["Hq"]):
                want = scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (h // G + 1) + (b + 1))
                np.testing.assert_allclose(logits[b, c, h, :P], want, atol=1e-12)


def test_verify_causal_uniform_mean():
    """Equal keys give uniform attention; with V_j = (j, g) the output of verify row t
    is the mean of 0..P_b+t, i.e. (P_b + t) / 2, which pins the causal window."""
    B, Hq, Hkv, d, R, page = 3, 4, 2, 64, 5, 16
    prefix = [0, 21, 130]
    lengths = [p + R for p in prefix]
    table, NB = make_table(lengths, page, shuffle_seed=4)
    rng = np.random.default_rng(0)
    q = bf16_round_bits(rng.normal(size=(B, R, Hq, d)))
    Ks = [np.zeros((L, Hkv, d), np.float32) for L in lengths]
    Vs = []
    for L in lengths:
        V = np.zeros((L, Hkv, d), np.float32)
        V[:, :, 0] = np.arange(L)[:, None]
        V[:, :, 1] = np.arange(Hkv)[None, :]
        Vs.append(V)
    out, _, _ = oracle.verify(q, paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page),
                              table, prefix, scale=0.125, P_max=max(prefix))
    for b, P in enumerate(prefix):
        for t in range(R):
            for h in range(Hq):
                assert out[b, t, h, 0] == pytest.approx((P + t) / 2.0, abs=1e-12)
                assert out[b, t, h, 1] == pytest.approx(h // (Hq // Hkv), abs=1e-12)


def test_verify_two_key_softmax_scale():
    """Prefix of one token, row 0 sees keys {0, 1}: z0 = scale * 4 * 2, z1 = 0, so
    o = sigmoid(z0) v0 + (1 - sigmoid(z0)) v1 (pins the scale factor)."""
    d, page = 64, 16
    table, NB = make_table([3], page)
    q = np.zeros((1, 2, 1, d), np.float32)
    q[0, :, 0, 0] = 4.0
    K = np.zeros((3, 1, d), np.float32)
    K[0, 0, 0] = 2.0
    V = np.zeros((3, 1, d), np.float32)
    V[0, 0, 0], V[1, 0, 0], V[2, 0, 0] = 1.0, -3.0, 5.0
    out, _, _ = oracle.verify(bf16_bits(q), paged_cache([K], table, NB, page),
                              paged_cache([V], table, NB, page), table, [1], scale=0.125,
                              P_max=1)
    z0 = 0.125 * 8.0
    sig = 1.0 / (1.0 + math.exp(-z0))
    assert out[0, 0, 0, 0] == pytest.approx(sig * 1.0 + (1 - sig) * -3.0, abs=1e-12)
    w = np.array([math.exp(z0), 1.0, 1.0])
    assert out[0, 1, 0, 0] == pytest.approx((w @ np.array([1.0, -3.0, 5.0])) / w.sum(), abs=1e-12)


def test_verify_one_hot_key_reproduces_value_row():
    d, page, P, R = 64, 16, 48, 2
    table, NB = make_table([P + R], page, shuffle_seed=9)
    K = np.zeros((P + R, 1, d), np.float32)
    for j in range(P + R):
        K[j, 0, j % d] = 1.0
    rng = np.random.default_rng(1)
    V = bits_to_float(bf16_round_bits(rng.normal(size=(P + R, 1, d)))).astype(np.float32)
    jstar = 29
    q = np.zeros((1, R, 1, d), np.float32)
    q[0, :, 0, jstar] = 200.0
    out, _, _ = oracle.verify(bf16_bits(q), paged_cache([K], table, NB, page),
                              paged_cache([V], table, NB, page), table, [P], scale=0.125, P_max=P)
    for t in range(R):
        np.testing.assert_allclose(out[0, t, 0], V[jstar, 0], atol=1e-8)


def test_verify_single_key_is_value_row():
    d, page = 64, 16
    table, NB = make_table([1], page)
    rng = np.random.default_rng(2)
    K = bits_to_float(bf16_round_bits(rng.normal(size=(1, 2, d)))).astype(np.float32)
    V = bits_to_float(bf16_round_bits(rng.normal(size=(1, 2, d)))).astype(np.float32)
    q = bf16_round_bits(rng.normal(size=(1, 1, 4, d)))
    out, _, _ = oracle.verify(q, paged_cache([K], table, NB, page), paged_cache([V], table, NB, page),
                              table, [0], scale=0.125, P_max=1, collect=False)
    for h in range(4):
        np.testing.assert_allclose(out[0, 0, h], V[0, h // 2], atol=0)


def test_verify_block_table_permutation_invariance():
    rng = np.random.default_rng(8)
    d, page, R, Hq, Hkv = 64, 16, 3, 4, 2
    prefix = [70, 33]
    lengths = [p + R for p in prefix]
    Ks = [bits_to_float(bf16_round_bits(rng.normal(size=(L, Hkv, d)))).astype(np.float32)
          for L in lengths]
    Vs = [bits_to_float(bf16_round_bits(rng.normal(size=(L, Hkv, d)))).astype(np.float32)
          for L in lengths]
    q = bf16_round_bits(rng.normal(size=(2, R, Hq, d)))
    results = []
    for seed in (None, 1, 2):
        table, NB = make_table(lengths, page, shuffle_seed=seed, extra_blocks=2)
        results.append(oracle.verify(q, paged_cache(Ks, table, NB, page, fill=7.0),
                                     paged_cache(Vs, table, NB, page, fill=-7.0), table, prefix,
                                     scale=0.125, P_max=80))
    for other in results[1:]:
        for a, b in zip(results[0], other):
            np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------------------
# sparse draft attention (Vegas sec. 2 drafting phase; sec. 3 page-size-1 paged attention
# over the selected indices)
# --------------------------------------------------------------------------------------

def _random_paged(rng, lengths, Hkv, d, page, seed):
    table, NB = make_table(lengths, page, shuffle_seed=seed)
    Ks = [bits_to_float(bf16_round_bits(rng.normal(size=(L, Hkv, d)))).astype(np.float32)
          for L in lengths]
    Vs = [bits_to_float(bf16_round_bits(rng.normal(size=(L, Hkv, d)))).astype(np.float32)
          for L in lengths]
    return table, NB, Ks, Vs


def test_sparse_with_all_indices_equals_full_attention():
    rng = np.random.default_rng(21)
    B, Hq, Hkv, d, R, page = 2, 8, 2, 64, 4, 16
    prefix = [90, 45]
    lengths = [p + R for p in prefix]
    table, NB, Ks, Vs = _random_paged(rng, lengths, Hkv, d, page, 3)
    kc, vc = paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page)
    q = bf16_round_bits(rng.normal(size=(B, R, Hq, d)))
    full, _, _ = oracle.verify(q, kc, vc, table, prefix, scale=0.125, P_max=90, collect=False)
    k_max = max(prefix)
    idx = np.zeros((B, k_max), np.int32)
    for b, P in enumerate(prefix):
        idx[b, :P] = np.arange(P)
    for t in range(R):
        out = oracle.sparse_decode(np.ascontiguousarray(q[:, t]), kc, vc, table, idx, prefix,
                                   prefix, [P + t + 1 for P in prefix], scale=0.125)
        np.testing.assert_allclose(out, full[:, t], rtol=0, atol=1e-12)


def test_sparse_uniform_mean_of_attended_positions():
    """Equal keys: the output is the mean of V over exactly idx[:n_sel] and the tail."""
    B, Hq, Hkv, d, page = 2, 4, 1, 64, 16
    lengths = [60, 40]
    table, NB = make_table(lengths, page, shuffle_seed=6)
    Ks = [np.zeros((L, Hkv, d), np.float32) for L in lengths]
    Vs = []
    for L in lengths:
        V = np.zeros((L, Hkv, d), np.float32)
        V[:, 0, 0] = np.arange(L)
        V[:, 0, 1] = np.arange(L) % 3
        Vs.append(V)
    idx = np.array([[0, 3, 17, 31, 44, -5], [2, 9, 11, -5, -5, -5]], np.int32)
    n_sel = [5, 3]
    tail_start = [50, 30]
    seq_len = [57, 30]
    rng = np.random.default_rng(0)
    q = bf16_round_bits(rng.normal(size=(B, Hq, d)))
    out = oracle.sparse_decode(q, paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page),
                               table, idx, n_sel, tail_start, seq_len, scale=0.125)
    for b in range(B):
        pos = list(idx[b, :n_sel[b]]) + list(range(tail_start[b], seq_len[b]))
        for h in range(Hq):
            assert out[b, h, 0] == pytest.approx(np.mean(pos), abs=1e-12)
            assert out[b, h, 1] == pytest.approx(np.mean(np.array(pos) % 3), abs=1e-12)


def test_sparse_verify_uniform_mean_over_selection_and_block():
    """Equal keys: verify row t averages V over exactly idx[:n_sel] and the verify
    block positions P .. P + t (Dustin's compressed cache, causal in the block)."""
    B, Hq, Hkv, d, page, R = 2, 4, 2, 64, 16, 3
    prefix = [50, 33]
    lengths = [p + R for p in prefix]
    table, NB = make_table(lengths, page, shuffle_seed=8)
    Ks = [np.zeros((L, Hkv, d), np.float32) for L in lengths]
    Vs = []
    for L in lengths:
        V = np.zeros((L, Hkv, d), np.float32)
        V[:, :, 0] = np.arange(L)[:, None]
        V[:, :, 1] = (np.arange(L) % 5)[:, None]
        Vs.append(V)
    idx = np.array([[0, 1, 7, 30, 49, -3], [4, 19, 32, -3, -3, -3]], np.int32)
    n_sel = [5, 3]
    rng = np.random.default_rng(1)
    q = bf16_round_bits(rng.normal(size=(B, R, Hq, d)))
    out = oracle.sparse_verify(q, paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page),
                               table, prefix, idx, n_sel, scale=0.125)
    for b in range(B):
        for t in range(R):
            pos = list(idx[b, :n_sel[b]]) + list(range(prefix[b], prefix[b] + t + 1))
            for h in range(Hq):
                assert out[b, t, h, 0] == pytest.approx(np.mean(pos), abs=1e-12)
                assert out[b, t, h, 1] == pytest.approx(np.mean(np.array(pos) % 5), abs=1e-12)


def test_sparse_verify_with_the_whole_prefix_is_full_verification():
    """Selecting every prefix position turns sparse verification into the full one."""
    s = _structured_verify(R=3)
    scale = 1.0 / math.sqrt(s["d"])
    out_full, _, _ = oracle.verify(s["q"], s["k"], s["v"], s["table"], s["prefix"], scale=scale,
                                   P_max=64, collect=False)
    k_max = int(max(s["prefix"]))
    idx = np.full((len(s["prefix"]), k_max), -1, np.int32)
    for b, P in enumerate(s["prefix"]):
        idx[b, :P] = np.arange(P)
    out = oracle.sparse_verify(s["q"], s["k"], s["v"], s["table"], s["prefix"], idx,
                               s["prefix"], scale=scale)
    np.testing.assert_allclose(out, out_full, rtol=0, atol=1e-12)


def test_sparse_single_position_is_value_row():
    rng = np.random.default_rng(4)
    d, page = 128, 16
    table, NB, Ks, Vs = _random_paged(rng, [20], 2, d, page, 1)
    q = bf16_round_bits(rng.normal(size=(1, 4, d)))
    out = oracle.sparse_decode(q, paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page),
                               table, np.zeros((1, 4), np.int32), [0], [0], [1], scale=0.088)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], Vs[0][0, h // 2], atol=0)
    out = oracle.sparse_decode(q, paged_cache(Ks, table, NB, page), paged_cache(Vs, table, NB, page),
                               table, np.array([[13, 0, 0, 0]], np.int32), [1], [5], [5],
                               scale=0.088)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], Vs[0][13, h // 2], atol=0)


# --------------------------------------------------------------------------------------
# whole path on the tiny seeded workload: planted heavy hitters are selected
# --------------------------------------------------------------------------------------

def test_tiny_workload_selects_planted_keys():
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch
    from sparse_attention_speculative_gb300.workloads import TINY
    batch = make_batch(TINY, "cpu")
    h = host_arrays(batch)
    out, logits, partial = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                         h["prefix_len"], scale=TINY.scale, P_max=TINY.P_max)
    score = oracle.score_from_logits(logits, h["prefix_len"])
    idx, n_sel = oracle.select(score, h["prefix_len"], k=TINY.k, n_sink=TINY.n_sink,
                               n_recent=TINY.n_recent)
    assert n_sel[0] == TINY.k
    planted = set(batch.planted[0].tolist())
    assert len(planted) == TINY.planted_count
    assert planted <= set(idx[0].tolist())
    np.testing.assert_allclose(oracle.score_from_partials(partial, h["prefix_len"]), score,
                               atol=1e-9)



# --------------------------------------------------------------------------------------
# Dustin hybrid budget (Methodology sec. 1) and semantic-retrieval-head mask (sec. 2)
# --------------------------------------------------------------------------------------

def test_select_hybrid_golden():
    with open(os.path.join(GOLDEN, "select_hybrid.json")) as f:
        g = json.load(f)
    st = np.array([g["score_target"]], np.float64)
    sd = np.array([g["score_draft"]], np.float64)
    idx, n_sel = oracle.select_hybrid(st, sd, [g["P"]], k=g["k"], m=g["m"], n_sink=g["n_sink"],
                                      n_recent=g["n_recent"])
    assert n_sel[0] == len(g["expected_idx"])
    assert idx[0, :n_sel[0]].tolist() == g["expected_idx"]


@pytest.mark.parametrize("seed", range(6))
def test_select_hybrid_limits_and_invariants(seed):
    rng = np.random.default_rng(seed)
    rows, P_max = 4, 300
    prefix = rng.integers(0, P_max + 1, size=rows).astype(np.int32)
    st = rng.integers(-5, 6, size=(rows, P_max)).astype(np.float64)  # ties on purpose
    sd = rng.normal(size=(rows, P_max))
    k, ns, nr = 60, 4, 16
    # m = 0: the target signal alone
    a, an = oracle.select_hybrid(st, sd, prefix, k=k, m=0, n_sink=ns, n_recent=nr)
    b, bn = oracle.select(st, prefix, k=k, n_sink=ns, n_recent=nr)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(an, bn)
    # m covering the whole remaining budget: the draft signal alone
    a, an = oracle.select_hybrid(st, sd, prefix, k=k, m=k, n_sink=ns, n_recent=nr)
    b, bn = oracle.select(sd, prefix, k=k, n_sink=ns, n_recent=nr)
    np.testing.assert_array_equal(a, b)
    # in between: protected kept, the best m by draft kept, the rest the best by target
    m = 7
    a, an = oracle.select_hybrid(st, sd, prefix, k=k, m=m, n_sink=ns, n_recent=nr)
    for r, P in enumerate(prefix.tolist()):
        n = min(k, P)
        got = a[r, :an[r]].tolist()
        assert an[r] == n and got == sorted(set(got))
        prot = set(range(min(ns, P))) | set(range(max(0, P - nr), P))
        assert prot <= set(got)
        cand = [j for j in range(P) if j not in prot]
        nd = min(m, n - len(prot))
        draft_best = sorted(cand, key=lambda j: (-sd[r, j], j))[:nd]
        assert set(draft_best) <= set(got)
        rest = [j for j in cand if j not in draft_best]
        want_t = sorted(rest, key=lambda j: (-st[r, j], j))[:n - len(prot) - nd]
        assert set(got) == prot | set(draft_best) | set(want_t)


def test_partial_masked_closed_form():
    s = _structured_verify(R=3)
    scale = 1.0 / math.sqrt(s["d"])
    _, logits, partial = oracle.verify(s["q"], s["k"], s["v"], s["table"], s["prefix"],
                                       scale=scale, P_max=64)
    Hq, G, Hkv, R = s["Hq"], s["G"], s["Hkv"], s["R"]
    np.testing.assert_array_equal(
        oracle.partial_masked(logits, s["prefix"], np.ones(Hq, np.uint8), Hkv), partial)
    assert np.all(oracle.partial_masked(logits, s["prefix"], np.zeros(Hq, np.uint8), Hkv) == 0)
    mask = np.array([1 if h % 3 == 0 else 0 for h in range(Hq)], np.uint8)
    got = oracle.partial_masked(logits, s["prefix"], mask, Hkv)
    for b, P in enumerate(s["prefix"]):
        j = np.arange(P)
        for g in range(Hkv):
            want = np.zeros(P)
            for t in (0, R - 1):
                for h in range(g * G, (g + 1) * G):
                    if mask[h]:
                        want += scale * ((t + 1) * ((j % 7) - 3) + (h + 1) * (g + 1) + (b + 1))
            np.testing.assert_allclose(got[b, g, :P], want, rtol=0, atol=1e-10)


# --------------------------------------------------------------------------------------
# per-query block top-k (the sparse-verification summary, "Sparse Verification Engine":
# each query keeps its top-k key/value blocks by a cheap relevance score; the score read
# here is the query's scaled dot product with the page's mean key)
# --------------------------------------------------------------------------------------

def test_block_topk_scores_closed_form():
    """On the structured input the logit of key j is known in closed form, so the page
    score is that closed form averaged over the page's prefix rows (rows at or past the
    prefix length, which hold the verify block's keys, are excluded)."""
    s = _structured_verify(prefix=(37, 50), R=3)
    scale = 1.0 / math.sqrt(s["d"])
    R, Hq, G = s["R"], s["Hq"], s["G"]
    scores, blocks = oracle.block_topk(s["q"], s["k"], s["table"], s["prefix"], kb=2,
                                       scale=scale, page_blocks_max=5)
    for b, P in enumerate(s["prefix"]):
        nblk = (P + 15) // 16
        for t in range(R):
            for h in range(Hq):
                for beta in range(nblk):
                    j = np.arange(16 * beta, min(16 * beta + 16, P))
                    want = scale * np.mean((t + 1) * ((j % 7) - 3) + (h + 1) * (h // G + 1)
                                           + (b + 1))
                    assert abs(scores[b, t, h, beta] - want) <= 1e-12
                assert np.all(scores[b, t, h, nblk:] == 0)


def _small_random_blocks(seed, prefix, Hq=4, Hkv=2, d=64, R=2, page=16):
    rng = np.random.default_rng(seed)
    lengths = [p + R for p in prefix]
    table, NB, Ks, _ = _random_paged(rng, lengths, Hkv, d, page, seed)
    q = bf16_round_bits(rng.normal(size=(len(prefix), R, Hq, d)))
    return q, paged_cache(Ks, table, NB, page), table, np.array(prefix, np.int32)


@pytest.mark.parametrize("kb", [1, 3, 5])
def test_block_topk_matches_bruteforce(kb):
    """For up to 9 pages, enumerate every kb-subset of pages; the chosen set maximises
    the summed page score (ties to the lexicographically smallest set)."""
    q, kc, table, prefix = _small_random_blocks(31 + kb, [130, 75, 16])
    scores, blocks = oracle.block_topk(q, kc, table, prefix, kb=kb, scale=0.125)
    B, R, Hq, _ = q.shape
    for b, P in enumerate(prefix):
        nblk = (P + 15) // 16
        for t in range(R):
            for h in range(Hq):
                sc = scores[b, t, h, :nblk]
                best, best_set = None, None
                for T in itertools.combinations(range(nblk), min(kb, nblk)):
                    total = sum(sc[i] for i in T)
                    if best is None or total > best + 1e-12:
                        best, best_set = total, T
                got = blocks[b, t, h]
                assert list(got[:len(best_set)]) == list(best_set)
                assert np.all(got[len(best_set):] == -1)


def test_block_topk_each_head_finds_its_planted_page():
    """Heads of one KV group share keys but not queries: with orthogonal queries and one
    page planted along each head's query, every head's top page is its own."""
    B, R, Hq, Hkv, d, page = 1, 2, 8, 2, 64, 16
    G = Hq // Hkv
    P = 16 * 12
    rng = np.random.default_rng(5)
    q = np.zeros((B, R, Hq, d), np.float32)
    for t in range(R):
        for h in range(Hq):
            q[0, t, h, h] = 1.0 + t
    K = bits_to_float(bf16_round_bits(0.05 * rng.normal(size=(P + R, Hkv, d)))).astype(np.float32)
    planted = {}
    for h in range(Hq):
        g = h // G
        beta = 1 + (5 * h + 3) % 11
        while beta in planted.values():
            beta = 1 + beta % 11
        planted[h] = beta
        K[16 * beta:16 * beta + 16, g, h] += 4.0
    K = bits_to_float(bf16_round_bits(K)).astype(np.float32)
    table, NB = make_table([P + R], page, shuffle_seed=3)
    kc = paged_cache([K], table, NB, page)
    _, blocks = oracle.block_topk(bf16_bits(q), kc, table, np.array([P], np.int32), kb=1,
                                  scale=0.125)
    for t in range(R):
        for h in range(Hq):
            assert blocks[0, t, h, 0] == planted[h], (t, h)


def test_block_topk_budget_limits_and_ties():
    q, kc, table, prefix = _small_random_blocks(9, [0, 40, 64])
    _, blocks = oracle.block_topk(q, kc, table, prefix, kb=6, scale=0.125)
    assert np.all(blocks[0] == -1)                                  # empty prefix
    assert np.all(blocks[1, :, :, :3] == np.arange(3))              # 3 pages, all kept
    assert np.all(blocks[1, :, :, 3:] == -1)
    assert np.all(blocks[2, :, :, :4] == np.arange(4))
    # identical keys everywhere: every page scores the same, the lowest pages win
    kc_same = np.broadcast_to(kc[:1, :, :1, :], kc.shape).copy()
    scores, blocks = oracle.block_topk(q, kc_same, table, prefix, kb=2, scale=0.125)
    assert np.all(blocks[1:, :, :, :] == np.array([0, 1]))
    for b in (1, 2):
        nblk = (prefix[b] + 15) // 16
        assert np.all(scores[b, :, :, :nblk] == scores[b, :, :, :1])


def test_block_topk_block_table_permutation_invariance():
    rng = np.random.default_rng(12)
    d, page, R, Hq, Hkv = 64, 16, 3, 8, 2
    prefix = [200, 77]
    lengths = [p + R for p in prefix]
    Ks = [bits_to_float(bf16_round_bits(rng.normal(size=(L, Hkv, d)))).astype(np.float32)
          for L in lengths]
    q = bf16_round_bits(rng.normal(size=(2, R, Hq, d)))
    results = []
    for seed in (None, 4, 9):
        table, NB = make_table(lengths, page, shuffle_seed=seed, extra_blocks=3)
        results.append(oracle.block_topk(q, paged_cache(Ks, table, NB, page, fill=9.0), table,
                                         prefix, kb=4, scale=0.125))
    for other in results[1:]:
        for a, b in zip(results[0], other):
            np.testing.assert_array_equal(a, b)
