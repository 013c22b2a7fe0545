"""Comparison rules of the parity tests (tolerances stated once, here).

  attention outputs : max |gpu - oracle| <= 2e-2 (bf16 inputs, fp32 accumulation,
                      bf16 output)
  logits, scores    : |gpu - oracle| / max(|oracle|, 1) <= 1e-3
  index sets        : equal, except that an index in only one of the two sets must
                      score within 1e-3 * max(1, |s_k|) of s_k, the lowest oracle score
                      that entered the set by score (protected positions never differ)
"""
from __future__ import annotations

import numpy as np

ATTN_ATOL = 2e-2
REL_TOL = 1e-3


def max_abs(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)))


def assert_attn_close(got, ref, what="attention output"):
    err = max_abs(got, ref)
    assert np.all(np.isfinite(got)), "%s has non-finite values" % what
    assert err <= ATTN_ATOL, "%s: max|err| %.3e > %.1e" % (what, err, ATTN_ATOL)
    return err


def assert_rel_close(got, ref, what="logits"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)
    worst = float(np.max(rel))
    assert worst <= REL_TOL, "%s: max rel err %.3e > %.1e" % (what, worst, REL_TOL)
    return worst


def protected_set(P, n_sink, n_recent):
    return set(range(min(n_sink, P))) | set(range(max(0, P - n_recent), P))


def assert_index_sets(got_idx, got_n, ref_idx, ref_n, s_ref, prefix, k, n_sink, n_recent):
    """Compare per-row selections (arrays [rows, k]) under the tolerance rule."""
    got_idx = np.asarray(got_idx)
    ref_idx = np.asarray(ref_idx)
    n_mismatch = 0
    for r, P in enumerate(np.asarray(prefix).tolist()):
        assert int(got_n[r]) == int(ref_n[r]) == min(k, P), (r, got_n[r], ref_n[r])
        n = int(ref_n[r])
        g = got_idx[r, :n]
        assert np.all(np.diff(g) > 0), "row %d: selection not strictly ascending" % r
        assert np.all(got_idx[r, n:] == -1), "row %d: unused slots not -1" % r
        got, want = set(g.tolist()), set(ref_idx[r, :n].tolist())
        prot = protected_set(P, n_sink, n_recent)
        assert prot <= got, "row %d: protected position missing" % r
        diff = got ^ want
        if not diff:
            continue
        filled = sorted(want - prot)
        assert filled, "row %d: mismatch with nothing filled by score" % r
        kth = min(float(s_ref[r, j]) for j in filled)
        for j in diff:
            assert j not in prot and 0 <= j < P, (r, j)
            assert abs(float(s_ref[r, j]) - kth) <= REL_TOL * max(1.0, abs(kth)), \
                "row %d: index %d score %.6f vs k-th %.6f" % (r, j, s_ref[r, j], kth)
        n_mismatch += len(diff) // 2
    return n_mismatch


def fp32_row_sum(partial):
    """Aggregate per-KV-group partials in fp32, in group order (the precision and order
    in which the select kernel takes its decision)."""
    partial = np.asarray(partial, dtype=np.float32)
    s = partial[:, 0, :].copy()
    for g in range(1, partial.shape[1]):
        s = (s + partial[:, g, :]).astype(np.float32)
    return s.astype(np.float64)
