"""The multi-layer iteration loop (the 36-layer attention-only configuration, scaled
down so the oracle checks every call): per iteration, the verify block's K/V are
appended, every layer runs verification + Collect-2-Query, one selection launch covers
all layers x sequences, a seeded accept count advances each prefix, and gamma draft
steps per layer attend the selection plus the dense tail.  Every call is compared with
the fp64 oracle on the same cache contents."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import assert_attn_close, assert_index_sets, assert_rel_close

pytestmark = pytest.mark.gpu


def _loop(w, layers, iterations, seed):
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    from sparse_attention_speculative_gb300.synth import (host_arrays, make_batch, seeded_bf16,
                                                          to_u16, write_tokens)
    build.build()
    oracle.build()
    torch.cuda.set_device(0)
    dev = "cuda"
    B, R, Hq, Hkv, d, gamma = w.B, w.R, w.Hq, w.Hkv, w.d, w.gamma
    extra = iterations * R
    batches = [make_batch(w, dev, layer=l, extra_capacity=extra) for l in range(layers)]
    prefix = list(w.prefix())
    P_max = max(prefix) + extra
    rng = np.random.default_rng(seed)
    for it in range(iterations):
        pl = torch.tensor(prefix, dtype=torch.int32, device=dev)
        partial = torch.empty((layers * B, Hkv, P_max), dtype=torch.float32, device=dev)
        # the fused path: each layer's scored verification fills its rows of one score
        # buffer and one histogram buffer
        score = torch.empty((layers * B, P_max), dtype=torch.float32, device=dev)
        hist = torch.empty((layers * B, vsd.HIST_BINS), dtype=torch.int32, device=dev)
        s_ref_rows = []
        for l, batch in enumerate(batches):
            tag = (seed * 1000 + it) * 100 + l
            # the verify block [previous bonus, d_1 .. d_gamma]: its K/V join the cache
            for b in range(B):
                pos = torch.arange(prefix[b], prefix[b] + R, device=dev)
                write_tokens(batch, b, pos, seeded_bf16((R, Hkv, d), 7 * tag + b, dev),
                             seeded_bf16((R, Hkv, d), 11 * tag + b, dev))
            batch.q = seeded_bf16((B, R, Hq, d), 13 * tag, dev)
            batch.prefix_len = pl
            out, logits, _ = vsd.vsd_verify_attn_collect(
                batch.q, batch.k_cache, batch.v_cache, batch.block_table, pl, P_max=P_max,
                scale=w.scale, partial=partial[l * B:(l + 1) * B])
            out_f = vsd.vsd_verify_attn_collect_scored(
                batch.q, batch.k_cache, batch.v_cache, batch.block_table, pl, P_max=P_max,
                scale=w.scale, score=score[l * B:(l + 1) * B],
                score_hist=hist[l * B:(l + 1) * B])[0]
            torch.cuda.synchronize()
            assert vsd.vsd_read_device_status() == 0
            assert torch.equal(out_f, out)
            h = host_arrays(batch)
            o_ref, l_ref, p_ref = oracle.verify(h["q"], h["k_cache"], h["v_cache"],
                                                h["block_table"], h["prefix_len"],
                                                scale=w.scale, P_max=P_max)
            assert_attn_close(out.float().cpu().numpy(), o_ref, "loop verify output")
            pa = partial[l * B:(l + 1) * B].cpu().numpy()
            for b, P in enumerate(prefix):
                assert_rel_close(pa[b, :, :P], p_ref[b, :, :P], "loop partial scores")
            s_ref_rows.append(oracle.score_from_logits(l_ref, h["prefix_len"]))
        # one selection launch for every (layer, sequence) row
        rows_pl = pl.repeat(layers)
        idx, n_sel, _ = vsd.vsd_select_topk(partial, rows_pl, k=w.k, n_sink=w.n_sink,
                                            n_recent=w.n_recent)
        idx_f, n_sel_f = vsd.vsd_select_topk_scored(score, hist, rows_pl, k=w.k,
                                                    n_sink=w.n_sink, n_recent=w.n_recent)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        assert torch.equal(idx_f, idx) and torch.equal(n_sel_f, n_sel)
        s_ref = np.concatenate(s_ref_rows, axis=0)
        rp = rows_pl.cpu().numpy()
        i64, n64 = oracle.select(s_ref, rp, k=w.k, n_sink=w.n_sink, n_recent=w.n_recent)
        assert_index_sets(idx.cpu().numpy(), n_sel.cpu().numpy(), i64, n64, s_ref, rp, w.k,
                          w.n_sink, w.n_recent)
        # accepted drafts: the prefix grows by a_b + 1 (accepted drafts and the old bonus)
        acc = rng.integers(0, gamma + 1, size=B)
        new_prefix = [prefix[b] + int(acc[b]) + 1 for b in range(B)]
        tail_start = pl.clone()
        for l, batch in enumerate(batches):
            for step in range(gamma):
                tag = ((seed * 1000 + it) * 100 + l) * 10 + step
                # the token this draft step feeds in: its K/V are appended first
                for b in range(B):
                    pos = torch.tensor([new_prefix[b] + step], device=dev)
                    write_tokens(batch, b, pos, seeded_bf16((1, Hkv, d), 17 * tag + b, dev),
                                 seeded_bf16((1, Hkv, d), 19 * tag + b, dev))
                seq_len = torch.tensor([new_prefix[b] + step + 1 for b in range(B)],
                                       dtype=torch.int32, device=dev)
                qd = seeded_bf16((B, Hq, d), 23 * tag, dev)
                rows = slice(l * B, (l + 1) * B)
                out = vsd.vsd_sparse_decode_attn(qd, batch.k_cache, batch.v_cache,
                                                 batch.block_table, idx[rows].contiguous(),
                                                 n_sel[rows].contiguous(), tail_start, seq_len,
                                                 scale=w.scale, max_tail=2 * gamma + 1)
                torch.cuda.synchronize()
                assert vsd.vsd_read_device_status() == 0
                h = host_arrays(batch)
                ref = oracle.sparse_decode(to_u16(qd), h["k_cache"], h["v_cache"],
                                           h["block_table"], idx[rows].cpu().numpy(),
                                           n_sel[rows].cpu().numpy(), tail_start.cpu().numpy(),
                                           seq_len.cpu().numpy(), scale=w.scale)
                assert_attn_close(out.float().cpu().numpy(), ref, "loop draft output")
        prefix = new_prefix


def test_layer_loop_scaled_down():
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("loop_small", B=3, P=3000, Hq=16, Hkv=4, d=128, gamma=5, k=256, n_sink=16,
                 n_recent=64, planted_frac=0.01, seed=5, prefix_lens=(3000, 1777, 2501))
    _loop(w, layers=3, iterations=3, seed=5)
