"""The multi-layer decode loop (the 36-layer attention-only configuration, scaled down
so the oracle checks every call), run through `DecodeLoop` exactly as the benchmark
runs it: per iteration the verify block's K/V are appended by the library, every layer
runs the scored verification, one selection launch covers all layers x sequences, the
accepted counts advance the prefixes on the device, and every draft step appends its
input token's K/V before attending the selection plus the dense tail.

The test keeps its own host copy of every cache and applies the same writes with plain
numpy indexing at positions it computes itself; each call's output is compared with the
fp64 oracle on that copy as it stood when the call ran, and at the end of every
iteration the device caches must equal the host copy bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import assert_attn_close, assert_index_sets

pytestmark = pytest.mark.gpu


def _write_rows(hk, hv, table, b, pos, k_rows, v_rows, page=16):
    """Host copy of a cache append: rows [n, Hkv, d] (uint16) at positions pos."""
    for t, p in enumerate(pos):
        blk = int(table[b, p // page])
        hk[blk, :, p % page, :] = k_rows[t]
        hv[blk, :, p % page, :] = v_rows[t]


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run_loop(w, layers, iterations, seed):
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    from sparse_attention_speculative_gb300.decode_loop import DecodeLoop
    from sparse_attention_speculative_gb300.synth import host_arrays, make_batch, seeded_bf16
    build.build()
    oracle.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    B, R, Hq, Hkv, d, gamma = w.B, w.R, w.Hq, w.Hkv, w.d, w.gamma
    prefix = list(w.prefix())
    P_max = max(prefix) + iterations * R
    batches = [make_batch(w, dev, layer=l, extra_capacity=4 * R + iterations * R)
               for l in range(layers)]
    host = [host_arrays(bt) for bt in batches]
    loop = DecodeLoop([bt.k_cache for bt in batches], [bt.v_cache for bt in batches],
                      [bt.block_table for bt in batches], prefix, Hq=Hq, gamma=gamma, k=w.k,
                      n_sink=w.n_sink, n_recent=w.n_recent, P_max=P_max, scale=w.scale)
    assert vsd.vsd_read_device_status() == 0
    rng = np.random.default_rng(seed)
    for it in range(iterations):
        tag = seed * 1000 + it
        cpu = torch.device("cpu")
        loop.h_q.copy_(seeded_bf16((layers, B, R, Hq, d), 13 * tag, cpu))
        loop.h_q_draft.copy_(seeded_bf16((layers, gamma, B, Hq, d), 23 * tag, cpu))
        loop.h_k_verify.copy_(seeded_bf16((layers, B, R, Hkv, d), 7 * tag, cpu))
        loop.h_v_verify.copy_(seeded_bf16((layers, B, R, Hkv, d), 11 * tag, cpu))
        loop.h_k_draft.copy_(seeded_bf16((layers, gamma, B, Hkv, d), 17 * tag, cpu))
        loop.h_v_draft.copy_(seeded_bf16((layers, gamma, B, Hkv, d), 19 * tag, cpu))
        acc = rng.integers(0, gamma + 1, size=B)
        loop.h_accepted.copy_(torch.from_numpy(acc.astype(np.int32)))
        loop.run(sync=True)
        assert vsd.vsd_read_device_status() == 0

        pl = np.array(prefix, dtype=np.int32)
        s_rows = []
        for l in range(layers):
            h = host[l]
            for b in range(B):
                _write_rows(h["k_cache"], h["v_cache"], h["block_table"], b,
                            range(prefix[b], prefix[b] + R), _bits(loop.h_k_verify[l, b]),
                            _bits(loop.h_v_verify[l, b]))
            o_ref, l_ref, _ = oracle.verify(_bits(loop.h_q[l]), h["k_cache"], h["v_cache"],
                                            h["block_table"], pl, scale=w.scale,
                                            P_max=loop.row_stride)
            assert_attn_close(loop.h_out[l].float().numpy(), o_ref, "loop verify output")
            s_rows.append(oracle.score_from_logits(l_ref, pl))
        s_ref = np.concatenate(s_rows, axis=0)
        rows_pl = np.tile(pl, layers)
        i_ref, n_ref = oracle.select(s_ref, rows_pl, k=w.k, n_sink=w.n_sink,
                                     n_recent=w.n_recent)
        idx = loop.h_idx.numpy().copy()
        n_sel = loop.h_n_sel.numpy().copy()
        assert_index_sets(idx, n_sel, i_ref, n_ref, s_ref, rows_pl, w.k, w.n_sink, w.n_recent)
        # the device bookkeeping: prefixes grow by the accepted drafts and one token
        new_prefix = [prefix[b] + int(acc[b]) + 1 for b in range(B)]
        assert loop.h_prefix_len_out.tolist() == new_prefix
        assert loop.h_tail_start_out.tolist() == prefix
        seq = [[prefix[b] + int(acc[b]) + 2 + i for b in range(B)] for i in range(gamma)]
        assert loop.h_seq_len_out.tolist() == seq
        for i in range(gamma):
            for l in range(layers):
                h = host[l]
                for b in range(B):
                    _write_rows(h["k_cache"], h["v_cache"], h["block_table"], b,
                                [seq[i][b] - 1], _bits(loop.h_k_draft[l, i, b:b + 1]),
                                _bits(loop.h_v_draft[l, i, b:b + 1]))
                rows = slice(l * B, (l + 1) * B)
                ref = oracle.sparse_decode(_bits(loop.h_q_draft[l, i]), h["k_cache"],
                                           h["v_cache"], h["block_table"], idx[rows],
                                           n_sel[rows], pl, np.array(seq[i], np.int32),
                                           scale=w.scale)
                assert_attn_close(loop.h_draft_out[i, l].float().numpy(), ref,
                                  "loop draft output (step %d, layer %d)" % (i, l))
        for l in range(layers):
            got = host_arrays(batches[l])
            assert np.array_equal(got["k_cache"], host[l]["k_cache"]), "layer %d K cache" % l
            assert np.array_equal(got["v_cache"], host[l]["v_cache"]), "layer %d V cache" % l
        prefix = new_prefix
    # a second run of the graph from the reset state repeats the first iteration's
    # lengths (the state lives on the device and is put back by reset())
    loop.reset()
    loop.synchronize()


def test_decode_loop_scaled_down():
    from sparse_attention_speculative_gb300.workloads import Workload
    w = Workload("loop_small", B=3, P=3000, Hq=16, Hkv=4, d=128, gamma=5, k=256, n_sink=16,
                 n_recent=64, planted_frac=0.01, seed=5, prefix_lens=(3000, 1777, 2501))
    _run_loop(w, layers=3, iterations=3, seed=5)


def test_append_and_advance_flag_bad_inputs():
    """Positions past the block table and block entries outside the cache are skipped
    and flagged; an accepted count outside [0, gamma] leaves the prefix unchanged."""
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    NB, Hkv, d = 8, 2, 64
    kc = torch.zeros((NB, Hkv, 16, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    table = torch.tensor([[3, 5], [1, -1]], dtype=torch.int32, device=dev)
    rows = torch.ones((2, 2, Hkv, d), dtype=torch.bfloat16, device=dev)
    vsd.vsd_read_device_status()
    # sequence 0 at 30, 31 (block 5, rows 14, 15); sequence 1 at 16, 17 (entry -1)
    pos = torch.tensor([30, 16], dtype=torch.int32, device=dev)
    vsd.vsd_append_kv(rows, 2 * rows, kc, vc, table, pos)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_BLOCK
    assert float(kc[5, :, 14:16].float().min()) == 1.0 and float(vc[5, :, 14:16].float().min()) == 2.0
    assert int((kc != 0).sum()) == 2 * Hkv * d  # nothing else written
    # past the table (32 positions per sequence)
    vsd.vsd_append_kv(rows, rows, kc, vc, table, torch.tensor([31, 0], dtype=torch.int32,
                                                             device=dev))
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_LENGTH
    acc = torch.tensor([2, 7], dtype=torch.int32, device=dev)
    pl = torch.tensor([100, 200], dtype=torch.int32, device=dev)
    ts = torch.empty(2, dtype=torch.int32, device=dev)
    sl = torch.empty((3, 2), dtype=torch.int32, device=dev)
    copies = torch.empty((2, 2), dtype=torch.int32, device=dev)
    vsd.vsd_advance_lengths(acc, pl, ts, sl, max_prefix=1000, prefix_copies=copies)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_LENGTH
    assert pl.tolist() == [103, 200] and ts.tolist() == [100, 200]
    assert sl.tolist() == [[104, 201], [105, 202], [106, 203]]
    assert copies.tolist() == [[103, 200], [103, 200]]
