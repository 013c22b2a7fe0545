"""The draft step of a decode loop (vsd_sparse_decode_attn_step), through the C ABI:
the step's input token stored and attended inside the call must give exactly what the
separate append followed by the plain draft call gives (same output bits, same cache
bits) and match the fp64 oracle on the cache after the store; the selection's cache rows
recorded by one step and reused by the next must change nothing in the result.  Each
case runs on every draft kernel: one split per CTA, the warp-specialised persistent
kernel (many splits) and the CUDA-core kernel (very long lists)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_utils import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_speculative_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)
    yield


def _case(name):
    """(workload, idx, n_sel, tail_start, seq_len, max_tail) on the GPU."""
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    dev = "cuda"
    if name == "one_split":      # 8 pairs x 17 splits: the one-split kernel
        w = Workload("ds1", B=1, P=32768, Hq=32, Hkv=8, d=128, gamma=4, k=2048, n_sink=16,
                     n_recent=256, seed=21)
        n_per = [2048]
    elif name == "persistent":   # 6 x 8 pairs x 33 splits: the warp-specialised kernel
        prefix = (6000, 5000, 4500, 300, 129, 2000)
        w = Workload("ds2", B=6, P=6000, Hq=32, Hkv=8, d=128, gamma=3, k=4096, n_sink=0,
                     n_recent=0, seed=22, prefix_lens=prefix)
        n_per = [4096, 2000, 129, 128, 100, 1999]
    elif name == "persistent_g8_d64":
        prefix = (7000, 6500, 5000, 4000)
        w = Workload("ds3", B=4, P=7000, Hq=64, Hkv=8, d=64, gamma=5, k=4096, n_sink=0,
                     n_recent=0, seed=23, prefix_lens=prefix)
        n_per = [4096, 4000, 3000, 257]
    elif name == "persistent_g1":
        prefix = (9000,) * 8
        w = Workload("ds4", B=8, P=9000, Hq=8, Hkv=8, d=128, gamma=2, k=4096, n_sink=0,
                     n_recent=0, seed=24, prefix_lens=prefix)
        n_per = [4096, 4095, 3000, 2048, 1024, 511, 130, 1]
    else:                        # a list of more than 1024 batches: the CUDA-core kernel
        P = 200000
        w = Workload("ds5", B=1, P=P, Hq=2, Hkv=1, d=64, gamma=2, k=140000, n_sink=4,
                     n_recent=64, seed=25, prefix_lens=(P,))
        n_per = [140000]
    batch = make_batch(w, dev)
    rng = np.random.default_rng(w.seed)
    idx = torch.full((w.B, w.k), -1, dtype=torch.int32, device=dev)
    for b, (P, n) in enumerate(zip(w.prefix(), n_per)):
        if n:
            sel = np.sort(rng.choice(P, size=n, replace=False)).astype(np.int32)
            idx[b, :n] = torch.from_numpy(sel).to(dev)
    n_sel = torch.tensor(n_per, dtype=torch.int32, device=dev)
    tails = rng.integers(1, w.R + 1, size=w.B)  # every tail holds the input token
    tail_start = batch.prefix_len.clone()
    seq_len = batch.prefix_len + torch.tensor(tails, dtype=torch.int32, device=dev)
    return w, batch, idx, n_sel, tail_start, seq_len, int(tails.max())


CASES = ["one_split", "persistent", "persistent_g8_d64", "persistent_g1", "cuda_core"]


@pytest.mark.parametrize("name", CASES)
def test_input_token_stored_and_attended_in_the_call(name):
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300.synth import host_arrays, to_u16
    w, batch, idx, n_sel, tail_start, seq_len, max_tail = _case(name)
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(w.seed + 1)
    k_new = torch.randn((w.B, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn((w.B, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    kc2, vc2 = batch.k_cache.clone(), batch.v_cache.clone()
    q = batch.q_draft[0]
    vsd.vsd_read_device_status()
    # reference path: the library's append, then the plain draft call
    vsd.vsd_append_kv(k_new.unsqueeze(1), v_new.unsqueeze(1), kc2, vc2, batch.block_table,
                      seq_len, pos_offset=-1)
    ref_out = vsd.vsd_sparse_decode_attn(q, kc2, vc2, batch.block_table, idx, n_sel,
                                         tail_start, seq_len, scale=w.scale, max_tail=max_tail)
    out = vsd.vsd_sparse_decode_attn_step(q, batch.k_cache, batch.v_cache, batch.block_table,
                                          idx, n_sel, tail_start, seq_len, scale=w.scale,
                                          max_tail=max_tail, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(batch.k_cache, kc2) and torch.equal(batch.v_cache, vc2)
    assert torch.equal(out, ref_out)
    h = host_arrays(batch)
    ref = oracle.sparse_decode(to_u16(q), h["k_cache"], h["v_cache"], h["block_table"],
                               idx.cpu().numpy(), n_sel.cpu().numpy(),
                               tail_start.cpu().numpy(), seq_len.cpu().numpy(), scale=w.scale)
    assert_attn_close(out.float().cpu().numpy(), ref, "draft step with its input token")


@pytest.mark.parametrize("name", CASES)
def test_selection_rows_recorded_then_reused(name):
    import sparse_attention_speculative_gb300 as vsd
    w, batch, idx, n_sel, tail_start, seq_len, max_tail = _case(name)
    dev = "cuda"
    rows = torch.full(idx.shape, -7, dtype=torch.int32, device=dev)
    q0, q1 = batch.q_draft[0], batch.q_draft[1]
    args = (batch.k_cache, batch.v_cache, batch.block_table, idx, n_sel, tail_start, seq_len)
    vsd.vsd_read_device_status()
    plain0 = vsd.vsd_sparse_decode_attn(q0, *args, scale=w.scale, max_tail=max_tail)
    plain1 = vsd.vsd_sparse_decode_attn(q1, *args, scale=w.scale, max_tail=max_tail)
    out0 = vsd.vsd_sparse_decode_attn_step(q0, *args, scale=w.scale, max_tail=max_tail,
                                           sel_rows=rows, flags=vsd.STEP_RECORD_ROWS)
    out1 = vsd.vsd_sparse_decode_attn_step(q1, *args, scale=w.scale, max_tail=max_tail,
                                           sel_rows=rows, flags=vsd.STEP_REUSE_ROWS)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    assert torch.equal(out0, plain0) and torch.equal(out1, plain1)
    # the recorded rows: block * Hkv * 16 + offset of every selected position
    table = batch.block_table.cpu().numpy().astype(np.int64)
    got = rows.cpu().numpy()
    ix = idx.cpu().numpy()
    for b, n in enumerate(n_sel.cpu().tolist()):
        j = ix[b, :n].astype(np.int64)
        want = table[b, j // 16] * w.Hkv * 16 + j % 16
        assert np.array_equal(got[b, :n], want), "row %d" % b
        assert np.all(got[b, n:] == -7), "positions past n_sel are not written"


def test_bad_recorded_row_is_flagged():
    import sparse_attention_speculative_gb300 as vsd
    w, batch, idx, n_sel, tail_start, seq_len, max_tail = _case("one_split")
    rows = torch.zeros(idx.shape, dtype=torch.int32, device="cuda")
    args = (batch.k_cache, batch.v_cache, batch.block_table, idx, n_sel, tail_start, seq_len)
    vsd.vsd_read_device_status()
    vsd.vsd_sparse_decode_attn_step(batch.q_draft[0], *args, scale=w.scale, max_tail=max_tail,
                                    sel_rows=rows, flags=vsd.STEP_RECORD_ROWS)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    rows[0, 5] = batch.k_cache.shape[0] * w.Hkv * 16 + 3   # past the cache
    rows[0, 9] = 16                                          # not a KV-head-0 row base
    vsd.vsd_sparse_decode_attn_step(batch.q_draft[1], *args, scale=w.scale, max_tail=max_tail,
                                    sel_rows=rows, flags=vsd.STEP_REUSE_ROWS)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == vsd.DEV_BAD_INDEX


def test_persistent_kernel_is_deterministic():
    """The warp-specialised kernel folds each consumer's splits into one partial and
    merges the partials in a fixed order: repeated calls give identical bits."""
    import sparse_attention_speculative_gb300 as vsd
    w, batch, idx, n_sel, tail_start, seq_len, max_tail = _case("persistent")
    args = (batch.k_cache, batch.v_cache, batch.block_table, idx, n_sel, tail_start, seq_len)
    outs = [vsd.vsd_sparse_decode_attn(batch.q_draft[0], *args, scale=w.scale,
                                       max_tail=max_tail).clone() for _ in range(4)]
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("name", CASES)
def test_early_gather_gives_the_same_bits(name):
    """With VSD_STEP_EARLY_GATHER the list is gathered before the call waits for its
    predecessor (here a draft call on another copy of the cache, which writes none of
    the inputs): the result is bit-identical to the call without it, with and without the
    input token and the recorded rows."""
    import sparse_attention_speculative_gb300 as vsd
    w, batch, idx, n_sel, tail_start, seq_len, max_tail = _case(name)
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(w.seed + 2)
    k_new = torch.randn((w.B, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn((w.B, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    other_k, other_v = batch.k_cache.clone(), batch.v_cache.clone()
    rows = torch.zeros(idx.shape, dtype=torch.int32, device=dev)
    q = batch.q_draft[0]
    kc_ref, vc_ref = batch.k_cache.clone(), batch.v_cache.clone()
    vsd.vsd_read_device_status()
    ref = vsd.vsd_sparse_decode_attn_step(q, kc_ref, vc_ref, batch.block_table, idx, n_sel,
                                          tail_start, seq_len, scale=w.scale, max_tail=max_tail,
                                          k_new=k_new, v_new=v_new)
    outs = []
    for flags in (vsd.STEP_EARLY_GATHER | vsd.STEP_RECORD_ROWS,
                  vsd.STEP_EARLY_GATHER | vsd.STEP_REUSE_ROWS, vsd.STEP_EARLY_GATHER):
        kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
        vsd.vsd_sparse_decode_attn(batch.q_draft[1], other_k, other_v, batch.block_table, idx,
                                   n_sel, tail_start, seq_len, scale=w.scale, max_tail=max_tail)
        outs.append(vsd.vsd_sparse_decode_attn_step(
            q, kc, vc, batch.block_table, idx, n_sel, tail_start, seq_len, scale=w.scale,
            max_tail=max_tail, k_new=k_new, v_new=v_new, sel_rows=rows, flags=flags))
        torch.cuda.synchronize()
        assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)
    assert vsd.vsd_read_device_status() == 0
    for o in outs:
        assert torch.equal(o, ref)
