"""The allocation-free verification call, checked against the regular one.

vsd_verify_attn_collect_noalloc serves callers that cannot hand the library device
memory on the decode path (an engine that has reserved all free HBM for its KV
cache, or a host that forbids cudaMalloc there because it can synchronize the
device).  It keeps its scratch in a fixed device array instead of a workspace.  This
file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.parity_utils import assert_attn_close, assert_rel_close

pytestmark = pytest.mark.gpu


def _regular(vsd, batch, w):
    return vsd.vsd_verify_attn_collect(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                       batch.prefix_len, P_max=w.P_max, scale=w.scale)


def _noalloc_c_abi(vsd, batch, w):
    """Call the entry point directly through the C ABI (ctypes), outputs preallocated."""
    lib = vsd.load()
    B, R, Hq, d = batch.q.shape
    geom = vsd.geom_for(B, Hq, batch.k_cache, batch.block_table)
    out = torch.full_like(batch.q, float("nan"))
    logits = torch.full((B, 2, Hq, w.P_max), float("nan"), dtype=torch.float32, device="cuda")
    partial = torch.full((B, w.Hkv, w.P_max), float("nan"), dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.vsd_verify_attn_collect_noalloc(
        ctypes.byref(geom), R, p(batch.q), p(batch.k_cache), p(batch.v_cache),
        p(batch.block_table), p(batch.prefix_len), 0, R - 1, w.P_max, ctypes.c_float(w.scale),
        p(logits), p(partial), p(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, "vsd_verify_attn_collect_noalloc returned %d" % rc
    return out, logits, partial


def _compare(got, ref, prefix):
    assert_attn_close(got[0].float().cpu().numpy(), ref[0].float().cpu().numpy(),
                      "no-alloc verify output")
    lg, lr = got[1].cpu().numpy(), ref[1].cpu().numpy()
    pg, pr = got[2].cpu().numpy(), ref[2].cpu().numpy()
    for b, P in enumerate(prefix):
        assert_rel_close(lg[b, :, :, :P], lr[b, :, :, :P], "no-alloc collected logits")
        assert_rel_close(pg[b, :, :P], pr[b, :, :P], "no-alloc partial scores")


def test_noalloc_matches_regular_entry_point_twice():
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import QWEN3_8B_32K, Workload
    build.build()
    torch.cuda.set_device(0)
    first = QWEN3_8B_32K
    second = Workload("ragged", B=3, P=9000, Hq=16, Hkv=4, d=128, gamma=3, k=64, n_sink=4,
                      n_recent=16, planted_frac=0.01, seed=12, prefix_lens=(9000, 130, 4100))
    for w in (first, second):  # two calls in a row; the second sees the first's scratch
        batch = make_batch(w, "cuda")
        ref = _regular(vsd, batch, w)
        got = _noalloc_c_abi(vsd, batch, w)
        torch.cuda.synchronize()
        assert vsd.vsd_read_device_status() == 0
        _compare(got, ref, list(w.prefix()))


def test_noalloc_rejects_geometry_beyond_its_scratch():
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    build.build()
    lib = vsd.load()
    # 512 (sequence, KV head) pairs with 64 verify rows each need more partial-result
    # scratch than the fixed array holds; the call must refuse before touching memory
    geom = vsd.Geom(64, 64, 8, 128, 16, 2100, 64 * 2100)
    need = ctypes.c_size_t(0)
    assert lib.vsd_verify_workspace_size(ctypes.byref(geom), 8, 32768, ctypes.byref(need)) == 0
    assert need.value > (16 << 20)
    rc = lib.vsd_verify_attn_collect_noalloc(ctypes.byref(geom), 8, None, None, None, None, None,
                                             0, 7, 32768, ctypes.c_float(0.088), None, None,
                                             None, None)
    assert rc == -4  # VSD_ERR_WORKSPACE
    np.testing.assert_equal(rc, -4)


def test_noalloc_near_its_scratch_bound():
    """A geometry whose partial-result scratch fills the fixed array almost to its end
    (the last slots are where an offset error would first write past it): the same
    results as the regular entry point."""
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300 import build
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import Workload
    build.build()
    torch.cuda.set_device(0)
    lib = vsd.load()
    limit = 16 << 20
    chosen = None
    for B in range(1, 200):  # 8 verify rows x 8 query heads per KV head: 33 KB slots
        geom = vsd.Geom(B, 64, 8, 128, 16, 64, 64 * B)
        need = ctypes.c_size_t(0)
        assert lib.vsd_verify_workspace_size(ctypes.byref(geom), 8, 1000,
                                             ctypes.byref(need)) == 0
        if need.value > limit:
            break
        chosen = (B, need.value)
    assert chosen is not None and chosen[1] > limit - (1 << 20), chosen
    B = chosen[0]
    w = Workload("noalloc_edge", B=B, P=1000, Hq=64, Hkv=8, d=128, gamma=7, k=64, n_sink=4,
                 n_recent=16, seed=13, prefix_lens=tuple(1000 - (b * 37) % 600 for b in range(B)))
    batch = make_batch(w, "cuda")
    w = w.with_(prefix_lens=tuple(int(x) for x in batch.prefix_len.cpu()))
    ref = _regular(vsd, batch, w)
    got = _noalloc_c_abi(vsd, batch, w)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    _compare(got, ref, list(w.prefix()))
