"""Every wait inside a kernel is bounded: a wait that runs out raises VSD_DEV_TIMEOUT,
the kernel stops issuing copies and tensor-core products, drains the ones it issued,
frees its TMEM and returns, and the GPU context stays usable.

The test builds a second copy of the library in which one wait of each waiting kernel
waits for a barrier that nothing completes before the kernel's end (a flag nothing
sets), with a 200 us wait limit, and runs the verification, the one-split and the
persistent draft step through its C ABI.  Each call must return within a second and
raise VSD_DEV_TIMEOUT and nothing else, and the regular library must still give
correct results after them."""
import ctypes
import time

import numpy as np
import pytest
import torch

from tests.parity_utils import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def short_wait_lib(tmp_path_factory):
    from sparse_attention_speculative_gb300 import build
    build.build()
    d = tmp_path_factory.mktemp("short_wait")
    path = build.build(extra_flags=("-DVSD_TEST_STALLED_WAIT", "-DVSD_WAIT_LIMIT_NS=200000ull"),
                       out=str(d / "libvsd_stall.so"), objdir=str(d / "obj"))
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.vsd_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.vsd_read_device_status.restype = ctypes.c_int
    return lib


def _status(lib):
    flags = ctypes.c_uint(0)
    assert lib.vsd_read_device_status(None, ctypes.byref(flags)) == 0
    return int(flags.value)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _timed(lib, fn):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = fn()
    assert rc == 0, rc
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    st = _status(lib)
    assert dt < 1.0, "a call with the short wait limit took %.3f s" % dt
    return st


def test_waits_that_run_out_end_the_kernels_cleanly(short_wait_lib):
    import sparse_attention_speculative_gb300 as vsd
    from sparse_attention_speculative_gb300.synth import make_batch
    from sparse_attention_speculative_gb300.workloads import QWEN3_8B_32K, Workload
    lib = short_wait_lib
    torch.cuda.set_device(0)
    seen = {}
    # verification (TMA rings, MMA issuer, softmax warps)
    w = QWEN3_8B_32K
    batch = make_batch(w, "cuda")
    geom = vsd.geom_for(w.B, w.Hq, batch.k_cache, batch.block_table)
    nb = vsd.vsd_verify_workspace_size(geom, w.R, w.P_max)
    ws = torch.zeros(nb + 256, dtype=torch.uint8, device="cuda")
    ws = ws[(-ws.data_ptr()) % 256:]
    out = torch.empty_like(batch.q)
    logits = torch.empty((w.B, 2, w.Hq, w.P_max), dtype=torch.float32, device="cuda")
    partial = torch.empty((w.B, w.Hkv, w.P_max), dtype=torch.float32, device="cuda")
    seen["verify"] = _timed(lib, lambda: lib.vsd_verify_attn_collect(
        ctypes.byref(geom), w.R, _p(batch.q), _p(batch.k_cache), _p(batch.v_cache),
        _p(batch.block_table), _p(batch.prefix_len), 0, w.R - 1, w.P_max,
        ctypes.c_float(w.scale), _p(logits), _p(partial), _p(out), _p(ws),
        ctypes.c_size_t(nb), None))
    # draft steps: one split per CTA (8 pairs) and the persistent kernel (many splits)
    for name, B, prefix in (("one_split", 1, (32768,)), ("persistent", 8, (9000,) * 8)):
        wd = Workload("to_" + name, B=B, P=prefix[0], Hq=32, Hkv=8, d=128, gamma=3, k=4096,
                      n_sink=0, n_recent=0, seed=77, prefix_lens=prefix)
        bd = make_batch(wd, "cuda")
        rng = np.random.default_rng(5)
        idx = torch.tensor(np.stack([np.sort(rng.choice(p, size=4096, replace=False))
                                     for p in prefix]).astype(np.int32), device="cuda")
        n_sel = torch.full((B,), 4096, dtype=torch.int32, device="cuda")
        tail = bd.prefix_len.clone()
        seq = bd.prefix_len + 3
        g2 = vsd.geom_for(B, wd.Hq, bd.k_cache, bd.block_table)
        nb2 = vsd.vsd_sparse_workspace_size(g2, 4096, 7)
        sws = torch.zeros(nb2 + 256, dtype=torch.uint8, device="cuda")
        sws = sws[(-sws.data_ptr()) % 256:]
        dout = torch.empty((B, wd.Hq, wd.d), dtype=torch.bfloat16, device="cuda")
        seen[name] = _timed(lib, lambda: lib.vsd_sparse_decode_attn(
            ctypes.byref(g2), _p(bd.q_draft[0]), _p(bd.k_cache), _p(bd.v_cache),
            _p(bd.block_table), _p(idx), _p(n_sel), 4096, _p(tail), _p(seq), 7,
            ctypes.c_float(wd.scale), _p(dout), _p(sws), ctypes.c_size_t(nb2), None))
        # a call that gave up may leave the per-pair counters behind: zero them (as the
        # workspace contract asks after VSD_DEV_TIMEOUT)
        sws.zero_()
    for name, st in seen.items():
        assert st == 0x8, "%s: status 0x%x (a stalled wait must raise VSD_DEV_TIMEOUT)" % (
            name, st)
    # the context is healthy: the regular library still matches the fp64 oracle
    import oracle
    from sparse_attention_speculative_gb300.synth import host_arrays
    oracle.build()
    o2, _, _ = vsd.vsd_verify_attn_collect(batch.q, batch.k_cache, batch.v_cache,
                                           batch.block_table, batch.prefix_len, P_max=w.P_max,
                                           scale=w.scale)
    torch.cuda.synchronize()
    assert vsd.vsd_read_device_status() == 0
    h = host_arrays(batch)
    o_ref, _, _ = oracle.verify(h["q"], h["k_cache"], h["v_cache"], h["block_table"],
                                h["prefix_len"], scale=w.scale, P_max=w.P_max)
    assert_attn_close(o2.float().cpu().numpy(), o_ref, "verify after the short-wait calls")
