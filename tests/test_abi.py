"""The C-ABI library: it builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vsd.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_speculative_gb300 import build
    from sparse_attention_speculative_gb300._lib import load
    build.build()
    return load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("vsd_verify_attn_collect", "vsd_select_topk", "vsd_sparse_decode_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "libvsd.so does not export %s" % name


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        s = lib.vsd_get_error_string(code)
        assert isinstance(s, bytes) and len(s) > 0


def _geom(**kw):
    from sparse_attention_speculative_gb300._lib import Geom
    base = dict(B=1, Hq=32, Hkv=8, head_dim=128, page_size=16, max_blocks_per_seq=64,
                num_blocks=64)
    base.update(kw)
    return Geom(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=30), -1),              # Hq not a multiple of Hkv
    (dict(head_dim=96), -2),        # unsupported head dim
    (dict(page_size=32), -2),       # unsupported page size
    (dict(Hq=24, Hkv=8), -2),       # G = 3 is not a power of two
    (dict(num_blocks=0), -1),
])
def test_verify_rejects_bad_geometry(lib, kw, code):
    g = _geom(**kw)
    rc = lib.vsd_verify_attn_collect(ctypes.byref(g), 5, None, None, None, None, None, 0, 4,
                                     1024, ctypes.c_float(0.088), None, None, None, None, 0, None)
    assert rc == code


def test_verify_rejects_too_many_rows(lib):
    g = _geom(Hq=64, Hkv=8)  # G = 8: R * G = 72 > 64
    rc = lib.vsd_verify_attn_collect(ctypes.byref(g), 9, None, None, None, None, None, 0, 8,
                                     1024, ctypes.c_float(0.088), None, None, None, None, 0, None)
    assert rc == -2


def test_select_rejects_budget_below_protected(lib):
    rc = lib.vsd_select_topk(1, 8, None, None, 1024, 10, 8, 8, None, None, None, None, 0, None)
    assert rc == -1


def test_select_rejects_null_outputs(lib):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    rc = lib.vsd_select_topk(1, 8, p, p, 1024, 64, 4, 16, None, None, None, None, 0, None)
    assert rc == -1


def test_sparse_rejects_missing_index_arrays(lib):
    g = _geom()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    rc = lib.vsd_sparse_decode_attn(ctypes.byref(g), p, p, p, p, None, None, 16, p, p, 0,
                                    ctypes.c_float(0.088), p, None, 0, None)
    assert rc == -1


def test_collect_all_rejects_wide_groups(lib):
    # the all-rows variant supports R * G <= 48; G = 8 with R = 8 is 64
    geom = _geom(Hq=64, Hkv=8)
    rc = lib.vsd_verify_attn_collect_all(ctypes.byref(geom), 8, None, None, None, None, None,
                                         1024, ctypes.c_float(0.1), None, None, None, None, 0,
                                         None)
    assert rc == -2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_sparse_workspace_holds_aligned_split_slots(lib, d, G):
    """The draft step's workspace: per-(sequence, KV head) counters, then one partial
    (m, l, o) slot per split -- the G maxima and sums padded to a multiple of four
    floats, then the G output rows of d floats -- so that every slot and every output
    row starts on a 16-byte boundary (the merge reads them as float4)."""
    B, Hkv = 3, 8
    g = _geom(B=B, Hq=Hkv * G, Hkv=Hkv, head_dim=d)
    k_max, max_tail = 2048, 9  # 2057 positions: 17 splits of 128
    size = ctypes.c_size_t(0)
    assert lib.vsd_sparse_workspace_size(ctypes.byref(g), k_max, max_tail,
                                         ctypes.byref(size)) == 0
    splits = -(-(k_max + max_tail) // 128)
    header = -(-2 * G // 4) * 4
    slot = header + G * d
    assert header * 4 % 16 == 0 and slot * 4 % 16 == 0
    counters = -(-B * Hkv * 4 // 256) * 256
    assert size.value == counters + B * Hkv * splits * slot * 4


def test_append_rejects_bad_arguments(lib):
    g = _geom()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    # a missing cache pointer, a negative row count, a misaligned row buffer
    assert lib.vsd_append_kv(ctypes.byref(g), 4, p, p, p, p, 0, None, p, None) == -1
    assert lib.vsd_append_kv(ctypes.byref(g), -1, p, p, p, p, 0, p, p, None) == -1
    q = ctypes.c_void_p(p.value + 4)
    assert lib.vsd_append_kv(ctypes.byref(g), 4, q, p, p, p, 0, p, p, None) == -1
    # nothing to store: no launch, no device needed
    assert lib.vsd_append_kv(ctypes.byref(g), 0, None, None, None, None, 0, None, None,
                             None) == 0
    assert lib.vsd_append_kv(ctypes.byref(_geom(head_dim=96)), 4, p, p, p, p, 0, p, p,
                             None) == -2


def test_advance_rejects_bad_arguments(lib):
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    assert lib.vsd_advance_lengths(4, 5, None, 100, p, p, p, 0, None, None) == -1
    assert lib.vsd_advance_lengths(4, 5, p, 100, p, p, p, 3, None, None) == -1
    assert lib.vsd_advance_lengths(-1, 5, p, 100, p, p, p, 0, None, None) == -1
    assert lib.vsd_advance_lengths(4, -1, p, 100, p, p, p, 0, None, None) == -1
    assert lib.vsd_advance_lengths(0, 5, None, 100, None, None, None, 0, None, None) == 0


def test_draft_step_rejects_bad_flags(lib):
    g = _geom()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)

    def call(flags, rows=p, k_new=None, v_new=None):
        return lib.vsd_sparse_decode_attn_step(ctypes.byref(g), p, k_new, v_new, p, p, p, p, p,
                                               16, p, p, 4, rows, ctypes.c_uint(flags),
                                               ctypes.c_float(0.088), p, None, 0, None)
    assert call(0x8) == -1            # unknown flag
    assert call(0x1 | 0x2) == -1      # record and reuse together
    assert call(0x2, rows=None) == -1  # reuse without the rows
    assert call(0x0, k_new=p) == -1   # k_new without v_new


def test_sparse_verify_rejects_bad_flags(lib):
    g = _geom()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) & ~255)
    rc = lib.vsd_sparse_verify_attn(ctypes.byref(g), 4, p, p, p, p, p, p, p, 16,
                                    ctypes.c_uint(0x8), ctypes.c_float(0.088), p, p, 1024, None)
    assert rc == -1


def test_scored_verify_rejects_bad_flags(lib):
    g = _geom()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) & ~255)

    def call(flags, k_new=None, v_new=None):
        return lib.vsd_verify_attn_collect_scored(ctypes.byref(g), 4, p, p, p, p, p, 0, 3, 1024,
                                                  ctypes.c_float(0.088), None, p, p, p, 0, 0,
                                                  ctypes.c_uint(flags), k_new, v_new, p, p, 1024,
                                                  None)
    assert call(0x1) == -1                # unknown flag
    assert call(0x0, k_new=p) == -1       # keys to store without their values
    assert call(0x0, v_new=p) == -1
