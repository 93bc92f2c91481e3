"""The C-ABI library loads without a GPU, exports every declared entry point,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from mixed_bit_kv_gb300 import rdkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return rdkv.lib()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(rdkv_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert len(declared) >= 15
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert set(rdkv.EXPORTED) <= declared


def test_version_and_struct_sizes(L):
    assert L.rdkv_version() >= 1
    assert ctypes.sizeof(rdkv.Shape) == 28
    assert ctypes.sizeof(rdkv.Sizes) == 56 + 4 * rdkv.COST_HEADS
    import numpy as np
    assert np.dtype(rdkv.HEAD_PLAN_DTYPE).itemsize == 128
    assert np.dtype(rdkv.PLAN_HEADER_DTYPE).itemsize == 96


def test_workspace_queries_are_host_only(L):
    s = rdkv.make_shape(1, 32768, 24, 8, 128, 128, "f16")
    assert L.rdkv_score_workspace_bytes(ctypes.byref(s)) > 0
    assert L.rdkv_allocate_workspace_bytes(ctypes.byref(s)) > 0
    assert L.rdkv_plan_bytes(ctypes.byref(s)) > 8 * 128
    assert L.rdkv_waterfill_workspace_bytes(4, 1000) > 0


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, rdkv.RDKV_ERR_UNSUPPORTED),
    ("h_q", 25, rdkv.RDKV_ERR_INVALID_ARG),
    ("window", 40000, rdkv.RDKV_ERR_INVALID_ARG),
    ("dtype", 7, rdkv.RDKV_ERR_UNSUPPORTED),
    ("h_q", 80, rdkv.RDKV_ERR_UNSUPPORTED),
])
def test_bad_shapes_are_rejected_before_any_launch(L, field, value, code):
    s = rdkv.make_shape(1, 32768, 24, 8, 128, 128, "f16")
    setattr(s, field, value)
    fake = ctypes.c_void_p(16)
    r = L.rdkv_score(ctypes.byref(s), fake, fake, fake, fake, fake, fake, fake, fake, 1 << 40, None)
    assert r == code
    assert L.rdkv_last_error_string()


def test_null_and_budget_errors(L):
    s = rdkv.make_shape(1, 1024, 4, 1, 64, 32, "f32")
    r = L.rdkv_score(ctypes.byref(s), None, None, None, None, None, None, None, None, 0, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    fake = ctypes.c_void_p(16)
    r = L.rdkv_waterfill(1, 10, fake, ctypes.c_float(float("nan")), fake, None, None, fake, 1 << 20, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    r = L.rdkv_waterfill(1, 10, fake, ctypes.c_float(-1.0), fake, None, None, fake, 1 << 20, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    r = L.rdkv_waterfill(1, 10, fake, ctypes.c_float(2.0), fake, None, None, fake, 8, None)
    assert r == rdkv.RDKV_ERR_WORKSPACE


def test_append_capacity_is_checked_on_the_host(L):
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    fake = ctypes.c_void_p(256)
    c = rdkv.CacheStruct(s, 256, None, None, 256, 256, None, 256, 8, 8, sizes)
    r = L.rdkv_append(ctypes.byref(c), fake, fake, None)
    assert r == rdkv.RDKV_ERR_CAPACITY
    assert c.len_c == 8


def test_decode_step_capacity_is_checked_on_the_host(L):
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    fake = ctypes.c_void_p(256)
    c = rdkv.CacheStruct(s, 256, None, None, 256, 256, None, 256, 8, 8, sizes)
    r = L.rdkv_decode_step(ctypes.byref(c), fake, fake, fake, fake, fake, 1 << 20, None)
    assert r == rdkv.RDKV_ERR_CAPACITY
    assert c.len_c == 8
    r = L.rdkv_decode_step(ctypes.byref(c), fake, None, fake, fake, fake, 1 << 20, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG


def test_binding_cache_object_on_host_memory(L):
    """The Python Cache wrapper builds its C struct and sizes its decode workspace without a GPU."""
    import torch
    s = rdkv.make_shape(2, 1000, 6, 2, 128, 40, "f16")
    plan = torch.zeros(L.rdkv_plan_bytes(ctypes.byref(s)), dtype=torch.uint8)
    sizes = rdkv.Sizes(4096, 64, 256, 200, 2048, 2048, 0, 4)
    c = rdkv.Cache(s, plan, sizes, 48, "cpu")
    assert c.c.len_dev == c.len_dev.data_ptr() and c.c.cap_c == 48 and c.len_c == 0
    ws = c.decode_workspace()
    assert ws.numel() >= L.rdkv_decode_workspace_bytes(ctypes.byref(c.c)) > 0
    assert c.decode_workspace() is ws
    assert c.fits(sizes) and not c.fits(rdkv.Sizes(1 << 30, 64, 256, 200, 2048, 2048, 0, 4))


def test_allocate_mode_argument_checks(L):
    s = rdkv.make_shape(1, 1024, 4, 1, 64, 32, "f32")
    fake = ctypes.c_void_p(256)
    f = ctypes.c_float
    r = L.rdkv_allocate_mode(ctypes.byref(s), 7, f(0), fake, fake, fake, fake, f(2), f(2), fake, fake, fake, fake,
                             fake, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"mode" in L.rdkv_last_error_string()
    r = L.rdkv_allocate_mode(ctypes.byref(s), rdkv.RDKV_ALLOC_TOPK, f(0), None, fake, fake, fake, f(2), f(2), fake,
                             fake, fake, fake, fake, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    r = L.rdkv_allocate_mode(ctypes.byref(s), rdkv.RDKV_ALLOC_THRESHOLD, f(float("nan")), fake, fake, fake, fake, f(2),
                             f(2), fake, fake, fake, fake, fake, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG


def test_recompress_argument_checks(L):
    """The zone-C re-compression calls reject bad arguments on the host, before any launch."""
    fake = ctypes.c_void_p(256)
    assert L.rdkv_merge_attn(0, fake, fake, 4, 64, fake, None, None) == rdkv.RDKV_ERR_INVALID_ARG
    assert L.rdkv_merge_attn(2, None, fake, 4, 64, fake, None, None) == rdkv.RDKV_ERR_INVALID_ARG
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    c = rdkv.CacheStruct(s, 256, None, None, 256, 256, None, 256, 32, 20, sizes)
    for n_move in (0, 21, 9):  # nothing, more than held, fewer than the rows that would stay
        assert L.rdkv_zone_c_take(ctypes.byref(c), n_move, fake, fake, None) == rdkv.RDKV_ERR_INVALID_ARG
    assert c.len_c == 20
    seg = rdkv.make_shape(1, 40, 4, 1, 64, 8, "f16")  # a segment has no window
    f = ctypes.c_float
    r = L.rdkv_recompress_score(ctypes.byref(seg), fake, fake, fake, rdkv.RDKV_F16, fake, 4, f(1), fake, fake, fake,
                                None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"window" in L.rdkv_last_error_string()
    seg = rdkv.make_shape(1, 40, 4, 1, 64, 0, "f16")
    r = L.rdkv_recompress_score(ctypes.byref(seg), fake, fake, fake, rdkv.RDKV_F16, fake, 0, f(1), fake, fake, fake,
                                None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    r = L.rdkv_recompress_score(ctypes.byref(seg), fake, fake, fake, rdkv.RDKV_F16, fake, 4, f(0), fake, fake, fake,
                                None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"weight_scale" in L.rdkv_last_error_string()
    r = L.rdkv_allocate_at_levels(ctypes.byref(seg), 2, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    r = L.rdkv_allocate_at_levels(ctypes.byref(seg), 0, None, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"levels" in L.rdkv_last_error_string()


def test_multi_decode_argument_checks(L):
    """The several-cache decode checks the list and the shared shape on the host."""
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    a = rdkv.CacheStruct(rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16"), 256, None, None, 256, 256, None, 256, 16, 8, sizes)
    b = rdkv.CacheStruct(rdkv.make_shape(1, 64, 4, 1, 128, 8, "f16"), 256, None, None, 256, 256, None, 256, 16, 8,
                         sizes)
    arr = (ctypes.POINTER(rdkv.CacheStruct) * 9)(*([ctypes.pointer(a)] * 9))
    fake = ctypes.c_void_p(256)
    assert L.rdkv_decode_multi_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), 9) == 0
    assert L.rdkv_decode_multi_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), 2) > 0
    r = L.rdkv_decode_attn_multi(ctypes.cast(arr, ctypes.c_void_p), 0, fake, fake, None, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    arr[1] = ctypes.pointer(b)
    r = L.rdkv_decode_attn_multi(ctypes.cast(arr, ctypes.c_void_p), 2, fake, fake, None, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"shape" in L.rdkv_last_error_string()
    # without plan costs on the host, several caches cannot be dealt
    arr[1] = ctypes.pointer(a)
    r = L.rdkv_decode_attn_multi(ctypes.cast(arr, ctypes.c_void_p), 2, fake, fake, None, fake, 1 << 30, None)
    assert r == rdkv.RDKV_ERR_UNSUPPORTED


def test_paged_zone_c_table_stride_is_checked(L):
    """A page table must cover cap_c rows: stride * 16 >= cap_c, checked before any launch."""
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    fake = ctypes.c_void_p(256)
    c = rdkv.CacheStruct(s, 256, None, None, 256, 256, None, 256, 40, 8, sizes, 256, 2)  # 2 pages: 32 rows < 40
    r = L.rdkv_append(ctypes.byref(c), fake, fake, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG and b"page table" in L.rdkv_last_error_string()
    assert c.len_c == 8


def test_allocate_requires_aligned_keys(L):
    # the channel passes read whole K rows with vector loads: a misaligned k is refused on the host
    s = rdkv.make_shape(1, 1024, 4, 1, 64, 32, "f16")
    fake = ctypes.c_void_p(256)
    ws = L.rdkv_allocate_workspace_bytes(ctypes.byref(s))
    r = L.rdkv_allocate(ctypes.byref(s), fake, fake, ctypes.c_void_p(258), ctypes.c_float(2.0), ctypes.c_float(2.0),
                        fake, fake, fake, fake, fake, fake, ws, None)
    assert r == rdkv.RDKV_ERR_INVALID_ARG
    assert b"aligned" in L.rdkv_last_error_string()


def test_timeout_selftest_rejects_a_non_positive_limit(L):
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sizes = rdkv.Sizes(0, 0, 0, 0, 0, 0, 0, 1)
    fake = ctypes.c_void_p(256)
    c = rdkv.CacheStruct(s, 256, None, None, 256, 256, None, 256, 8, 8, sizes)
    for limit in (0, -5):
        r = L.rdkv_decode_timeout_selftest(ctypes.byref(c), fake, fake, fake, 1 << 20, limit, None)
        assert r == rdkv.RDKV_ERR_INVALID_ARG
        assert b"wait_cycles" in L.rdkv_last_error_string()


def test_shape_workspace_query(L):
    s = rdkv.make_shape(1, 32768, 24, 8, 128, 128, "f16")
    assert L.rdkv_workspace_bytes(ctypes.byref(s), rdkv.RDKV_CALL_SCORE) == L.rdkv_score_workspace_bytes(ctypes.byref(s))
    assert L.rdkv_workspace_bytes(ctypes.byref(s), rdkv.RDKV_CALL_ALLOCATE) == \
        L.rdkv_allocate_workspace_bytes(ctypes.byref(s))
    assert L.rdkv_workspace_bytes(ctypes.byref(s), 99) == 0
    bad = rdkv.make_shape(1, 32768, 24, 8, 96, 128, "f16")
    assert L.rdkv_workspace_bytes(ctypes.byref(bad), rdkv.RDKV_CALL_SCORE) == 0
    # the decode bound covers the cache-exact query: group sizes 1, 3, 4, 8, both head sizes, batches up
    # to 8, plans with few and with many tiles (index slots) and zone-C capacities from 0 to 4096 rows
    for G in (1, 3, 4, 8):
        for D in (64, 128):
            for batch, h_kv in ((1, 1), (2, 4), (8, 8)):
                for slots, extra in ((0, 0), (32 * 7, 8), (32 * 5000, 300), (32 * 200000, 4096)):
                    shape = rdkv.make_shape(batch, 4096, G * h_kv, h_kv, D, 128, "f16")
                    n_heads = batch * h_kv
                    sizes = rdkv.Sizes(1 << 20, 64, slots, slots, 4096, 4096, 0, n_heads)
                    c = rdkv.CacheStruct(shape, 256, 256, 256, 256, 256, 256, 256, 128 + extra, 128, sizes)
                    exact = L.rdkv_decode_workspace_bytes(ctypes.byref(c))
                    assert exact > 0, (G, D, batch, slots)
                    assert L.rdkv_workspace_bytes(ctypes.byref(shape), rdkv.RDKV_CALL_DECODE) >= exact, \
                        (G, D, batch, h_kv, slots, extra)


def test_ragged_decode_argument_checks(L):
    """The ragged launch refuses, before any launch, lists it cannot serve: no sequence or more than
    eight, a cache of batch > 1, sequences with other heads, more than RDKV_COST_HEADS heads."""
    fake = ctypes.c_void_p(256)

    def cache(batch=1, h_q=8, h_kv=2, n=1000):
        s = rdkv.make_shape(batch, n, h_q, h_kv, 128, 32, "f16")
        sizes = rdkv.Sizes(4096, 0, 64, 64, 1024, 1024, 0, batch * h_kv)
        return rdkv.CacheStruct(s, 256, 256, 256, 256, 256, 256, 256, 40, 32, sizes)

    def arr(cs):
        a = (ctypes.POINTER(rdkv.CacheStruct) * len(cs))(*[ctypes.pointer(c) for c in cs])
        return ctypes.cast(a, ctypes.c_void_p)

    good = [cache(n=1000), cache(n=3000)]
    assert L.rdkv_decode_ragged_workspace_bytes(arr(good), 2) > 0
    for cs, n, code in (([], 0, rdkv.RDKV_ERR_INVALID_ARG),
                        ([cache()] * 9, 9, rdkv.RDKV_ERR_INVALID_ARG),
                        ([cache(), cache(batch=2)], 2, rdkv.RDKV_ERR_INVALID_ARG),
                        ([cache(), cache(h_q=16)], 2, rdkv.RDKV_ERR_INVALID_ARG),
                        ([cache(h_q=64, h_kv=16)] * 5, 5, rdkv.RDKV_ERR_UNSUPPORTED)):
        ptr = arr(cs) if cs else ctypes.c_void_p(0)
        assert L.rdkv_decode_ragged_workspace_bytes(ptr, n) == 0
        r = L.rdkv_decode_ragged(ptr, n, fake, fake, None, fake, 1 << 30, None)
        assert r == code, (n, r)


def test_allocate_pack_argument_checks(L):
    """The one-launch allocation and pack rejects bad arguments on the host, before any CUDA call."""
    s = rdkv.make_shape(1, 1024, 4, 1, 64, 32, "f16")
    need = L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(s), 0)
    assert need > 0 and L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(s), 1) >= need
    assert L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(s), 2) == 0
    sizes = rdkv.Sizes(4096, 64, 1024, 900, 2048, 2048, 0, 1)
    fake = ctypes.c_void_p(256)
    c = rdkv.CacheStruct(s, 256, 256, 256, 256, 256, 256, 256, 64, 0, sizes)
    f = ctypes.c_float

    def call(per_head=0, k=fake, bv=2.0, ws_bytes=need):
        return L.rdkv_allocate_pack(ctypes.byref(c), per_head, fake, fake, k, fake, f(bv), f(2.0), fake, fake, fake,
                                    fake, fake, ws_bytes, None)

    assert call(per_head=2) == rdkv.RDKV_ERR_INVALID_ARG
    assert call(bv=float("nan")) == rdkv.RDKV_ERR_INVALID_ARG
    assert call(k=None) == rdkv.RDKV_ERR_INVALID_ARG
    assert call(k=ctypes.c_void_p(264)) == rdkv.RDKV_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(ws_bytes=need - 1) == rdkv.RDKV_ERR_WORKSPACE
    assert c.len_c == 0
