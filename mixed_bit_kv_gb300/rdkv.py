"""Python binding of librdkv (include/rdkv.h): the same entry points, argument marshalling only.

Torch supplies device memory and the current CUDA stream; every computation
runs in the library's CUDA kernels.  Loading fails loudly when the library is
missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librdkv.so")

RDKV_OK, RDKV_ERR_INVALID_ARG, RDKV_ERR_UNSUPPORTED, RDKV_ERR_CAPACITY = 0, 1, 2, 3
RDKV_ERR_CUDA, RDKV_ERR_TIMEOUT, RDKV_ERR_WORKSPACE = 4, 5, 6
RDKV_F16, RDKV_F32 = 0, 1
RDKV_ALLOC_POOLED, RDKV_ALLOC_PER_HEAD, RDKV_ALLOC_TOPK, RDKV_ALLOC_THRESHOLD = 0, 1, 2, 3

EXPORTED = (
    "rdkv_last_error_string", "rdkv_version", "rdkv_launch_count",
    "rdkv_score_workspace_bytes", "rdkv_score",
    "rdkv_waterfill_workspace_bytes", "rdkv_waterfill",
    "rdkv_plan_bytes", "rdkv_allocate_workspace_bytes", "rdkv_allocate", "rdkv_allocate_mode", "rdkv_plan_sizes",
    "rdkv_pack", "rdkv_append",
    "rdkv_decode_workspace_bytes", "rdkv_decode_attn", "rdkv_decode_step", "rdkv_decode_status",
    "rdkv_decode_attn_noalloc",
    "rdkv_decode_attn_lse", "rdkv_decode_step_lse", "rdkv_merge_attn", "rdkv_zone_c_take", "rdkv_recompress_score",
    "rdkv_allocate_at_levels", "rdkv_decode_multi_workspace_bytes", "rdkv_decode_attn_multi",
    "rdkv_decode_multi_status", "rdkv_zone_bounds", "rdkv_decode_timeout_selftest", "rdkv_workspace_bytes",
    "rdkv_decode_ragged_workspace_bytes", "rdkv_decode_ragged", "rdkv_decode_ragged_status",
    "rdkv_allocate_pack_workspace_bytes", "rdkv_allocate_pack",
)
RDKV_CALL_SCORE, RDKV_CALL_ALLOCATE, RDKV_CALL_DECODE = 0, 1, 2


class RDKVError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"rdkv status {code}: {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("batch", "n_tokens", "h_q", "h_kv", "head_dim", "window", "dtype")]


COST_HEADS = 64  # RDKV_COST_HEADS


class Sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("zone_a_bytes", "zone_b_rows", "index_slots", "kept_tokens",
                                               "max_tile_bytes", "max_stage_bytes")] + [
        ("status", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("head_cost", ctypes.c_int32 * COST_HEADS)]


class CacheStruct(ctypes.Structure):
    _fields_ = [("shape", Shape), ("plan", ctypes.c_void_p), ("zone_a", ctypes.c_void_p),
                ("zone_b", ctypes.c_void_p), ("zone_c_k", ctypes.c_void_p), ("zone_c_v", ctypes.c_void_p),
                ("index_map", ctypes.c_void_p), ("len_dev", ctypes.c_void_p), ("cap_c", ctypes.c_int32),
                ("len_c", ctypes.c_int32),
                ("sizes", Sizes), ("zone_c_pages", ctypes.c_void_p), ("zone_c_page_stride", ctypes.c_int32),
                ("zone_a_pages", ctypes.c_void_p), ("zone_b_pages", ctypes.c_void_p)]

PAGE_ROWS = 16  # RDKV_ZONE_C_PAGE_ROWS
A_PAGE_BYTES = 65536  # RDKV_ZONE_A_PAGE_BYTES
B_PAGE_ROWS = 16  # RDKV_ZONE_B_PAGE_ROWS


HEAD_PLAN_DTYPE = [("n_v", "<i4", 4), ("tiles", "<i4", 4), ("n_k", "<i4", 5), ("k_words", "<i4", 4),
                   ("row_words", "<i4"), ("k_slots", "<i4"), ("meta_slots", "<i4"), ("tile_bytes", "<i4", 4),
                   ("a_off", "<i8"), ("a_bytes", "<i8"), ("b_row", "<i8"), ("slot_off", "<i8")]
PLAN_HEADER_DTYPE = [("status", "<i4"), ("n_heads", "<i4"), ("batch", "<i4"), ("h_kv", "<i4"),
                     ("head_dim", "<i4"), ("slot_stride", "<i4"), ("heads_off", "<i8"), ("slots_off", "<i8"),
                     ("lambda_off", "<i8"), ("zone_a_bytes", "<i8"), ("zone_b_rows", "<i8"),
                     ("index_slots", "<i8"), ("kept_tokens", "<i8"), ("max_tile_bytes", "<i8"),
                     ("max_stage_bytes", "<i8")]

_lib = None
_P = ctypes.c_void_p


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RDKVError(-1, f"{LIB_PATH} is missing: build it with mixed_bit_kv_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        sp, szp, cp = ctypes.POINTER(Shape), ctypes.POINTER(Sizes), ctypes.POINTER(CacheStruct)
        sig = {
            "rdkv_last_error_string": (ctypes.c_char_p, []),
            "rdkv_version": (ctypes.c_int32, []),
            "rdkv_launch_count": (ctypes.c_uint64, []),
            "rdkv_score_workspace_bytes": (ctypes.c_size_t, [sp]),
            "rdkv_score": (ctypes.c_int, [sp, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_waterfill_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int64]),
            "rdkv_waterfill": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, _P, ctypes.c_float, _P, _P, _P, _P,
                                              ctypes.c_size_t, _P]),
            "rdkv_plan_bytes": (ctypes.c_size_t, [sp]),
            "rdkv_allocate_workspace_bytes": (ctypes.c_size_t, [sp]),
            "rdkv_allocate": (ctypes.c_int, [sp, _P, _P, _P, ctypes.c_float, ctypes.c_float, _P, _P, _P, _P, _P, _P,
                                             ctypes.c_size_t, _P]),
            "rdkv_allocate_mode": (ctypes.c_int, [sp, ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, ctypes.c_float,
                                                  ctypes.c_float, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_plan_sizes": (ctypes.c_int, [_P, szp, _P]),
            "rdkv_pack": (ctypes.c_int, [cp, _P, _P, _P, _P, _P]),
            "rdkv_append": (ctypes.c_int, [cp, _P, _P, _P]),
            "rdkv_decode_workspace_bytes": (ctypes.c_size_t, [cp]),
            "rdkv_decode_attn": (ctypes.c_int, [cp, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_decode_step": (ctypes.c_int, [cp, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_decode_status": (ctypes.c_int, [cp, _P, _P]),
            "rdkv_workspace_bytes": (ctypes.c_size_t, [sp, ctypes.c_int32]),
            "rdkv_decode_timeout_selftest": (ctypes.c_int, [cp, _P, _P, _P, ctypes.c_size_t, ctypes.c_int64, _P]),
            "rdkv_decode_attn_noalloc": (ctypes.c_int, [cp, _P, _P, _P]),
            "rdkv_decode_attn_lse": (ctypes.c_int, [cp, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_decode_step_lse": (ctypes.c_int, [cp, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_merge_attn": (ctypes.c_int, [ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
            "rdkv_zone_c_take": (ctypes.c_int, [cp, ctypes.c_int32, _P, _P, _P]),
            "rdkv_recompress_score": (ctypes.c_int, [sp, _P, _P, _P, ctypes.c_int32, _P, ctypes.c_int32,
                                                     ctypes.c_float, _P, _P, _P, _P]),
            "rdkv_zone_bounds": (ctypes.c_int, [sp, ctypes.c_float, ctypes.c_float, szp]),
            "rdkv_decode_multi_workspace_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32]),
            "rdkv_decode_attn_multi": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_decode_multi_status": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P]),
            "rdkv_allocate_at_levels": (ctypes.c_int, [sp, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                       ctypes.c_size_t, _P]),
            "rdkv_decode_ragged_workspace_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32]),
            "rdkv_decode_ragged": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "rdkv_decode_ragged_status": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P]),
            "rdkv_allocate_pack_workspace_bytes": (ctypes.c_size_t, [sp, ctypes.c_int32]),
            "rdkv_allocate_pack": (ctypes.c_int, [cp, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_float, ctypes.c_float,
                                                  _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(code):
    if code != RDKV_OK:
        raise RDKVError(code, lib().rdkv_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def make_shape(batch, n_tokens, h_q, h_kv, head_dim, window, dtype):
    code = RDKV_F16 if dtype in (torch.float16, "f16") else RDKV_F32
    return Shape(batch, n_tokens, h_q, h_kv, head_dim, window, code)


def shape_of(q, k, window):
    """Shape of prefill tensors q [B, N, H_q, D], k [B, N, H_kv, D]."""
    B, N, Hq, D = q.shape
    return make_shape(B, N, Hq, k.shape[2], D, window, q.dtype)


# ---------------------------------------------------------------- step 1
def rdkv_score(shape, q, k, v, stream=None, out=None, ws=None):
    """Outputs are allocated unless `out` (a dict from an earlier call) is given."""
    dev = q.device
    B, N, Hkv, D = shape.batch, shape.n_tokens, shape.h_kv, shape.head_dim
    Np = N - shape.window
    f32 = dict(dtype=torch.float32, device=dev)
    if out is None:
        out = dict(w_tok=torch.empty(B, Hkv, N, **f32), w_chan=torch.empty(B, Hkv, D, **f32),
                   sigma_tok=torch.empty(B, Hkv, N, **f32), g_tok=torch.empty(B, Hkv, max(Np, 0), **f32))
    L = lib()
    if ws is None:
        ws = _ws(L.rdkv_score_workspace_bytes(ctypes.byref(shape)), dev)
    _check(L.rdkv_score(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out["w_tok"]), _ptr(out["w_chan"]),
                        _ptr(out["sigma_tok"]), _ptr(out["g_tok"]), _ptr(ws), ws.numel(), _stream(stream)))
    return out


# ---------------------------------------------------------------- steps 2 and 3
def rdkv_waterfill(g, avg_bits, stream=None):
    """g [n_inst, n_units] fp32 on the GPU -> (bits uint8, lambda fp32 [n_inst], status int32 [1])."""
    n_inst, n_units = g.shape
    dev = g.device
    bits = torch.empty(n_inst, n_units, dtype=torch.uint8, device=dev)
    lam = torch.empty(n_inst, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    L = lib()
    ws = _ws(L.rdkv_waterfill_workspace_bytes(n_inst, n_units), dev)
    _check(L.rdkv_waterfill(n_inst, n_units, _ptr(g), float(avg_bits), _ptr(bits), _ptr(lam), _ptr(status),
                            _ptr(ws), ws.numel(), _stream(stream)))
    return bits, lam, status


def rdkv_allocate(shape, g_tok, w_chan, k, avg_bits_v, avg_bits_k, stream=None, out=None, ws=None):
    """Outputs (widths, spreads, gains and the plan buffer) are allocated unless `out` is given."""
    dev = k.device
    B, Hkv, D = shape.batch, shape.h_kv, shape.head_dim
    Np = shape.n_tokens - shape.window
    L = lib()
    if out is None:
        out = dict(bits_tok=torch.empty(B, Hkv, max(Np, 0), dtype=torch.uint8, device=dev),
                   sigma_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
                   g_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
                   bits_chan=torch.empty(B, Hkv, D, dtype=torch.uint8, device=dev),
                   plan=torch.zeros(L.rdkv_plan_bytes(ctypes.byref(shape)), dtype=torch.uint8, device=dev))
    if ws is None:
        ws = _ws(L.rdkv_allocate_workspace_bytes(ctypes.byref(shape)), dev)
    _check(L.rdkv_allocate(ctypes.byref(shape), _ptr(g_tok), _ptr(w_chan), _ptr(k), float(avg_bits_v),
                           float(avg_bits_k), _ptr(out["bits_tok"]), _ptr(out["sigma_chan"]), _ptr(out["g_chan"]),
                           _ptr(out["bits_chan"]), _ptr(out["plan"]), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rdkv_allocate_mode(shape, mode, w_tok, g_tok, w_chan, k, avg_bits_v, avg_bits_k, param=0.0, stream=None):
    """Allocation variant `mode` (RDKV_ALLOC_*): outputs as rdkv_allocate."""
    dev = k.device
    B, Hkv, D = shape.batch, shape.h_kv, shape.head_dim
    Np = shape.n_tokens - shape.window
    L = lib()
    out = dict(bits_tok=torch.empty(B, Hkv, max(Np, 0), dtype=torch.uint8, device=dev),
               sigma_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
               g_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
               bits_chan=torch.empty(B, Hkv, D, dtype=torch.uint8, device=dev),
               plan=torch.zeros(L.rdkv_plan_bytes(ctypes.byref(shape)), dtype=torch.uint8, device=dev))
    ws = _ws(L.rdkv_allocate_workspace_bytes(ctypes.byref(shape)), dev)
    _check(L.rdkv_allocate_mode(ctypes.byref(shape), int(mode), float(param), _ptr(w_tok), _ptr(g_tok), _ptr(w_chan),
                                _ptr(k), float(avg_bits_v), float(avg_bits_k), _ptr(out["bits_tok"]),
                                _ptr(out["sigma_chan"]), _ptr(out["g_chan"]), _ptr(out["bits_chan"]), _ptr(out["plan"]),
                                _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rdkv_plan_sizes(plan, stream=None):
    sz = Sizes()
    _check(lib().rdkv_plan_sizes(_ptr(plan), ctypes.byref(sz), _stream(stream)))
    return sz


# ---------------------------------------------------------------- TriZone cache
class Cache:
    """Device buffers of one packed TriZone cache plus the C struct that points at them."""

    def __init__(self, shape, plan, sizes, cap_c, device, pages=None, ab_pool=None):
        """pages: None for a contiguous zone C, else (pool_k, pool_v, table): fp16 pools
        [n_pages, PAGE_ROWS, D] and an int32 page table [B * H_kv, stride] (see ``page_pool``).
        ab_pool: None for contiguous zones A and B, else a ``ZonePool`` whose pages hold them."""
        D = shape.head_dim
        self.shape, self.plan, self.sizes = shape, plan, sizes
        self.ab_pool, self.a_table, self.b_table = ab_pool, None, None
        if ab_pool is None:
            self.zone_a = torch.zeros(max(sizes.zone_a_bytes, 16), dtype=torch.uint8, device=device)
            self.zone_b = torch.zeros(max(sizes.zone_b_rows, 1), D, dtype=torch.float16, device=device)
        else:
            self.zone_a, self.zone_b = ab_pool.zone_a, ab_pool.zone_b
            self.a_table, self.b_table = ab_pool.take(sizes)
        if pages is None:
            self.zone_c_k = torch.zeros(shape.batch, shape.h_kv, max(cap_c, 1), D, dtype=torch.float16, device=device)
            self.zone_c_v = torch.zeros_like(self.zone_c_k)
            self.pages, table_ptr, stride = None, None, 0
        else:
            self.zone_c_k, self.zone_c_v, self.pages = pages
            table_ptr, stride = self.pages.data_ptr(), self.pages.shape[1]
        self.index_map = torch.zeros(max(sizes.index_slots, 1), dtype=torch.int32, device=device)
        self.len_dev = torch.zeros(1, dtype=torch.int32, device=device)
        self.c = CacheStruct(shape, plan.data_ptr(), self.zone_a.data_ptr(), self.zone_b.data_ptr(),
                             self.zone_c_k.data_ptr(), self.zone_c_v.data_ptr(), self.index_map.data_ptr(),
                             self.len_dev.data_ptr(), cap_c, 0, sizes, table_ptr, stride,
                             None if self.a_table is None else self.a_table.data_ptr(),
                             None if self.b_table is None else self.b_table.data_ptr())
        self._ws = None

    def zone_a_bytes(self):
        """The cache's zone A as its logical bytes (gathered through the page table when paged)."""
        n = int(self.sizes.zone_a_bytes)
        if self.a_table is None:
            return self.zone_a[:n]
        o = torch.arange(n, device=self.zone_a.device)
        return self.zone_a[self.a_table[o // A_PAGE_BYTES].long() * A_PAGE_BYTES + o % A_PAGE_BYTES]

    def zone_b_rows(self):
        """The cache's zone-B rows [rows, D] (gathered through the page table when paged)."""
        n = int(self.sizes.zone_b_rows)
        if self.b_table is None:
            return self.zone_b[:n]
        r = torch.arange(n, device=self.zone_b.device)
        return self.zone_b.reshape(-1, self.shape.head_dim)[self.b_table[r // B_PAGE_ROWS].long() * B_PAGE_ROWS
                                                             + r % B_PAGE_ROWS]

    def release(self):
        """Returns the cache's zone-A and zone-B pages to its pool (the cache must not be used after)."""
        if self.ab_pool is not None and self.a_table is not None:
            self.ab_pool.give_back(self.a_table, self.b_table)
            self.a_table = self.b_table = None

    def zone_c_rows(self):
        """Zone C as logical rows: (k, v) fp16 [B, H_kv, cap_c, D], gathered through the page table."""
        s, cap = self.shape, self.c.cap_c
        if self.pages is None:
            return self.zone_c_k[:, :, :cap], self.zone_c_v[:, :, :cap]
        rows = torch.arange(cap, device=self.pages.device)
        phys = self.pages[:, rows // PAGE_ROWS].long() * PAGE_ROWS + rows % PAGE_ROWS  # [heads, cap]
        D = s.head_dim
        k = self.zone_c_k.reshape(-1, D)[phys].reshape(s.batch, s.h_kv, cap, D)
        v = self.zone_c_v.reshape(-1, D)[phys].reshape(s.batch, s.h_kv, cap, D)
        return k, v

    def fits(self, sizes):
        """True when a plan with these totals can be packed into this cache's buffers."""
        if self.ab_pool is not None:
            return False
        return (sizes.zone_a_bytes <= self.zone_a.numel() and sizes.zone_b_rows <= self.zone_b.shape[0]
                and sizes.index_slots <= self.index_map.numel())

    @property
    def len_c(self):
        return self.c.len_c

    def decode_workspace(self):
        """Zero-filled once; the decode leaves it ready for the next call."""
        nb = lib().rdkv_decode_workspace_bytes(ctypes.byref(self.c))
        if self._ws is None or self._ws.numel() < nb:
            self._ws = torch.zeros(max(int(nb), 256), dtype=torch.uint8, device=self.zone_a.device)
        return self._ws


def page_pool(shape, cap_c, device, extra_pages=0, seed=None):
    """A zone-C page pool for one cache: fp16 pools [n_pages, PAGE_ROWS, D] and the page table
    [B * H_kv, ceil(cap_c / PAGE_ROWS)] naming a distinct page per 16-row block (in a seeded random
    order when seed is given, to show that nothing depends on pages being adjacent)."""
    heads = shape.batch * shape.h_kv
    stride = max(1, -(-cap_c // PAGE_ROWS))
    n_pages = heads * stride + extra_pages
    order = torch.arange(n_pages)
    if seed is not None:
        order = order[torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))]
    table = order[:heads * stride].reshape(heads, stride).to(torch.int32).to(device)
    pool_k = torch.zeros(n_pages, PAGE_ROWS, shape.head_dim, dtype=torch.float16, device=device)
    return pool_k, torch.zeros_like(pool_k), table


class ZonePool:
    """Shared pools of zone-A pages (A_PAGE_BYTES each) and zone-B pages (B_PAGE_ROWS fp16 rows of D)
    for the caches of several sequences, with a host-side free list: ``take`` hands a cache the page
    tables its sizes need (distinct pages, in a seeded random order when seed is given, to show that
    nothing depends on pages being adjacent), ``give_back`` returns them."""

    def __init__(self, head_dim, a_pages, b_pages, device, seed=None):
        self.D = head_dim
        self.zone_a = torch.zeros(max(a_pages, 1) * A_PAGE_BYTES, dtype=torch.uint8, device=device)
        self.zone_b = torch.zeros(max(b_pages, 1) * B_PAGE_ROWS, head_dim, dtype=torch.float16, device=device)
        order_a, order_b = torch.arange(max(a_pages, 1)), torch.arange(max(b_pages, 1))
        if seed is not None:
            g = torch.Generator().manual_seed(seed)
            order_a, order_b = order_a[torch.randperm(order_a.numel(), generator=g)], order_b[
                torch.randperm(order_b.numel(), generator=g)]
        self.free_a, self.free_b = order_a.tolist(), order_b.tolist()
        self.device = device

    def take(self, sizes):
        na = max(1, -(-int(sizes.zone_a_bytes) // A_PAGE_BYTES))
        nb = max(1, -(-int(sizes.zone_b_rows) // B_PAGE_ROWS))
        if na > len(self.free_a) or nb > len(self.free_b):
            raise RDKVError(RDKV_ERR_CAPACITY, f"zone pool exhausted: {na} A pages, {nb} B pages wanted, "
                                               f"{len(self.free_a)}, {len(self.free_b)} free")
        ta, self.free_a = self.free_a[:na], self.free_a[na:]
        tb, self.free_b = self.free_b[:nb], self.free_b[nb:]
        return (torch.tensor(ta, dtype=torch.int32, device=self.device),
                torch.tensor(tb, dtype=torch.int32, device=self.device))

    def give_back(self, a_table, b_table):
        self.free_a += a_table.tolist()
        self.free_b += b_table.tolist()


def rdkv_pack(shape, plan, k, v, bits_tok, bits_chan, cap_c, stream=None, sizes=None, into=None, pages=None,
              ab_pool=None):
    """Packs into a new Cache (zone C paged when `pages` from ``page_pool`` is given; zones A and B in
    pages of `ab_pool`, a ``ZonePool``, when given), or into the buffers of `into` when they are large
    enough."""
    sizes = sizes if sizes is not None else rdkv_plan_sizes(plan, stream)
    if into is not None and into.fits(sizes) and into.c.cap_c == cap_c:
        cache = into
        cache.plan, cache.sizes = plan, sizes
        cache.c.plan, cache.c.sizes = plan.data_ptr(), sizes
    else:
        cache = Cache(shape, plan, sizes, cap_c, k.device, pages=pages, ab_pool=ab_pool)
    _check(lib().rdkv_pack(ctypes.byref(cache.c), _ptr(k), _ptr(v), _ptr(bits_tok), _ptr(bits_chan),
                           _stream(stream)))
    return cache


def rdkv_allocate_pack(shape, g_tok, w_chan, k, v, avg_bits_v, avg_bits_k, cap_c, per_head=False, stream=None,
                       out=None, ws=None, cache=None, pages=None):
    """Allocation and pack in one launch.  The zones are sized from rdkv_zone_bounds (a new Cache unless
    `cache`, built on those bounds, is given); the plan buffer is out["plan"].  Returns (out, cache):
    call ``finish_sizes`` (synchronising) before the decode so that the cache carries the exact
    totals."""
    dev = k.device
    B, Hkv, D = shape.batch, shape.h_kv, shape.head_dim
    Np = shape.n_tokens - shape.window
    L = lib()
    if out is None:
        out = dict(bits_tok=torch.empty(B, Hkv, max(Np, 0), dtype=torch.uint8, device=dev),
                   sigma_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
                   g_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
                   bits_chan=torch.empty(B, Hkv, D, dtype=torch.uint8, device=dev),
                   plan=torch.zeros(L.rdkv_plan_bytes(ctypes.byref(shape)), dtype=torch.uint8, device=dev))
    if ws is None:
        ws = _ws(L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(shape), int(per_head)), dev)
    if cache is None:
        cache = Cache(shape, out["plan"], rdkv_zone_bounds(shape, avg_bits_v, avg_bits_k), cap_c, dev, pages=pages)
    _check(L.rdkv_allocate_pack(ctypes.byref(cache.c), int(per_head), _ptr(g_tok), _ptr(w_chan), _ptr(k), _ptr(v),
                                float(avg_bits_v), float(avg_bits_k), _ptr(out["bits_tok"]), _ptr(out["sigma_chan"]),
                                _ptr(out["g_chan"]), _ptr(out["bits_chan"]), _ptr(ws), ws.numel(), _stream(stream)))
    return out, cache


def finish_sizes(cache, stream=None):
    """Reads the plan's exact totals (synchronising) into the cache, for the decode."""
    sizes = rdkv_plan_sizes(cache.plan, stream)
    cache.sizes = sizes
    cache.c.sizes = sizes
    return cache


def rdkv_append(cache, k_new, v_new, stream=None):
    _check(lib().rdkv_append(ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new), _stream(stream)))


def rdkv_decode_attn(cache, q, out=None, stream=None):
    B, Hq, D = q.shape
    out = out if out is not None else torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
    ws = cache.decode_workspace()
    _check(lib().rdkv_decode_attn(ctypes.byref(cache.c), _ptr(q), _ptr(out), _ptr(ws), ws.numel(),
                                  _stream(stream)))
    return out


def rdkv_decode_step(cache, q, k_new, v_new, out=None, stream=None):
    """One decode step in one launch: append (k_new, v_new) to zone C and attend with q over the cache."""
    B, Hq, D = q.shape
    out = out if out is not None else torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
    ws = cache.decode_workspace()
    _check(lib().rdkv_decode_step(ctypes.byref(cache.c), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _ptr(ws),
                                  ws.numel(), _stream(stream)))
    return out


def rdkv_decode_attn_noalloc(cache, q, out, stream=None):
    """Decode with the library's built-in scratch; `out` must be given (this path allocates nothing)."""
    _check(lib().rdkv_decode_attn_noalloc(ctypes.byref(cache.c), _ptr(q), _ptr(out), _stream(stream)))
    return out


def rdkv_decode_status(cache, stream=None):
    ws = cache.decode_workspace()
    return lib().rdkv_decode_status(ctypes.byref(cache.c), _ptr(ws), _stream(stream))


def rdkv_decode_timeout_selftest(cache, q, wait_cycles=2_000_000, stream=None):
    """The decode kernel with every stage armed for bytes no copy delivers: each bounded wait runs out
    after wait_cycles SM cycles and the status word reports RDKV_ERR_TIMEOUT (read it with
    rdkv_decode_status).  Returns the (meaningless) output tensor."""
    B, Hq, D = q.shape
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
    ws = cache.decode_workspace()
    _check(lib().rdkv_decode_timeout_selftest(ctypes.byref(cache.c), _ptr(q), _ptr(out), _ptr(ws), ws.numel(),
                                              int(wait_cycles), _stream(stream)))
    return out


# ---------------------------------------------------------------- plan inspection (tests)
def read_plan(plan):
    """Host view of a device plan buffer: header dict, head records, slot table, lambdas."""
    import numpy as np
    raw = plan.cpu().numpy()
    hdr = np.frombuffer(raw.tobytes(), dtype=np.dtype(PLAN_HEADER_DTYPE), count=1)[0]
    n = int(hdr["n_heads"])
    heads = np.frombuffer(raw.tobytes(), dtype=np.dtype(HEAD_PLAN_DTYPE), count=n, offset=int(hdr["heads_off"]))
    slots = np.frombuffer(raw.tobytes(), dtype="<i2", count=n * int(hdr["slot_stride"]),
                          offset=int(hdr["slots_off"])).reshape(n, int(hdr["slot_stride"]))
    lam = np.frombuffer(raw.tobytes(), dtype="<f4", count=2 * int(hdr["batch"]) * int(hdr["h_kv"]),
                        offset=int(hdr["lambda_off"]))
    return hdr, heads, slots, lam


# ---------------------------------------------------------------- zone-C re-compression
def rdkv_decode_attn_lse(cache, q, out=None, lse=None, stream=None):
    """rdkv_decode_attn plus the natural-log softmax denominator lse [B, H_q] of every query head."""
    B, Hq, D = q.shape
    out = out if out is not None else torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
    lse = lse if lse is not None else torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    ws = cache.decode_workspace()
    _check(lib().rdkv_decode_attn_lse(ctypes.byref(cache.c), _ptr(q), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                      _stream(stream)))
    return out, lse


def rdkv_decode_step_lse(cache, q, k_new, v_new, out=None, lse=None, stream=None):
    """rdkv_decode_step plus lse [B, H_q]."""
    B, Hq, D = q.shape
    out = out if out is not None else torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
    lse = lse if lse is not None else torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    ws = cache.decode_workspace()
    _check(lib().rdkv_decode_step_lse(ctypes.byref(cache.c), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _ptr(lse),
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def rdkv_merge_attn(outs, lses, out=None, lse=None, stream=None):
    """Attention over the union of disjoint key sets: outs [P, ..., D], lses [P, ...] fp32 (contiguous)."""
    P, D = outs.shape[0], outs.shape[-1]
    rows = lses[0].numel()
    out = out if out is not None else torch.empty(outs.shape[1:], dtype=torch.float32, device=outs.device)
    lse = lse if lse is not None else torch.empty(lses.shape[1:], dtype=torch.float32, device=outs.device)
    _check(lib().rdkv_merge_attn(P, _ptr(outs), _ptr(lses), rows, D, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def rdkv_zone_c_take(cache, n_move, stream=None):
    """Rows [0, n_move) of zone C out of the cache as k, v [B, n_move, H_kv, D] in the cache's dtype;
    the rest move to the front."""
    s = cache.shape
    dt = torch.float16 if s.dtype == RDKV_F16 else torch.float32
    k = torch.empty(s.batch, n_move, s.h_kv, s.head_dim, dtype=dt, device=cache.zone_c_k.device)
    v = torch.empty_like(k)
    _check(lib().rdkv_zone_c_take(ctypes.byref(cache.c), int(n_move), _ptr(k), _ptr(v), _stream(stream)))
    return k, v


def rdkv_recompress_score(seg_shape, k, v, q_recent, lse_recent, weight_scale=1.0, stream=None):
    """Token weights, V spreads and gains [B, H_kv, n] of moved tokens from recent queries
    q_recent [B, R, H_q, D] and their decode lse [B, R, H_q], weights times weight_scale."""
    B, n, Hkv = seg_shape.batch, seg_shape.n_tokens, seg_shape.h_kv
    dev = k.device
    out = {name: torch.empty(B, Hkv, n, dtype=torch.float32, device=dev) for name in ("w_tok", "sigma_tok", "g_tok")}
    qd = RDKV_F16 if q_recent.dtype == torch.float16 else RDKV_F32
    _check(lib().rdkv_recompress_score(ctypes.byref(seg_shape), _ptr(k), _ptr(v), _ptr(q_recent), qd, _ptr(lse_recent),
                                       int(q_recent.shape[1]), ctypes.c_float(weight_scale), _ptr(out["w_tok"]),
                                       _ptr(out["sigma_tok"]),
                                       _ptr(out["g_tok"]), _stream(stream)))
    return out


def plan_levels(plan):
    """Device view of a plan's water levels: float32 [2, n_inst] (V levels, then K levels)."""
    import numpy as np
    raw = plan[:256].cpu().numpy()
    hdr = np.frombuffer(raw.tobytes(), dtype=np.dtype(PLAN_HEADER_DTYPE), count=1)[0]
    n = 2 * int(hdr["batch"]) * int(hdr["h_kv"])
    off = int(hdr["lambda_off"])
    return plan[off:off + 4 * n].view(torch.float32)


def rdkv_allocate_at_levels(seg_shape, levels, g_tok, w_chan, k, per_head=False, stream=None):
    """Widths of a segment at given water levels [2, n_inst] (n_inst = batch, or batch * h_kv per head);
    outputs as rdkv_allocate."""
    dev = k.device
    B, Hkv, D, n = seg_shape.batch, seg_shape.h_kv, seg_shape.head_dim, seg_shape.n_tokens
    L = lib()
    out = dict(bits_tok=torch.empty(B, Hkv, n, dtype=torch.uint8, device=dev),
               sigma_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
               g_chan=torch.empty(B, Hkv, D, dtype=torch.float32, device=dev),
               bits_chan=torch.empty(B, Hkv, D, dtype=torch.uint8, device=dev),
               plan=torch.zeros(L.rdkv_plan_bytes(ctypes.byref(seg_shape)), dtype=torch.uint8, device=dev))
    ws = _ws(L.rdkv_allocate_workspace_bytes(ctypes.byref(seg_shape)), dev)
    _check(L.rdkv_allocate_at_levels(ctypes.byref(seg_shape), int(bool(per_head)), _ptr(levels), _ptr(g_tok),
                                     _ptr(w_chan), _ptr(k), _ptr(out["bits_tok"]), _ptr(out["sigma_chan"]),
                                     _ptr(out["g_chan"]), _ptr(out["bits_chan"]), _ptr(out["plan"]), _ptr(ws), ws.numel(),
                                     _stream(stream)))
    return out


def recompress(live, prefill_plan, w_chan, q_recent, lse_recent, n_move, per_head=False, stream=None):
    """Moves the oldest n_move zone-C rows of `live` into a new segment (a Cache with window 0):
    weights from the recent queries and their decode lse, widths at the water levels of
    `prefill_plan` (the plan the prefill allocation wrote), the prefill's channel weights w_chan."""
    k, v = rdkv_zone_c_take(live, n_move, stream)
    return recompress_from_rows(live, k, v, prefill_plan, w_chan, q_recent, lse_recent, per_head, stream)


def recompress_from_rows(live, k, v, prefill_plan, w_chan, q_recent, lse_recent, per_head=False, stream=None):
    """The segment of rows k, v [B, n, H_kv, D] already taken out of `live` (rdkv_zone_c_take)."""
    s = live.shape
    n_move = k.shape[1]
    seg = Shape(s.batch, int(n_move), s.h_q, s.h_kv, s.head_dim, 0, s.dtype)
    # a prefill weight sums the attention of up to N query rows: the recent sums are scaled by N / R
    sc = rdkv_recompress_score(seg, k, v, q_recent, lse_recent, s.n_tokens / q_recent.shape[1], stream)
    al = rdkv_allocate_at_levels(seg, plan_levels(prefill_plan), sc["g_tok"], w_chan, k, per_head, stream)
    cache = rdkv_pack(seg, al["plan"], k, v, al["bits_tok"], al["bits_chan"], 0, stream)
    cache._keep = (sc, al)
    return cache


def decode_segments(segments, live, q, stream=None):
    """Attention of q [B, H_q, D] over the segments' zones A and B and the live cache (its zones and
    zone C), merged: (out [B, H_q, D], lse [B, H_q])."""
    parts = list(segments) + [live]
    B, Hq, D = q.shape
    outs = torch.empty(len(parts), B, Hq, D, dtype=torch.float32, device=q.device)
    lses = torch.empty(len(parts), B, Hq, dtype=torch.float32, device=q.device)
    for i, c in enumerate(parts):
        rdkv_decode_attn_lse(c, q, out=outs[i], lse=lses[i], stream=stream)
    return rdkv_merge_attn(outs, lses, stream=stream)


class MultiDecode:
    """One launch over several caches (segments, then the live cache): keeps the array of their C
    structs and the zero-filled workspace the list needs."""

    def __init__(self, parts):
        self.parts = list(parts)
        self._arr = (ctypes.POINTER(CacheStruct) * len(self.parts))(*[ctypes.pointer(c.c) for c in self.parts])
        self._ws = None

    def workspace(self):
        nb = lib().rdkv_decode_multi_workspace_bytes(ctypes.cast(self._arr, _P), len(self.parts))
        if nb == 0:
            _check(RDKV_ERR_INVALID_ARG)
        if self._ws is None or self._ws.numel() < nb:
            self._ws = torch.zeros(max(int(nb), 256), dtype=torch.uint8, device=self.parts[0].zone_a.device)
        return self._ws

    def attn(self, q, out=None, lse=None, stream=None):
        B, Hq, D = q.shape
        out = out if out is not None else torch.empty(B, Hq, D, dtype=torch.float32, device=q.device)
        lse = lse if lse is not None else torch.empty(B, Hq, dtype=torch.float32, device=q.device)
        ws = self.workspace()
        _check(lib().rdkv_decode_attn_multi(ctypes.cast(self._arr, _P), len(self.parts), _ptr(q), _ptr(out), _ptr(lse),
                                            _ptr(ws), ws.numel(), _stream(stream)))
        return out, lse

    def status(self, stream=None):
        return lib().rdkv_decode_multi_status(ctypes.cast(self._arr, _P), len(self.parts), _ptr(self.workspace()),
                                              _stream(stream))


# ---------------------------------------------------------------- compression without synchronisation
class RaggedDecode:
    """One decode launch over the sequences of a ragged batch (rdkv_decode_ragged): caches of batch 1
    with their own prompt lengths (zones often in one ZonePool), queries q [n_seq, H_q, D]."""

    def __init__(self, seqs):
        self.seqs = list(seqs)
        self._arr = (ctypes.POINTER(CacheStruct) * len(self.seqs))(*[ctypes.pointer(c.c) for c in self.seqs])
        self._ws = None

    def workspace(self):
        nb = lib().rdkv_decode_ragged_workspace_bytes(ctypes.cast(self._arr, _P), len(self.seqs))
        if nb == 0:
            raise RDKVError(RDKV_ERR_INVALID_ARG, lib().rdkv_last_error_string().decode())
        if self._ws is None or self._ws.numel() < nb:
            self._ws = torch.zeros(int(nb), dtype=torch.uint8, device=self.seqs[0].zone_a.device)
        return self._ws

    def attn(self, q, out=None, lse=None, stream=None):
        n, Hq, D = q.shape
        out = out if out is not None else torch.empty(n, Hq, D, dtype=torch.float32, device=q.device)
        ws = self.workspace()
        _check(lib().rdkv_decode_ragged(ctypes.cast(self._arr, _P), len(self.seqs), _ptr(q), _ptr(out), _ptr(lse),
                                        _ptr(ws), ws.numel(), _stream(stream)))
        return out

    def status(self, stream=None):
        return lib().rdkv_decode_ragged_status(ctypes.cast(self._arr, _P), len(self.seqs), _ptr(self.workspace()),
                                               _stream(stream))


def rdkv_zone_bounds(shape, avg_bits_v, avg_bits_k):
    """Upper bounds of the plan totals (host arithmetic only)."""
    sz = Sizes()
    _check(lib().rdkv_zone_bounds(ctypes.byref(shape), ctypes.c_float(avg_bits_v), ctypes.c_float(avg_bits_k),
                                  ctypes.byref(sz)))
    return sz


class Compressor:
    """Weights, allocation and pack of one prefill shape as one stream-ordered sequence with every
    buffer allocated up front (zones sized by rdkv_zone_bounds): run() neither allocates nor waits
    for the device, so it can be captured in a CUDA graph; finish() reads the exact plan totals
    (synchronising) so that the decode sizes its work from them."""

    def __init__(self, shape, avg_bits_v, avg_bits_k, cap_c, device, pages=None, fused=False):
        """fused: allocation and pack as one persistent launch (rdkv_allocate_pack) instead of the
        allocation's and the pack's own kernels."""
        self.shape, self.avg, self.fused = shape, (float(avg_bits_v), float(avg_bits_k)), fused
        self.bounds = rdkv_zone_bounds(shape, avg_bits_v, avg_bits_k)
        L = lib()
        B, Hkv, D, N = shape.batch, shape.h_kv, shape.head_dim, shape.n_tokens
        Np = N - shape.window
        f32 = dict(dtype=torch.float32, device=device)
        self.score_out = dict(w_tok=torch.empty(B, Hkv, N, **f32), w_chan=torch.empty(B, Hkv, D, **f32),
                              sigma_tok=torch.empty(B, Hkv, N, **f32), g_tok=torch.empty(B, Hkv, max(Np, 0), **f32))
        self.score_ws = _ws(L.rdkv_score_workspace_bytes(ctypes.byref(shape)), device)
        self.alloc_out = dict(bits_tok=torch.empty(B, Hkv, max(Np, 0), dtype=torch.uint8, device=device),
                              sigma_chan=torch.empty(B, Hkv, D, **f32), g_chan=torch.empty(B, Hkv, D, **f32),
                              bits_chan=torch.empty(B, Hkv, D, dtype=torch.uint8, device=device),
                              plan=torch.zeros(L.rdkv_plan_bytes(ctypes.byref(shape)), dtype=torch.uint8,
                                               device=device))
        self.alloc_ws = _ws(L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(shape), 0) if fused
                            else L.rdkv_allocate_workspace_bytes(ctypes.byref(shape)), device)
        self.cache = Cache(shape, self.alloc_out["plan"], self.bounds, cap_c, device, pages=pages)

    def run(self, q, k, v, stream=None):
        s, L = self.shape, lib()
        so, ao = self.score_out, self.alloc_out
        _check(L.rdkv_score(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(so["w_tok"]), _ptr(so["w_chan"]),
                            _ptr(so["sigma_tok"]), _ptr(so["g_tok"]), _ptr(self.score_ws), self.score_ws.numel(),
                            _stream(stream)))
        self.cache.c.sizes = self.bounds
        if self.fused:
            rdkv_allocate_pack(s, so["g_tok"], so["w_chan"], k, v, self.avg[0], self.avg[1], self.cache.c.cap_c,
                               stream=stream, out=ao, ws=self.alloc_ws, cache=self.cache)
            return self.cache
        _check(L.rdkv_allocate(ctypes.byref(s), _ptr(so["g_tok"]), _ptr(so["w_chan"]), _ptr(k),
                               ctypes.c_float(self.avg[0]), ctypes.c_float(self.avg[1]), _ptr(ao["bits_tok"]),
                               _ptr(ao["sigma_chan"]), _ptr(ao["g_chan"]), _ptr(ao["bits_chan"]), _ptr(ao["plan"]),
                               _ptr(self.alloc_ws), self.alloc_ws.numel(), _stream(stream)))
        _check(L.rdkv_pack(ctypes.byref(self.cache.c), _ptr(k), _ptr(v), _ptr(ao["bits_tok"]), _ptr(ao["bits_chan"]),
                           _stream(stream)))
        return self.cache

    def finish(self, stream=None):
        sizes = rdkv_plan_sizes(self.alloc_out["plan"], stream)
        self.cache.sizes = sizes
        self.cache.c.sizes = sizes
        return self.cache
