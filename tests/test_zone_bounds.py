"""rdkv_zone_bounds (host arithmetic of the library, no GPU) against the exact plan totals the oracle's
allocation and plan produce: every bound holds for random gains, ragged shapes, extreme budgets and
both the pooled and the per-head allocation."""
import ctypes

import numpy as np
import pytest

import oracle as O
from mixed_bit_kv_gb300 import rdkv


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return rdkv.lib()


def _bounds(L, B, N, Hq, Hkv, D, W, av, ak):
    s = rdkv.make_shape(B, N, Hq, Hkv, D, W, "f16")
    return rdkv.rdkv_zone_bounds(s, av, ak)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("budget", [0.0, 0.4, 2.5, 5.0, 16.0])
def test_bounds_hold_for_random_allocations(L, seed, budget):
    rng = np.random.default_rng(100 * seed + int(budget * 10))
    B, Hkv, D = 2, int(rng.integers(1, 4)), int(rng.choice([64, 128]))
    N = int(rng.integers(40, 700))
    W = int(rng.integers(0, min(N, 60)))
    Np = N - W
    bounds = _bounds(L, B, N, 2 * Hkv, Hkv, D, W, budget, budget)
    for per_head in (False, True):
        bits_tok = np.zeros((B, Hkv, Np), np.uint8)
        bits_chan = np.zeros((B, Hkv, D), np.uint8)
        for b in range(B):
            g = (rng.standard_normal((Hkv, Np)) ** 2 * rng.choice([1e-3, 1.0, 1e3])).astype(np.float32)
            w_chan = (rng.random((Hkv, D)) + 0.01).astype(np.float32)
            k = rng.standard_normal((Np, Hkv, D)).astype(np.float32)
            al = (O.allocate_per_head if per_head else O.allocate)(g, w_chan, k, budget, budget)
            bits_tok[b], bits_chan[b] = al["bits_tok"], al["bits_chan"]
        plan = O.make_plan(bits_tok, bits_chan, D)
        assert plan["zone_a_bytes"] <= bounds.zone_a_bytes
        assert plan["zone_b_rows"] <= bounds.zone_b_rows
        assert plan["index_slots"] <= bounds.index_slots
        assert plan["kept_tokens"] <= bounds.kept_tokens
        assert plan["max_tile_bytes"] <= bounds.max_tile_bytes
        assert plan["max_stage_bytes"] <= bounds.max_stage_bytes


def test_bounds_of_the_widest_allocations(L):
    """All 16 bits (every token in zone B, every K channel raw) and all 8 bits are within the bounds."""
    B, N, Hkv, D, W = 1, 300, 2, 128, 20
    Np = N - W
    bounds = _bounds(L, B, N, 4, Hkv, D, W, 16.0, 16.0)
    for vb, kb in ((16, 16), (8, 8), (8, 16), (16, 2)):
        plan = O.make_plan(np.full((B, Hkv, Np), vb, np.uint8), np.full((B, Hkv, D), kb, np.uint8), D)
        for key in ("zone_a_bytes", "zone_b_rows", "index_slots", "max_tile_bytes", "max_stage_bytes"):
            assert plan[key] <= getattr(bounds, key), (vb, kb, key)
    assert bounds.n_heads == B * Hkv and bounds.status == 0


def test_bounds_reject_bad_budgets(L):
    s = rdkv.make_shape(1, 64, 4, 1, 64, 8, "f16")
    sz = rdkv.Sizes()
    assert L.rdkv_zone_bounds(ctypes.byref(s), ctypes.c_float(-1), ctypes.c_float(2), ctypes.byref(sz)) == \
        rdkv.RDKV_ERR_INVALID_ARG
