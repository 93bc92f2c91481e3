"""Pins of the oracle's zone-C re-compression (reading R10) against facts it does not compute itself:
closed forms, invariants, library routines on special cases and brute force on tiny inputs.
CPU only."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle as O


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_attention_lse_matches_library_logsumexp():
    D = 16
    q, K, V = _rand(D, 1), _rand((37, D), 2, 1.5), _rand((37, D), 3)
    out, lse = O.attention_lse(q, K, V)
    s = K @ q / math.sqrt(D)
    assert abs(lse - logsumexp(s)) <= 1e-12 * max(1.0, abs(lse))
    np.testing.assert_allclose(out, O.attention(q, K, V), rtol=0, atol=1e-13)
    out0, lse0 = O.attention_lse(q, np.zeros((0, D)), np.zeros((0, D)))
    assert lse0 == -np.inf and np.all(out0 == 0)


def test_merge_of_disjoint_parts_equals_attention_over_the_union():
    """Softmax over a union of key sets from the parts' outputs and log-sum-exps (closed form)."""
    D = 8
    q = _rand(D, 4)
    K, V = _rand((50, D), 5, 2.0), _rand((50, D), 6)
    cuts = [0, 7, 7, 31, 50]  # includes an empty part
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = O.attention_lse(q, K[a:b], V[a:b])
        outs.append(o)
        lses.append(l)
    out, lse = O.merge_attention(np.stack(outs), np.array(lses))
    ref_out, ref_lse = O.attention_lse(q, K, V)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    assert abs(lse - ref_lse) <= 1e-12 * abs(ref_lse)
    # no keys anywhere: output 0, lse -inf
    out, lse = O.merge_attention(np.zeros((2, 1, D)), np.full((2, 1), -np.inf))
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_take_zone_c_round_trip():
    B, Hkv, cap, D = 2, 3, 12, 4
    zk = _rand((B, Hkv, cap, D), 7).astype(np.float16)
    zv = _rand((B, Hkv, cap, D), 8).astype(np.float16)
    cache = dict(zone_c_k=zk.copy(), zone_c_v=zv.copy(), len_c=10)
    k, v = O.take_zone_c(cache, 6)
    assert k.shape == (B, 6, Hkv, D) and cache["len_c"] == 4
    assert np.array_equal(k.transpose(0, 2, 1, 3), zk[:, :, :6]) and np.array_equal(v.transpose(0, 2, 1, 3), zv[:, :, :6])
    assert np.array_equal(cache["zone_c_k"][:, :, :4], zk[:, :, 6:10])
    assert np.array_equal(cache["zone_c_v"][:, :, :4], zv[:, :, 6:10])
    with pytest.raises(ValueError):
        O.take_zone_c(cache, 5)


def test_recent_weights_sum_to_queries_times_group():
    """With each query's lse taken over exactly the moved keys, every softmax row sums to 1:
    sum_t w_t = R * G per KV head."""
    n, R, Hq, Hkv, D = 23, 5, 6, 2, 16
    k, q = _rand((n, Hkv, D), 9, 1.5), _rand((R, Hq, D), 10)
    G = Hq // Hkv
    lse = np.array([[logsumexp(k[:, h // G, :] @ q[r, h] / math.sqrt(D)) for h in range(Hq)] for r in range(R)])
    w = O.recent_token_weights(k, q, lse)
    np.testing.assert_allclose(w.sum(axis=1), R * G, rtol=1e-12)
    # the scale multiplies every weight
    np.testing.assert_allclose(O.recent_token_weights(k, q, lse, 2.5), 2.5 * w, rtol=1e-15)


def test_recent_weights_brute_force():
    """Scalar loops on a tiny case."""
    n, R, Hq, Hkv, D = 3, 2, 4, 2, 3
    k, q = _rand((n, Hkv, D), 11), _rand((R, Hq, D), 12)
    lse = _rand((R, Hq), 13)
    w = O.recent_token_weights(k, q, lse)
    for j in range(Hkv):
        for t in range(n):
            tot = 0.0
            for r in range(R):
                for h in (2 * j, 2 * j + 1):
                    dot = sum(float(q[r, h, c]) * float(k[t, j, c]) for c in range(D))
                    tot += math.exp(dot / math.sqrt(D) - float(lse[r, h]))
            assert abs(w[j, t] - tot) <= 1e-12 * tot


def test_allocation_at_the_prefill_levels_reproduces_the_water_filling():
    """At the levels the water-filling found for a budget, the incremental rule gives the same
    widths (V and K) as the full allocation of section 2.2."""
    rng = np.random.default_rng(14)
    Hkv, Np, D = 2, 61, 8
    g = (rng.standard_normal((Hkv, Np)) ** 2).astype(np.float32)
    w_chan = (rng.random((Hkv, D)) + 0.1).astype(np.float32)
    k = rng.standard_normal((Np, Hkv, D)).astype(np.float32)
    full = O.allocate(g, w_chan, k, 3.0, 4.0)
    inc = O.allocate_at_levels(g, w_chan, k, full["lam_v"], full["lam_k"])
    assert np.array_equal(inc["bits_tok"], full["bits_tok"])
    assert np.array_equal(inc["bits_chan"], full["bits_chan"])
    assert np.array_equal(inc["g_chan"], full["g_chan"])


def test_allocation_at_extreme_levels():
    rng = np.random.default_rng(15)
    g = (rng.random((1, 9)) + 0.01).astype(np.float32)
    g[0, 3] = 0.0
    k = rng.standard_normal((9, 1, 4)).astype(np.float32)
    w_chan = np.ones((1, 4), np.float32)
    top = O.allocate_at_levels(g, w_chan, k, np.float32(0.0), np.float32(0.0))
    assert np.all(top["bits_tok"][0, g[0] > 0] == 16) and top["bits_tok"][0, 3] == 0
    none = O.allocate_at_levels(g, w_chan, k, np.float32(np.inf), np.float32(np.inf))
    assert np.all(none["bits_tok"] == 0) and np.all(none["bits_chan"] == 0)


def test_decode_lse_of_an_all_16_bit_cache_is_the_textbook_log_sum_exp():
    """All widths 16: the cache holds the fp16 keys exactly, so the lse is logsumexp of the fp16
    logits over prefix and window, and the output is decode()'s."""
    B, N, Hq, Hkv, D, W = 1, 40, 4, 2, 32, 8
    k = _rand((B, N, Hkv, D), 16).astype(np.float32)
    v = _rand((B, N, Hkv, D), 17).astype(np.float32)
    q = _rand((B, Hq, D), 18)
    bits_tok = np.full((B, Hkv, N - W), 16, np.uint8)
    bits_chan = np.full((B, Hkv, D), 16, np.uint8)
    cache = O.pack(k, v, bits_tok, bits_chan, W)
    out, lse = O.decode_lse(cache, q)
    np.testing.assert_allclose(out, O.decode(cache, q), rtol=0, atol=1e-13)
    kh = k.astype(np.float16).astype(np.float64)
    for h in range(Hq):
        s = kh[0, :, h // 2, :] @ q[0, h] / math.sqrt(D)
        assert abs(lse[0, h] - logsumexp(s)) <= 1e-10
