"""Pins of the CPU oracle against facts it does not compute itself.

Each test ties one oracle function to a closed form, an invariant, a special
case that reduces to a library routine, a value the pages print, or brute
force on tiny inputs.  They run on the CPU (no GPU marker).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- KV-size formula
def test_kv_size_formula_page_values():
    pins = json.load(open(os.path.join(GOLDEN, "kv_size_pins.json")))
    for c in pins["cases"]:
        got = O.kv_cache_bytes(c["L"], c["H_kv"], c["D"], c["P"], c["N"])
        assert got == c["bytes"], c["what"]
        if "gib_3dp" in c:
            assert round(got / 1024 ** 3, 3) == c["gib_3dp"], c["what"]


# ---------------------------------------------------------------- token weights
def test_token_weights_rows_sum_to_one():
    """Every causal softmax row sums to 1, so sum_t w_t = N * G per KV head."""
    N, Hq, Hkv, D = 67, 6, 2, 16
    q, k = _rand((N, Hq, D), 1), _rand((N, Hkv, D), 2, 2.0)
    w = O.token_weights(q, k, row_block=20)
    np.testing.assert_allclose(w.sum(axis=1), N * (Hq // Hkv), rtol=1e-12)


def test_token_weights_equal_keys_harmonic():
    """Equal logits: row tau spreads 1/(tau+1) over t <= tau, so w_t = G * (H_N - H_t)."""
    N, Hq, Hkv, D = 40, 4, 1, 8
    q = _rand((N, Hq, D), 3)
    k = np.tile(_rand((1, Hkv, D), 4), (N, 1, 1))
    w = O.token_weights(q, k)
    harm = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, N + 1))])
    expect = Hq * (harm[N] - harm[np.arange(N)])
    np.testing.assert_allclose(w[0], expect, rtol=1e-12)


def test_token_weights_match_sdpa_column_sums():
    """With V = identity, causal SDPA returns the attention matrix itself (torch library routine)."""
    N, Hq, Hkv, D = 33, 6, 2, 16
    G = Hq // Hkv
    q, k = _rand((N, Hq, D), 5), _rand((N, Hkv, D), 6, 1.5)
    qt = torch.tensor(q).permute(1, 0, 2)[None]                       # [1, Hq, N, D]
    kt = torch.tensor(k).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    eye = torch.eye(N, dtype=torch.float64).expand(1, Hq, N, N)
    A = torch.nn.functional.scaled_dot_product_attention(qt, kt, eye, is_causal=True)[0]   # [Hq, N, N]
    expect = A.sum(dim=1).reshape(Hkv, G, N).sum(dim=1).numpy()
    np.testing.assert_allclose(O.token_weights(q, k, row_block=7), expect, rtol=1e-10, atol=1e-13)


def test_token_weights_tail_is_exact():
    N, Hq, Hkv, D = 50, 2, 1, 8
    q, k = _rand((N, Hq, D), 7), _rand((N, Hkv, D), 8)
    full = O.token_weights(q, k)
    tail = O.token_weights(q, k, first_row=37)
    np.testing.assert_allclose(tail[:, 37:], full[:, 37:], rtol=1e-12)


def test_row_lse_zero_query_and_normalisation():
    N, Hq, Hkv, D = 30, 2, 1, 8
    k = _rand((N, Hkv, D), 9)
    q = np.zeros((N, Hq, D))
    rows = [0, 5, 29]
    np.testing.assert_allclose(O.row_lse(q, k, 1, rows), np.log(np.array(rows) + 1.0), rtol=1e-13)
    q = _rand((N, Hq, D), 10)
    lse = O.row_lse(q, k, 0, [17])[0]
    s = q[17, 0] @ k[:18, 0].T / math.sqrt(D)
    assert abs(np.exp(s - lse).sum() - 1.0) < 1e-13


# ---------------------------------------------------------------- channel weights
def test_channel_weights_closed_form():
    """Constant columns: ||Q_c|| = sqrt(N*G)*|a_c|, ||K_c|| = sqrt(N)*|b_c|."""
    N, Hq, Hkv, D = 20, 6, 2, 8
    a = _rand((Hq, D), 11)
    b = _rand((Hkv, D), 12)
    G = Hq // Hkv
    q = np.tile(a[None], (N, 1, 1))
    k = np.tile(b[None], (N, 1, 1))
    w = O.channel_weights(q, k)
    qn = np.sqrt(N * (a.reshape(Hkv, G, D) ** 2).sum(axis=1))
    expect = qn * math.sqrt(N) * np.abs(b) / math.sqrt(D)
    np.testing.assert_allclose(w, expect, rtol=1e-13)


def test_channel_weights_library_norms():
    N, Hq, Hkv, D = 25, 4, 2, 8
    q, k = _rand((N, Hq, D), 13), _rand((N, Hkv, D), 14)
    w = O.channel_weights(q, k)
    for j in range(Hkv):
        Qj = q[:, 2 * j:2 * j + 2, :].reshape(-1, D)
        for c in range(D):
            e = np.linalg.norm(Qj[:, c]) * np.linalg.norm(k[:, j, c]) / math.sqrt(D)
            assert abs(w[j, c] - e) <= 1e-13 * e


# ---------------------------------------------------------------- sigma and gains
def test_value_spread_library_and_closed_form():
    v = _rand((9, 3, 16), 15)
    np.testing.assert_allclose(O.value_spread(v), np.std(v, axis=2).T, rtol=1e-13)
    row = np.array([2.5, -2.5] * 8).reshape(1, 1, 16) + 7.0
    assert abs(O.value_spread(row)[0, 0] - 2.5) < 1e-14


def test_token_gains_are_float32_products():
    w = np.array([[1.0 / 3.0, 2.0]])
    s = np.array([[3.0, 0.1]])
    g = O.token_gains(w, s, 2)
    assert g.dtype == np.float32
    assert g[0, 0] == np.float32(np.float32(1 / 3) * np.float32(3.0))
    assert g[0, 1] == np.float32(np.float32(2.0) * np.float32(0.1))


# ---------------------------------------------------------------- water-filling
def test_slopes_exact():
    assert SLOPES_EXPECTED == [float(s) for s in O.SLOPES]


SLOPES_EXPECTED = [0.375, 0.09375, 0.0146484375, 255.0 / 524288.0]


def _distortion(g, bits):
    return float(np.sum(np.asarray(g, np.float64) * 2.0 ** -np.asarray(bits, np.float64)))


def _mckp_brute_force(g, budget):
    best = math.inf
    for choice in itertools.product(O.WIDTHS.tolist(), repeat=len(g)):
        if sum(choice) <= budget:
            best = min(best, _distortion(g, choice))
    return best


@pytest.mark.parametrize("seed", range(12))
def test_waterfill_optimal_against_brute_force(seed):
    """The Lagrangian solution is optimal for the budget it spends (brute force over 5**U choices)."""
    rng = np.random.default_rng(100 + seed)
    U = int(rng.integers(2, 7))
    g = (rng.lognormal(0.0, 2.0, U)).astype(np.float32)
    avg = float(rng.uniform(0.0, 12.0))
    bits, lam = O.waterfill(g, avg)
    spent = int(bits.astype(np.int64).sum())
    assert spent <= O.budget_bits(avg, U)
    assert _distortion(g, bits) <= _mckp_brute_force(g, spent) * (1 + 1e-6)


def test_waterfill_special_budgets():
    g = np.array([0.5, 3.0, 0.0, 7.0], np.float32)
    bits, lam = O.waterfill(g, 16.0)
    assert bits.tolist() == [16, 16, 0, 16] and lam == 0.0
    bits, lam = O.waterfill(g, 0.0)
    assert bits.tolist() == [0, 0, 0, 0]
    assert lam == np.float32(7.0) * O.SLOPES[0]            # the largest breakpoint


def test_waterfill_hand_example():
    """Two equal units, 2 bits each on average: both take 2 bits at lambda = g * 0.09375."""
    bits, lam = O.waterfill(np.array([1.0, 1.0], np.float32), 2.0)
    assert bits.tolist() == [2, 2] and lam == np.float32(0.09375)


@pytest.mark.parametrize("seed", range(5))
def test_waterfill_lambda_is_minimal_and_monotone(seed):
    rng = np.random.default_rng(200 + seed)
    g = rng.lognormal(0, 1.5, 300).astype(np.float32)
    g[rng.integers(0, 300, 20)] = 0.0
    prev = None
    for avg in (0.0, 0.7, 1.9, 2.5, 4.0, 9.0, 15.9, 16.0):
        bits, lam = O.waterfill(g, avg)
        B = O.budget_bits(avg, g.size)
        beta = O.breakpoints(g)
        assert int(bits.astype(np.int64).sum()) <= B
        if lam > 0:
            below = np.nextafter(lam, np.float32(0))
            assert int(O.widths_at(beta, below).astype(np.int64).sum()) > B
        assert np.all(bits[g == 0] == 0)
        if prev is not None:
            assert np.all(bits >= prev)
        prev = bits


def test_kept_channel_spread_library():
    k = _rand((12, 2, 8), 16)
    bits = np.array([[0, 2, 4, 0, 16, 8, 0, 0, 2, 2], [0] * 10], np.uint8)
    s = O.kept_channel_spread(k, bits)
    kept = np.nonzero(bits[0])[0]
    np.testing.assert_allclose(s[0], np.std(k[kept, 0, :], axis=0), rtol=1e-13)
    assert np.all(s[1] == 0)


# ---------------------------------------------------------------- quantiser
def test_quantizer_closed_form_and_rounding():
    codes, sc, ze = O.quantize_groups(np.array([0.0, 1.0, 2.0, 3.0], np.float32), 2)
    assert codes.tolist() == [0, 1, 2, 3] and float(sc) == 1.0 and float(ze) == 0.0
    # ties go to even: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2
    codes, sc, ze = O.quantize_groups(np.array([0.0, 0.5, 1.5, 2.5, 3.0], np.float32), 2)
    assert codes.tolist() == [0, 0, 2, 2, 3]
    codes, sc, ze = O.quantize_groups(np.full(32, 1.25, np.float32), 4)
    assert codes.tolist() == [0] * 32 and float(sc) == 0.0 and float(ze) == 1.25


@pytest.mark.parametrize("b", [2, 4, 8])
def test_quantizer_error_bound(b):
    x = (np.random.default_rng(b).standard_normal((400, 32)) * 3).astype(np.float16).astype(np.float32)
    codes, sc, ze = O.quantize_groups(x, b)
    assert codes.max() <= (1 << b) - 1
    s = sc.astype(np.float64)[:, None]
    xh = ze.astype(np.float64)[:, None] + s * codes
    bound = s / 2 + ((1 << b) - 1) * s * 2.0 ** -10 + 1e-6
    assert np.all(np.abs(xh - x) <= bound)
    # fp16 inputs: the group minimum is exact in fp16, so it is reproduced exactly
    assert np.all(xh.min(axis=1) == x.min(axis=1))


# ---------------------------------------------------------------- layout
def test_word_layout_golden():
    for c in json.load(open(os.path.join(GOLDEN, "word_layout.json")))["cases"]:
        b = c["b"]
        word = sum(int(code) << O.bit_offset(e, b) for e, code in enumerate(c["codes"]))
        assert word == c["word"], c


def test_tile_layout_golden():
    g = json.load(open(os.path.join(GOLDEN, "tile_layout.json")))
    for c in g["k_positions"]:
        assert O.k_word_position(c["t"], c["w"]) == c["pos"], c
    for c in g["k_slots_in_block"]:
        assert O.k_slot_in_block(c["b"], c["i"], c["e"]) == c["slot"], c
    for c in g["v_code_positions"]:
        assert O.v_code_position(c["p"], c["c"], c["b"], c["D"]) == (c["word"], c["bit"]), c
    for c in g["v_meta_positions"]:
        assert O.v_meta_position(c["p"], c["grp"], c["D"]) == (c["scale"], c["zero"]), c
    # every rule is a permutation of what it places
    for rw in (1, 3, 11):
        pos = sorted(O.k_word_position(t, w) for t in range(32) for w in range(rw))
        assert pos == list(range(32 * rw))
    for b in (16, 8, 4, 2):
        per = 32 // b
        assert sorted(O.k_slot_in_block(b, i, e) for i in range(b // 2) for e in range(per)) == list(range(16))
    for b in (2, 4, 8):
        for D in (64, 128):
            bits = sorted(32 * w + bit for p in range(16) for c in range(D)
                          for (w, bit) in [O.v_code_position(p, c, b, D)])
            # each (pair, channel) takes b bits of the low half; together with the odd token's high
            # half they fill all D*b words exactly once
            assert len(set(bits)) == 16 * D and max(w for w, _ in (O.v_code_position(p, c, b, D)
                                                               for p in range(16) for c in range(D))) == D * b - 1
            assert all(bit % 32 + b <= 16 for bit in bits)
    for D in (64, 128):
        NG = D // 32
        idx = sorted(x for p in range(16) for g in range(NG) for x in O.v_meta_position(p, g, D))
        assert idx == list(range(32 * NG))


def test_plan_sizes_golden():
    """Hand-worked plans: every size and order field, the slot tables, the offsets of a second head,
    the batch totals and the decode's byte count."""
    for case in json.load(open(os.path.join(GOLDEN, "plan_sizes.json")))["cases"]:
        D, Np = case["head_dim"], case["n_prefix"]
        H = len(case["bits_chan"])
        bits_tok = np.zeros((1, H, Np), np.uint8)
        for j, runs in enumerate(case["bits_tok_runs"]):
            for a, b_, w in runs:
                bits_tok[0, j, a:b_] = w
        bits_chan = np.array(case["bits_chan"], np.uint8)[None]
        plan = O.make_plan(bits_tok, bits_chan, D)
        for j, exp in enumerate(case["heads"]):
            hp = plan["heads"][j]
            for key, val in exp.items():
                got = hp[key].tolist() if key == "slots" else hp[key]
                assert got == val, (case["name"], j, key, got, val)
        for key, val in case["totals"].items():
            assert plan[key] == val, (case["name"], key)
        nb = O.decode_bytes(plan, D, case["h_q"], H, case["len_c"], 1)
        assert nb == case["decode_bytes"], (case["name"], nb)


def test_packed_words_sit_where_the_layout_puts_them():
    """A K word and a V word of the packed tile, rebuilt from the quantiser's codes with the layout
    rules, are found at their positions; the head's K metadata leads its zone-A bytes."""
    w, q, k, v, al, cache = _tiny_cache(3.0, 3.0)
    hp = cache["plan"]["heads"][0]
    za = cache["zone_a"].view(np.uint32)
    kept = np.sort(np.concatenate([t[t >= 0] for t in hp["tokens"]]))
    # first tile of the first non-empty 2/4/8-bit class
    ci = next(i for i in range(3) if hp["tiles"][i] > 0)
    off_words = (hp["a_off"] + hp["meta_bytes"] + sum(hp["tiles"][i] * hp["tile_bytes"][i] for i in range(ci))) // 4
    tt = hp["tokens"][ci][:32]
    t = 9 if tt[9] >= 0 else 0
    # the first word of every quantised K segment of token t: element e holds slot slot_in_block(b, 0, e)
    wbase = sbase = 0
    s_q0 = hp["k_slots"] - hp["meta_slots"]
    meta = cache["zone_a"][hp["a_off"]:hp["a_off"] + 4 * hp["meta_slots"]].view(np.float16)
    for b, nw in zip((16, 8, 4, 2), hp["k_words"]):
        if b < 16 and nw > 0:
            word = 0
            for e in range(32 // b):
                s = sbase + O.k_slot_in_block(b, 0, e)
                ch = hp["slots"][s]
                if ch < 0:
                    continue
                codes, sc, ze = O.quantize_groups(k[kept, 0, ch].astype(np.float32)[None], b)
                assert meta[2 * (s - s_q0)] == sc[0] and meta[2 * (s - s_q0) + 1] == ze[0]
                word |= int(codes[0][np.nonzero(kept == tt[t])[0][0]]) << O.bit_offset(e, b)
            assert int(za[off_words + O.k_word_position(t, wbase)]) == word, b
        wbase += nw
        sbase += 16 * hp["k_blocks"][(16, 8, 4, 2).index(b)]
    # a V word: pair p of the tile, the words of lane (g, q) hold its channels
    b = (2, 4, 8)[ci]
    D = w.head_dim
    vbase = off_words + 32 * hp["row_words"]
    p = 5
    codes_even = O.quantize_groups(v[tt[2 * p], 0].reshape(-1, 32), b)[0].ravel()
    codes_odd = O.quantize_groups(v[tt[2 * p + 1], 0].reshape(-1, 32), b)[0].ravel() if tt[2 * p + 1] >= 0 else None
    c = 37
    widx, bit = O.v_code_position(p, c, b, D)
    word = int(za[vbase + widx])
    assert (word >> bit) & ((1 << b) - 1) == codes_even[c]
    if codes_odd is not None:
        assert (word >> (bit + 16)) & ((1 << b) - 1) == codes_odd[c]


def _tiny_cache(avg_v, avg_k, cap_extra=4, seed_w="tiny"):
    w = synth.WORKLOADS[seed_w]
    q, k, v = (t.numpy() for t in synth.prefill(w))
    sc = O.score(q, k, v, w.window)
    al = O.allocate(sc["g_tok"], sc["w_chan"], k, avg_v, avg_k)
    cache = O.pack(k[None], v[None], al["bits_tok"][None], al["bits_chan"][None], w.window,
                   cap_c=w.window + cap_extra)
    return w, q, k, v, al, cache


def test_pack_unpack_round_trip_matches_quantiser():
    """Unpacked values equal zero + scale * code of each group quantised on its own."""
    w, q, k, v, al, cache = _tiny_cache(3.0, 3.0)
    hp = cache["plan"]["heads"][0]
    pos, Kh, Vh = O.unpack(cache, w.head_dim)[0]
    assert sorted(pos.tolist()) == np.nonzero(al["bits_tok"][0])[0].tolist()
    for i, t in enumerate(pos):
        bv = int(al["bits_tok"][0, t])
        if bv == 16:
            np.testing.assert_array_equal(Vh[i], v[t, 0].astype(np.float16).astype(np.float64))
        else:
            c, s, z = O.quantize_groups(v[t, 0].reshape(-1, 32), bv)
            np.testing.assert_array_equal(Vh[i], (z.astype(np.float64)[:, None] + s.astype(np.float64)[:, None] * c).ravel())
    # K: channel c is quantised over every kept prefix token of the head
    for c in range(w.head_dim):
        bk = int(al["bits_chan"][0, c])
        got = Kh[:, c]
        if bk == 0:
            assert np.all(got == 0)
        elif bk == 16:
            np.testing.assert_array_equal(got, k[pos, 0, c].astype(np.float16).astype(np.float64))
        else:
            kept = np.sort(pos)
            cc, s, z = O.quantize_groups(k[kept, 0, c], bk)
            exp = float(z) + float(s) * cc.astype(np.float64)
            np.testing.assert_array_equal(got, exp[np.searchsorted(kept, pos)])


def test_pack_sizes_and_index():
    w, q, k, v, al, cache = _tiny_cache(3.0, 3.0)
    hp = cache["plan"]["heads"][0]
    assert cache["zone_a"].size == hp["meta_bytes"] + sum(n * b for n, b in zip(hp["tiles"], hp["tile_bytes"]))
    assert all(tb % 16 == 0 for tb in hp["tile_bytes"]) and hp["meta_bytes"] % 16 == 0
    idx = cache["index"]
    assert sorted(idx[idx >= 0].tolist()) == np.nonzero(al["bits_tok"][0])[0].tolist()


# ---------------------------------------------------------------- decode
def _sdpa(qv, K, V):
    qt = torch.tensor(qv)[None, None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        qt, torch.tensor(K)[None, None], torch.tensor(V)[None, None])[0, 0, 0].numpy()


def test_decode_all_16_bits_is_full_attention():
    """Budget >= 16 bits per unit keeps every token and channel in fp16: plain attention."""
    w, q, k, v, al, cache = _tiny_cache(16.0, 16.0)
    assert np.all(al["bits_tok"] == 16) and np.all(al["bits_chan"] == 16)
    qn, kn, vn = (t.numpy() for t in synth.decode_step(w, 0))
    O.append(cache, kn, vn)
    out = O.decode(cache, qn)
    K = np.concatenate([k[:, 0], kn[:, 0]]).astype(np.float16).astype(np.float64)
    V = np.concatenate([v[:, 0], vn[:, 0]]).astype(np.float16).astype(np.float64)
    for h in range(w.h_q):
        np.testing.assert_allclose(out[0, h], _sdpa(qn[0, h].astype(np.float64), K, V), rtol=1e-10, atol=1e-12)


def test_decode_zero_budget_is_window_attention():
    w, q, k, v, al, cache = _tiny_cache(0.0, 0.0)
    assert np.all(al["bits_tok"] == 0)
    qn, kn, vn = (t.numpy() for t in synth.decode_step(w, 1))
    O.append(cache, kn, vn)
    out = O.decode(cache, qn)
    N, W = w.n_tokens, w.window
    K = np.concatenate([k[N - W:, 0], kn[:, 0]]).astype(np.float16).astype(np.float64)
    V = np.concatenate([v[N - W:, 0], vn[:, 0]]).astype(np.float16).astype(np.float64)
    for h in range(w.h_q):
        np.testing.assert_allclose(out[0, h], _sdpa(qn[0, h].astype(np.float64), K, V), rtol=1e-10, atol=1e-12)


def test_decode_softmax_weights_sum_to_one():
    """A constant value row comes back unchanged: the attention weights sum to 1."""
    w, q, k, v, al, cache = _tiny_cache(3.0, 3.0)
    cache["zone_b"][:] = np.float16(0.75)
    cache["zone_c_v"][:] = np.float16(0.75)
    un = O.unpack(cache, w.head_dim)
    pos, Kh, Vh = un[0]
    Vh[:] = 0.75
    out = O.decode(cache, q[-1:, :, :], unpacked=un)
    np.testing.assert_allclose(out, 0.75, rtol=1e-14)


def test_decode_bytes_all_16_matches_kv_formula():
    w, q, k, v, al, cache = _tiny_cache(16.0, 16.0)
    Np = w.n_prefix
    got = O.decode_bytes(cache["plan"], w.head_dim, w.h_q, w.h_kv, len_c=w.window, batch=1)
    expect = O.kv_cache_bytes(1, w.h_kv, w.head_dim, 2, w.n_tokens) + w.h_q * w.head_dim * 6
    assert got == expect


# ---------------------------------------------------------------- allocation variants
def test_topk_keep_brute_force_and_argsort():
    rng = np.random.default_rng(11)
    for trial in range(300):
        U = int(rng.integers(1, 9))
        w = rng.choice([0.0, 0.5, 1.0, 2.0, 3.5, 7.0], size=U).astype(np.float32) if trial % 2 else \
            rng.lognormal(0, 1, U).astype(np.float32)
        avg = float(rng.choice([0.0, 1.0, 3.0, 5.5, 8.0, 16.0]))
        bits, lam = O.topk_keep(w, avg)
        k = int(np.floor(np.float32(avg) * U)) // 16
        # brute force: the smallest candidate level >= 0 that at most k weights exceed
        cands = sorted(set([0.0] + [float(x) for x in w]))
        best = next(c for c in cands if np.sum(w > np.float32(c)) <= k)
        assert float(lam) == best, (w, avg, lam, best)
        assert np.array_equal(bits, np.where(w > lam, 16, 0))
        assert int(np.sum(bits)) // 16 <= k
        if len(set(w.tolist())) == U and np.all(w > 0):   # distinct weights: exactly the k largest
            top = set(np.argsort(-w)[:k].tolist())
            assert set(np.nonzero(bits)[0].tolist()) == top


def test_topk_keep_ties_and_extremes():
    w = np.full(10, 2.0, np.float32)
    bits, lam = O.topk_keep(w, 3.2)                         # k = 2 of 10 equal weights: none strictly above
    assert float(lam) == 2.0 and not bits.any()
    bits, lam = O.topk_keep(w, 16.0)                        # k = U: all kept, lambda 0
    assert float(lam) == 0.0 and np.all(bits == 16)
    bits, lam = O.topk_keep(np.array([0, 0, 5], np.float32), 16.0)
    assert list(bits) == [0, 0, 16]                         # zero weights never kept


def test_threshold_keep_closed_form():
    w = np.array([0.0, 0.1, 0.5, 0.5, 2.0], np.float32)
    assert list(O.threshold_keep(w, 0.5)) == [0, 0, 0, 0, 16]
    assert list(O.threshold_keep(w, 0.0)) == [0, 16, 16, 16, 16]


def test_allocate_per_head_reduces_to_pooled_for_one_head_and_keeps_budgets():
    w, q, k, v, al, cache = _tiny_cache(3.0, 3.0)
    sc = O.score(q, k, v, w.window)
    one = O.allocate_per_head(sc["g_tok"], sc["w_chan"], k, 3.0, 3.0)
    pooled = O.allocate(sc["g_tok"], sc["w_chan"], k, 3.0, 3.0)
    for key in ("bits_tok", "bits_chan", "sigma_chan", "g_chan"):
        assert np.array_equal(one[key], pooled[key]), key
    assert float(one["lam_v"][0]) == float(pooled["lam_v"]) and float(one["lam_k"][0]) == float(pooled["lam_k"])
    # two heads: every head spends at most its own budget, and its level is the smallest that fits
    rng = np.random.default_rng(5)
    g = rng.lognormal(0, 2, (2, 300)).astype(np.float32)
    wc = rng.lognormal(0, 1, (2, 64)).astype(np.float32)
    kk = rng.standard_normal((300 + 10, 2, 64)).astype(np.float32)
    r = O.allocate_per_head(g, wc, kk, 2.5, 2.0)
    for j in range(2):
        assert int(r["bits_tok"][j].astype(np.int64).sum()) <= int(np.floor(np.float32(2.5) * 300))
        assert int(r["bits_chan"][j].astype(np.int64).sum()) <= int(np.floor(np.float32(2.0) * 64))
        lower = np.nextafter(r["lam_v"][j], np.float32(-1))
        if r["lam_v"][j] > 0:
            assert int(O.widths_at(O.breakpoints(g[j]), lower).astype(np.int64).sum()) > int(np.floor(np.float32(2.5) * 300))


def test_bench_decode_bytes_agree_with_the_oracle():
    """bench.py counts the decode's algorithmic bytes with its own copy of the formula (the product
    path does not import the oracle): both must give the same number on the same plans."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(os.path.dirname(__file__), "..", "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    for avg in (0.5, 2.0, 3.0, 7.0, 16.0):
        w, q, k, v, al, cache = _tiny_cache(avg, avg)
        heads = cache["plan"]["heads"]
        for len_c in (0, w.window, w.window + 3):
            ours = O.decode_bytes(cache["plan"], w.head_dim, w.h_q, w.h_kv, len_c=len_c, batch=1)
            theirs = bench.decode_bytes_per_call(heads, w.head_dim, w.h_q, 1, len_c)
            assert theirs == pytest.approx(ours, rel=0, abs=1e-6), (avg, len_c)
