"""GPU parity: every step of the RDKV path through the C ABI against the CPU oracle.

Bars (from the method's arithmetic): weights max relative error 1e-3;
allocations and packed bytes bit-exact given identical gains; decode output
max abs error 2e-3 against the oracle's float64 attention on the same
quantised values.
"""
import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# parity cases: shapes and generators of the workloads at sizes the oracle finishes in seconds,
# with ragged tails (N not a multiple of the 32-token tile)
CASES = {
    "tiny_f32": synth.WORKLOADS["tiny"],
    "small_f16": synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2,
                                                   decode_steps=6),
    "d64_f16": synth.WORKLOADS["tiny"].scaled(dtype="f16", n_tokens=777, h_q=8, h_kv=2, window=17, batch=1),
    "zipf_f16": synth.WORKLOADS["llama8b"].scaled(n_tokens=1500, h_q=8, h_kv=2, window=128, batch=1),
    # one query head per KV head; two (fp32, D = 64); eight (fp32, D = 128: the K operand's high part
    # and remainder as two products, the zone-C queries' remainder too)
    "mha_f16": synth.WORKLOADS["llama3b"].scaled(n_tokens=900, h_q=4, h_kv=4, window=32, batch=1, decode_steps=4),
    "g2_f32": synth.WORKLOADS["tiny"].scaled(n_tokens=700, h_q=4, h_kv=2, window=20),
    "g8_f32": synth.WORKLOADS["llama3b"].scaled(dtype="f32", n_tokens=600, h_q=16, h_kv=2, window=24, batch=1,
                                                 decode_steps=4),
    # 32 (sequence, KV head) pairs: the decode's two-blocks-per-SM layout
    "many_g8_d128": synth.WORKLOADS["llama3b"].scaled(n_tokens=400, h_q=32, h_kv=4, window=16, batch=8,
                                                      decode_steps=3),
    "many_g4_d64_f32": synth.WORKLOADS["tiny"].scaled(n_tokens=300, h_q=16, h_kv=4, window=16, batch=8),
    "many_g8_d64": synth.WORKLOADS["tiny"].scaled(dtype="f16", n_tokens=350, h_q=32, h_kv=4, window=16, batch=8),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _inputs(w):
    q, k, v = synth.prefill_batch(w)
    return (q, k, v), tuple(t.to(DEV) for t in (q, k, v))


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-30)


# ---------------------------------------------------------------- step 1: weights
@pytest.mark.parametrize("case", list(CASES))
def test_score_matches_oracle(case):
    w = CASES[case]
    (q, k, v), (qd, kd, vd) = _inputs(w)
    shape = rdkv.shape_of(qd, kd, w.window)
    got = rdkv.rdkv_score(shape, qd, kd, vd)
    for b in range(w.batch):
        ref = O.score(q[b].numpy(), k[b].numpy(), v[b].numpy(), w.window)
        for key in ("w_tok", "w_chan", "sigma_tok", "g_tok"):
            g = got[key][b].cpu().numpy()
            assert _rel(g, ref[key]).max() <= 1e-3, (case, key, _rel(g, ref[key]).max())
        assert abs(float(got["w_tok"][b].sum(dim=1).double().mean()) - w.n_tokens * w.group) <= 1e-3 * w.n_tokens * w.group


# ---------------------------------------------------------------- steps 2/3: water-filling
@pytest.mark.parametrize("seed", range(6))
def test_waterfill_bit_exact(seed):
    rng = np.random.default_rng(seed)
    n_inst = int(rng.integers(1, 5))
    U = int(rng.integers(1, 30000))
    g = rng.lognormal(0, 2.5, (n_inst, U)).astype(np.float32)
    g[rng.random((n_inst, U)) < 0.05] = 0.0
    if seed % 2:
        g[:, : U // 3] = g[:, :1]               # many equal gains (ties)
    for avg in (0.0, 0.37, 2.0, 2.5, 7.9, 16.0, 20.0):
        bits, lam, status = rdkv.rdkv_waterfill(torch.tensor(g, device=DEV), avg)
        assert int(status.item()) == 0
        for i in range(n_inst):
            rb, rl = O.waterfill(g[i], avg)
            assert np.array_equal(bits[i].cpu().numpy(), rb), (seed, avg, i)
            assert float(lam[i]) == float(rl)


def test_waterfill_flags_invalid_gains():
    g = torch.tensor([[1.0, float("nan"), 2.0, -3.0, float("inf"), 0.5]], device=DEV)
    bits, lam, status = rdkv.rdkv_waterfill(g, 4.0)
    assert int(status.item()) == rdkv.RDKV_ERR_INVALID_ARG
    b = bits[0].cpu().numpy()
    assert b[1] == 0 and b[3] == 0 and b[4] == 0


# ---------------------------------------------------------------- full path up to the pack
def _compress(w, avg_v, avg_k, cap_extra=8):
    (q, k, v), (qd, kd, vd) = _inputs(w)
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg_v, avg_k)
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + cap_extra,
                           sizes=sizes)
    return (q, k, v), (qd, kd, vd), shape, sc, al, sizes, cache


@pytest.mark.parametrize("case", list(CASES))
def test_allocate_and_plan_match_oracle(case):
    w = CASES[case]
    avg = w.budgets[0]
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, avg, avg)
    g_tok = sc["g_tok"].cpu().numpy()
    bits_tok = al["bits_tok"].cpu().numpy()
    g_chan = al["g_chan"].cpu().numpy()
    bits_chan = al["bits_chan"].cpu().numpy()
    hdr, heads, slots, lam = rdkv.read_plan(al["plan"])
    for b in range(w.batch):
        rb, rl = O.waterfill(g_tok[b], avg)                        # identical gains -> identical widths
        assert np.array_equal(bits_tok[b].ravel(), rb)
        assert float(lam[b]) == float(rl)
        sig_ref = O.kept_channel_spread(k[b].numpy(), bits_tok[b])
        assert _rel(al["sigma_chan"][b].cpu().numpy(), sig_ref)[sig_ref > 0].max() <= 1e-5
        rb, rl = O.waterfill(g_chan[b], avg)
        assert np.array_equal(bits_chan[b].ravel(), rb)
        assert float(lam[w.batch + b]) == float(rl)
    plan = O.make_plan(bits_tok, bits_chan, w.head_dim)
    assert int(hdr["status"]) == 0 and sizes.status == 0
    for key in ("zone_a_bytes", "zone_b_rows", "index_slots", "kept_tokens", "max_tile_bytes", "max_stage_bytes"):
        assert int(hdr[key]) == plan[key] == getattr(sizes, key), key
    for i, hp in enumerate(plan["heads"]):
        for key in ("n_v", "tiles", "n_k", "k_words", "tile_bytes"):
            assert list(heads[i][key]) == list(hp[key]), (i, key)
        for key in ("row_words", "k_slots", "meta_slots", "a_off", "a_bytes", "b_row", "slot_off"):
            assert int(heads[i][key]) == hp[key], (i, key)
        assert np.array_equal(slots[i][: hp["k_slots"]], hp["slots"])
        assert np.all(slots[i][hp["k_slots"]:] == -1)


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("budget", ["page", "low", "high"])
def test_pack_bit_exact(case, budget):
    w = CASES[case]
    avg = {"page": w.budgets[0], "low": 0.7, "high": 9.0}[budget]
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, avg, avg)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + 8)
    torch.cuda.synchronize()
    za = cache.zone_a.cpu().numpy()[: ref["zone_a"].size]
    if not np.array_equal(za, ref["zone_a"]):
        bad = np.nonzero(za != ref["zone_a"])[0]
        pytest.fail(f"zone A differs at {bad.size} bytes, first {bad[:8]}")
    assert np.array_equal(cache.zone_b.cpu().numpy()[: ref["zone_b"].shape[0]].view(np.uint16),
                          ref["zone_b"].view(np.uint16))
    assert np.array_equal(cache.index_map.cpu().numpy()[: ref["index"].size], ref["index"])
    assert np.array_equal(cache.zone_c_k.cpu().numpy()[:, :, : w.window].view(np.uint16),
                          ref["zone_c_k"][:, :, : w.window].view(np.uint16))
    assert np.array_equal(cache.zone_c_v.cpu().numpy()[:, :, : w.window].view(np.uint16),
                          ref["zone_c_v"][:, :, : w.window].view(np.uint16))
    assert cache.len_c == w.window


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("budget", ["page", "zero", "full", "high"])
def test_decode_matches_oracle(case, budget):
    w = CASES[case]
    avg = {"page": w.budgets[0], "zero": 0.0, "full": 16.0, "high": 9.0}[budget]
    steps = 5
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, avg, avg, cap_extra=steps)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + steps)
    un = O.unpack(ref, w.head_dim)
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        out = rdkv.rdkv_decode_attn(cache, qn.to(DEV)).cpu().numpy()
        exp = O.decode(ref, qn.numpy(), unpacked=un)
        err = np.abs(out - exp).max()
        assert err <= 2e-3, (case, budget, step, err)
    assert rdkv.rdkv_decode_status(cache) == 0


@pytest.mark.parametrize("case", ["small_f16", "zipf_f16"])
def test_decode_block_dealing_host_and_kernel(case):
    """The blocks are dealt to the heads on the host from the plan's cost estimates (filled by
    rdkv_plan_sizes), or by the kernel itself when they are missing; any estimate gives the
    same attention (only the split of the work changes)."""
    w = CASES[case]
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, w.budgets[0], w.budgets[0], cap_extra=2)
    n_heads = w.batch * w.h_kv
    costs = list(sizes.head_cost)
    assert all(c > 0 for c in costs[:n_heads]) and all(c == 0 for c in costs[n_heads:])
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + 2)
    qn, kn, vn = synth.decode_step(w, 0)
    rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
    O.append(ref, kn.numpy(), vn.numpy())
    exp = O.decode(ref, qn.numpy())
    outs = []
    for variant in ("host", "kernel", "skewed"):
        for h in range(rdkv.COST_HEADS):
            cache.c.sizes.head_cost[h] = {"host": costs[h], "kernel": 0,
                                          "skewed": (1 if h % 2 else 1000000) if h < n_heads else 0}[variant]
        out = rdkv.rdkv_decode_attn(cache, qn.to(DEV)).cpu().numpy()
        assert np.abs(out - exp).max() <= 2e-3, variant
        outs.append(out)
    assert rdkv.rdkv_decode_status(cache) == 0
    # a different split of the tokens moves the softmax's running reference and with it the
    # fp16 rounding of the probabilities: the outputs agree to that rounding
    d = np.abs(outs[0] - outs[1])
    assert d.max() <= 2e-3 and d.mean() <= 5e-5, (d.max(), d.mean())


def test_decode_without_window_and_empty_zone_c():
    """W = 0: before any append the cache may be empty for a zero budget (output 0)."""
    w = CASES["small_f16"].scaled(window=0)
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, 0.0, 0.0, cap_extra=3)
    qn, kn, vn = synth.decode_step(w, 0)
    out = rdkv.rdkv_decode_attn(cache, qn.to(DEV)).cpu().numpy()
    assert np.all(out == 0)
    rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
    out = rdkv.rdkv_decode_attn(cache, qn.to(DEV)).cpu().numpy()
    np.testing.assert_allclose(out, np.broadcast_to(vn.numpy().astype(np.float16).astype(np.float64).repeat(
        w.group, axis=1), out.shape), atol=1e-6)


def test_append_capacity():
    w = CASES["tiny_f32"]
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, 3.0, 3.0, cap_extra=1)
    qn, kn, vn = synth.decode_step(w, 0)
    rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
    with pytest.raises(rdkv.RDKVError) as e:
        rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
    assert e.value.code == rdkv.RDKV_ERR_CAPACITY


# ---------------------------------------------------------------- fused decode step
@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("budget", ["page", "full"])
def test_decode_step_matches_oracle(case, budget):
    """append + attend in one launch: the output against the oracle, the stored rows bit-exact."""
    w = CASES[case]
    avg = {"page": w.budgets[0], "full": 16.0}[budget]
    steps = 20  # crosses a 16-row zone-C block boundary for every window size
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, avg, avg, cap_extra=steps)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + steps)
    un = O.unpack(ref, w.head_dim)
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV)).cpu().numpy()
        O.append(ref, kn.numpy(), vn.numpy())
        exp = O.decode(ref, qn.numpy(), unpacked=un)
        err = np.abs(out - exp).max()
        assert err <= 2e-3, (case, budget, step, err)
    assert rdkv.rdkv_decode_status(cache) == 0
    assert cache.len_c == w.window + steps and int(cache.len_dev.item()) == w.window + steps
    n = w.window + steps
    assert np.array_equal(cache.zone_c_k.cpu().numpy()[:, :, :n].view(np.uint16), ref["zone_c_k"][:, :, :n].view(np.uint16))
    assert np.array_equal(cache.zone_c_v.cpu().numpy()[:, :, :n].view(np.uint16), ref["zone_c_v"][:, :, :n].view(np.uint16))


def test_decode_step_agrees_with_append_then_attend():
    w = CASES["small_f16"]
    steps = 6
    (q, k, v), (qd, kd, vd), shape, sc, al, sizes, c1 = _compress(w, w.budgets[0], w.budgets[0], cap_extra=steps)
    c2 = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + steps, sizes=sizes)
    for step in range(steps):
        qn, kn, vn = (t.to(DEV) for t in synth.decode_step(w, step))
        a = rdkv.rdkv_decode_step(c1, qn, kn, vn)
        rdkv.rdkv_append(c2, kn, vn)
        b = rdkv.rdkv_decode_attn(c2, qn)
        # the same values in the same blocks; which warp meets which tile first may differ, and with
        # it the reference max that p = 2^(s - m) is rounded to fp16 against (p rounds to 2^-11
        # relative either way), so single elements may differ by up to the parity bar; a structural
        # difference (a token missed or counted twice) moves every element of a head
        d = (a - b).abs()
        assert float(d.max()) <= 2e-3, float(d.max())
        assert float(d.mean()) <= 5e-5, float(d.mean())


def test_decode_step_in_a_replayed_graph():
    """A captured step replayed: every replay appends one row and attends over all of them."""
    w = CASES["small_f16"]
    steps = 5
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, w.budgets[0], w.budgets[0], cap_extra=steps + 1)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + steps + 1)
    un = O.unpack(ref, w.head_dim)
    q0, k0, v0 = (t.to(DEV) for t in synth.decode_step(w, 0))
    qb, kb, vb = q0.clone(), k0.clone(), v0.clone()
    out = torch.empty(w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=DEV)
    cache.decode_workspace()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        saved = int(cache.len_dev.item())
        with torch.cuda.graph(g, stream=s):
            rdkv.rdkv_decode_step(cache, qb, kb, vb, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert int(cache.len_dev.item()) == saved  # capture launches nothing
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        qb.copy_(qn.to(DEV)); kb.copy_(kn.to(DEV)); vb.copy_(vn.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        O.append(ref, kn.numpy(), vn.numpy())
        exp = O.decode(ref, qn.numpy(), unpacked=un)
        assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3, step
    assert int(cache.len_dev.item()) == w.window + steps
    assert rdkv.rdkv_decode_status(cache) == 0


def test_decode_step_past_capacity_on_the_device():
    """A step that finds zone C full attends with its token, stores nothing and reports it."""
    w = CASES["tiny_f32"]
    (q, k, v), _, shape, sc, al, sizes, cache = _compress(w, 3.0, 3.0, cap_extra=1)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + 2)
    un = O.unpack(ref, w.head_dim)
    qn, kn, vn = synth.decode_step(w, 0)
    rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
    O.append(ref, kn.numpy(), vn.numpy())
    assert int(cache.len_dev.item()) == cache.c.cap_c
    before = cache.zone_c_k.clone()
    cache.c.len_c -= 1  # make the host mirror lag, as a replayed graph would
    qn, kn, vn = synth.decode_step(w, 1)
    out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV)).cpu().numpy()
    O.append(ref, kn.numpy(), vn.numpy())  # the oracle's zone C has room for it: same attention
    exp = O.decode(ref, qn.numpy(), unpacked=un)
    assert np.abs(out - exp).max() <= 2e-3
    assert int(cache.len_dev.item()) == cache.c.cap_c
    assert torch.equal(cache.zone_c_k, before)
    assert rdkv.rdkv_decode_status(cache) == rdkv.RDKV_ERR_CAPACITY
    assert rdkv.rdkv_decode_status(cache) == 0  # read and cleared


# ---------------------------------------------------------------- allocation variants
@pytest.mark.parametrize("case", ["small_f16", "zipf_f16", "tiny_f32"])
@pytest.mark.parametrize("mode", ["per_head", "topk", "threshold"])
def test_allocation_modes_match_oracle(case, mode):
    """Variants on the same plan, pack and decode: widths and levels bit-exact given the same
    weights, then the packed bytes and the decode against the oracle."""
    w = CASES[case]
    avg = w.budgets[0]
    (q, k, v), (qd, kd, vd) = _inputs(w)
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    Np = w.n_tokens - w.window
    w_tok = sc["w_tok"].cpu().numpy()
    tau = float(np.float32(np.median(w_tok[:, :, :Np])))
    code = {"per_head": rdkv.RDKV_ALLOC_PER_HEAD, "topk": rdkv.RDKV_ALLOC_TOPK,
            "threshold": rdkv.RDKV_ALLOC_THRESHOLD}[mode]
    al = rdkv.rdkv_allocate_mode(shape, code, sc["w_tok"], sc["g_tok"], sc["w_chan"], kd, avg, avg, param=tau)
    hdr, heads, slots, lam = rdkv.read_plan(al["plan"])
    bits_tok = al["bits_tok"].cpu().numpy()
    bits_chan = al["bits_chan"].cpu().numpy()
    H = w.h_kv
    for b in range(w.batch):
        if mode == "per_head":
            r = O.allocate_per_head(sc["g_tok"][b].cpu().numpy(), sc["w_chan"][b].cpu().numpy(), k[b].numpy(), avg, avg)
            # identical V widths -> identical kept sets -> spreads within float rounding; K widths
            # are compared given the library's own channel gains
            assert np.array_equal(bits_tok[b], r["bits_tok"])
            assert np.array_equal(lam[b * H:(b + 1) * H], r["lam_v"])
            for j in range(H):
                rb, rl = O.waterfill(al["g_chan"][b, j].cpu().numpy(), avg)
                assert np.array_equal(bits_chan[b, j], rb) and float(lam[w.batch * H + b * H + j]) == float(rl)
        else:
            for j in range(H):
                wj = w_tok[b, j, :Np]
                if mode == "topk":
                    rb, rl = O.topk_keep(wj, avg)
                else:
                    rb, rl = O.threshold_keep(wj, tau), np.float32(tau)
                assert np.array_equal(bits_tok[b, j], rb), (b, j)
                assert float(lam[b * H + j]) == float(rl)
            assert np.all(bits_chan[b] == 16)
    plan = O.make_plan(bits_tok, bits_chan, w.head_dim)
    for key in ("zone_a_bytes", "zone_b_rows", "index_slots", "kept_tokens"):
        assert int(hdr[key]) == plan[key], key
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    steps = 3
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + steps, sizes=sizes)
    ref = O.pack(k.numpy(), v.numpy(), bits_tok, bits_chan, w.window, cap_c=w.window + steps)
    torch.cuda.synchronize()
    assert np.array_equal(cache.zone_a.cpu().numpy()[: ref["zone_a"].size], ref["zone_a"])
    un = O.unpack(ref, w.head_dim)
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV)).cpu().numpy()
        O.append(ref, kn.numpy(), vn.numpy())
        assert np.abs(out - O.decode(ref, qn.numpy(), unpacked=un)).max() <= 2e-3, (mode, step)


def test_pooled_mode_equals_rdkv_allocate():
    w = CASES["small_f16"]
    (q, k, v), (qd, kd, vd) = _inputs(w)
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    a = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, 2.5, 2.0)
    b = rdkv.rdkv_allocate_mode(shape, rdkv.RDKV_ALLOC_POOLED, None, sc["g_tok"], sc["w_chan"], kd, 2.5, 2.0)
    for key in ("bits_tok", "bits_chan", "plan"):
        assert torch.equal(a[key], b[key]), key
