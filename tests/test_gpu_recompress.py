"""GPU parity of zone-C re-compression (reading R10) through the C ABI against the CPU oracle.

Bars: log-sum-exp and attention outputs max abs 2e-3 (the decode's bar); merge of parts 1e-5;
rows taken from zone C, widths at the prefill's levels and the segment's packed bytes bit-exact
(widths given identical gains); token weights and spreads max relative error 1e-3 (the weights'
bar).
"""
import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

CASES = {
    "tiny_f32": synth.WORKLOADS["tiny"],
    "small_f16": synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2,
                                                   decode_steps=6),
    "zipf_f16": synth.WORKLOADS["llama8b"].scaled(n_tokens=1500, h_q=8, h_kv=2, window=128, batch=1),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _compress(w, avg, cap_extra):
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg, avg)
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + cap_extra,
                           sizes=sizes)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + cap_extra)
    return (q, k, v), sc, al, cache, ref


def _run_steps(w, cache, ref, steps):
    """Fused decode steps with lse; returns the recent queries and lse as device tensors [B, R, ...]."""
    qs, ls = [], []
    un = O.unpack(ref, w.head_dim)
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        out, lse = rdkv.rdkv_decode_step_lse(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        if step % 7 == 0 or step == steps - 1:
            exp, exp_lse = O.decode_lse(ref, qn.numpy(), unpacked=un)
            assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3, step
            assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3, step
        qs.append(qn.to(DEV))
        ls.append(lse.clone())
    assert rdkv.rdkv_decode_status(cache) == 0
    return torch.stack(qs, dim=1).contiguous(), torch.stack(ls, dim=1).contiguous()


@pytest.mark.parametrize("case", list(CASES))
def test_decode_attn_lse_matches_oracle(case):
    w = CASES[case]
    (q, k, v), sc, al, cache, ref = _compress(w, w.budgets[0], 4)
    qn, kn, vn = synth.decode_step(w, 0)
    rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
    O.append(ref, kn.numpy(), vn.numpy())
    out, lse = rdkv.rdkv_decode_attn_lse(cache, qn.to(DEV))
    exp, exp_lse = O.decode_lse(ref, qn.numpy())
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
    # the plain call computes the same output (up to the order in which warps take tiles)
    d = (rdkv.rdkv_decode_attn(cache, qn.to(DEV)) - out).abs()
    assert d.max().item() <= 2e-3 and d.mean().item() <= 5e-5


def test_merge_matches_oracle():
    g = torch.Generator().manual_seed(5)
    P, B, Hq, D = 3, 2, 5, 64
    outs = torch.randn(P, B, Hq, D, generator=g)
    lses = torch.randn(P, B, Hq, generator=g) * 4
    lses[1, 0, 2] = -float("inf")                 # a part without keys for one row
    lses[:, 1, 4] = -float("inf")                 # a row without keys anywhere
    out, lse = rdkv.rdkv_merge_attn(outs.to(DEV), lses.to(DEV))
    exp, exp_lse = O.merge_attention(outs.numpy(), lses.numpy())
    np.testing.assert_allclose(out.cpu().numpy(), exp, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lse.cpu().numpy(), exp_lse, rtol=1e-6, atol=1e-6)
    assert lse[1, 4].item() == -float("inf") and torch.all(out[1, 4] == 0)
    # out aliasing the first part
    o2 = outs.to(DEV).contiguous()
    rdkv.rdkv_merge_attn(o2, lses.to(DEV), out=o2[0])
    np.testing.assert_allclose(o2[0].cpu().numpy(), exp, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("case", list(CASES))
def test_recompress_matches_oracle_step_by_step(case):
    """Decode steps with lse, then the oldest zone-C rows move into a segment: the rows taken, the
    weights from the recent queries, the widths at the prefill's levels, the segment's bytes, and
    the merged attention over segment and live cache, each against the oracle."""
    w = CASES[case]
    steps = w.window + 8
    (q, k, v), sc, al, cache, ref = _compress(w, w.budgets[0], steps)
    q_rec, lse_rec = _run_steps(w, cache, ref, steps)
    n_move = cache.len_c - w.window
    zk_before = cache.zone_c_k.cpu().numpy().copy()
    # rows out of zone C
    k_seg, v_seg = rdkv.rdkv_zone_c_take(cache, n_move)
    rk, rv = O.take_zone_c(ref, n_move)
    assert np.array_equal(k_seg.float().cpu().numpy(), rk.astype(np.float32))
    assert np.array_equal(v_seg.float().cpu().numpy(), rv.astype(np.float32))
    assert cache.len_c == w.window == ref["len_c"] and int(cache.len_dev.item()) == w.window
    zk = cache.zone_c_k.cpu().numpy()
    assert np.array_equal(zk[:, :, :w.window], ref["zone_c_k"][:, :, :w.window])
    assert np.array_equal(zk[:, :, :w.window], zk_before[:, :, n_move:n_move + w.window])
    # weights of the moved tokens from the recent queries
    seg = rdkv.Shape(w.batch, n_move, w.h_q, w.h_kv, w.head_dim, 0, cache.shape.dtype)
    scale = w.n_tokens / steps
    gs = rdkv.rdkv_recompress_score(seg, k_seg, v_seg, q_rec, lse_rec, scale)
    for b in range(w.batch):
        eg = O.recompress_gains(rk[b], rv[b], q_rec[b].cpu().numpy(), lse_rec[b].cpu().numpy(), scale)
        for name in ("w_tok", "sigma_tok"):
            got = gs[name][b].cpu().numpy().astype(np.float64)
            exp = eg[name].astype(np.float64)
            assert np.all(np.abs(got - exp) <= 1e-3 * np.abs(exp) + 1e-30), (b, name)
    # widths at the prefill's water levels, given the library's gains
    levels = rdkv.plan_levels(al["plan"])
    seg_al = rdkv.rdkv_allocate_at_levels(seg, levels, gs["g_tok"], sc["w_chan"], k_seg)
    lam = levels.cpu().numpy()
    g_tok = gs["g_tok"].cpu().numpy()
    bits_tok = seg_al["bits_tok"].cpu().numpy()
    g_chan = seg_al["g_chan"].cpu().numpy()
    bits_chan = seg_al["bits_chan"].cpu().numpy()
    w_chan = sc["w_chan"].cpu().numpy()
    for b in range(w.batch):
        lam_v, lam_k = lam[b], lam[w.batch + b]
        assert np.array_equal(bits_tok[b].ravel(), O.widths_at(O.breakpoints(g_tok[b]), lam_v))
        sig = O.kept_channel_spread(rk[b], bits_tok[b])
        got = seg_al["sigma_chan"][b].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - sig) <= 1e-3 * np.abs(sig) + 1e-6)
        assert np.array_equal(bits_chan[b].ravel(), O.widths_at(O.breakpoints(g_chan[b]), lam_k))
        inc = O.allocate_at_levels(g_tok[b], w_chan[b], rk[b], lam_v, lam_k)
        assert np.array_equal(inc["bits_tok"], bits_tok[b])
    _, _, _, seg_lam = rdkv.read_plan(seg_al["plan"])
    assert np.array_equal(seg_lam[:2 * w.batch], lam[:2 * w.batch])
    # the segment's bytes
    seg_cache = rdkv.rdkv_pack(seg, seg_al["plan"], k_seg, v_seg, seg_al["bits_tok"], seg_al["bits_chan"], 0)
    seg_ref = O.pack(rk, rv, bits_tok, bits_chan, 0, cap_c=0)
    assert np.array_equal(seg_cache.zone_a.cpu().numpy()[:seg_ref["zone_a"].size], seg_ref["zone_a"])
    nb = seg_ref["zone_b"].shape[0]
    assert np.array_equal(seg_cache.zone_b.cpu().numpy()[:nb], seg_ref["zone_b"])
    # attention over the segment and the live cache (its zones A, B and the rows left in zone C)
    qn = synth.decode_step(w, steps)[0]
    out, lse = rdkv.decode_segments([seg_cache], cache, qn.to(DEV))
    o1, l1 = O.decode_lse(seg_ref, qn.numpy())
    o2, l2 = O.decode_lse(ref, qn.numpy())
    exp, exp_lse = O.merge_attention(np.stack([o1, o2]), np.stack([l1, l2]))
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
    # one launch over both caches
    md = rdkv.MultiDecode([seg_cache, cache])
    out, lse = md.attn(qn.to(DEV))
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
    assert md.status() == 0
    # one cache through the several-cache call: the plain decode's result
    one, one_lse = rdkv.MultiDecode([cache]).attn(qn.to(DEV))
    assert np.abs(one.cpu().numpy() - o2).max() <= 2e-3 and np.abs(one_lse.cpu().numpy() - l2).max() <= 2e-3


def test_recompress_helper_and_a_second_segment():
    """The binding's one-call helper, twice in a row: two segments and the live cache."""
    w = CASES["small_f16"]
    steps = 2 * (w.window + 8)
    (q, k, v), sc, al, cache, ref = _compress(w, w.budgets[0], steps)
    segs, seg_refs = [], []
    done = 0
    for rnd in range(2):
        qs, ls = [], []
        for step in range(done, done + w.window + 8):
            qn, kn, vn = synth.decode_step(w, step)
            out, lse = rdkv.rdkv_decode_step_lse(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV)) if not segs else (None, None)
            if segs:  # with segments, the decode is the merge of the parts; append first
                rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
                out, lse = rdkv.decode_segments(segs, cache, qn.to(DEV))
            O.append(ref, kn.numpy(), vn.numpy())
            qs.append(qn.to(DEV))
            ls.append(lse.clone())
        done += w.window + 8
        n_move = cache.len_c - w.window
        q_rec, lse_rec = torch.stack(qs, 1).contiguous(), torch.stack(ls, 1).contiguous()
        seg_cache = rdkv.recompress(cache, al["plan"], sc["w_chan"], q_rec, lse_rec, n_move)
        al_seg = seg_cache._keep[1]
        rk, rv = O.take_zone_c(ref, n_move)
        seg_refs.append(O.pack(rk, rv, al_seg["bits_tok"].cpu().numpy(), al_seg["bits_chan"].cpu().numpy(), 0,
                               cap_c=0))
        assert np.array_equal(seg_cache.zone_a.cpu().numpy()[:seg_refs[-1]["zone_a"].size], seg_refs[-1]["zone_a"])
        segs.append(seg_cache)
    qn = synth.decode_step(w, done)[0]
    out, lse = rdkv.decode_segments(segs, cache, qn.to(DEV))
    parts = [O.decode_lse(r, qn.numpy()) for r in seg_refs + [ref]]
    exp, exp_lse = O.merge_attention(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
    out, lse = rdkv.MultiDecode(segs + [cache]).attn(qn.to(DEV))  # three caches, one launch
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3


def test_recompress_edges_all_rows_and_an_empty_segment():
    """Edges: every zone-C row moved (none stay); a segment that keeps no token (levels +inf); the
    one-launch decode over an empty segment, the moved rows' segment and the cache matches the
    oracle."""
    w = CASES["small_f16"].scaled(window=8)
    steps = 8
    (q, k, v), sc, al, cache, ref = _compress(w, w.budgets[0], steps)
    q_rec, lse_rec = _run_steps(w, cache, ref, steps)
    n_move = cache.len_c  # all 16 rows: none stay
    k_seg, v_seg = rdkv.rdkv_zone_c_take(cache, n_move)
    rk, rv = O.take_zone_c(ref, n_move)
    assert cache.len_c == 0 and int(cache.len_dev.item()) == 0
    assert np.array_equal(k_seg.float().cpu().numpy(), rk.astype(np.float32))
    seg = rdkv.recompress_from_rows(cache, k_seg, v_seg, al["plan"], sc["w_chan"], q_rec, lse_rec)
    al_seg = seg._keep[1]
    seg_ref = O.pack(rk, rv, al_seg["bits_tok"].cpu().numpy(), al_seg["bits_chan"].cpu().numpy(), 0, cap_c=0)
    # a segment at infinite levels keeps nothing
    s_seg = rdkv.Shape(w.batch, n_move, w.h_q, w.h_kv, w.head_dim, 0, cache.shape.dtype)
    inf_levels = torch.full((2 * w.batch,), float("inf"), device=DEV)
    gs = rdkv.rdkv_recompress_score(s_seg, k_seg, v_seg, q_rec, lse_rec)
    al_empty = rdkv.rdkv_allocate_at_levels(s_seg, inf_levels, gs["g_tok"], sc["w_chan"], k_seg)
    empty = rdkv.rdkv_pack(s_seg, al_empty["plan"], k_seg, v_seg, al_empty["bits_tok"], al_empty["bits_chan"], 0)
    assert empty.sizes.kept_tokens == 0 and int(al_empty["bits_tok"].sum().item()) == 0
    qn = synth.decode_step(w, steps)[0]
    out, lse = rdkv.MultiDecode([empty, seg, cache]).attn(qn.to(DEV))
    o1, l1 = O.decode_lse(seg_ref, qn.numpy())
    o2, l2 = O.decode_lse(ref, qn.numpy())  # zones A and B of the prefill; zone C now empty
    exp, exp_lse = O.merge_attention(np.stack([o1, o2]), np.stack([l1, l2]))
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
