"""Allocation and pack in one persistent launch (rdkv_allocate_pack) against the step-by-step path
(rdkv_allocate or the per-head levels of rdkv_allocate_mode, then rdkv_pack into zones of the same
bounds): every output byte-identical -- widths, spreads, gains, the whole plan buffer, zones A and
B, the index map, zone C and its length -- and the packed bytes equal to the oracle's pack of the
same widths.  Shapes cover both dtypes and head sizes, batches, several index chunks (more than
8192 prefix tokens), budgets 0 and 16, a prompt that is all window, the capacity refusal, and a
CUDA graph capture of the whole compression."""
import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

CASES = {
    "tiny_f32": (synth.WORKLOADS["tiny"], None),
    "small_f16_b2": (synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2), None),
    "zipf_f16": (synth.WORKLOADS["llama8b"].scaled(n_tokens=1500, h_q=8, h_kv=2, window=128), None),
    "chunks_f16": (synth.WORKLOADS["llama3b"].scaled(n_tokens=20000, h_q=3, h_kv=1, window=64), None),
    "d64_f16": (synth.WORKLOADS["llama3b"].scaled(n_tokens=3000, h_q=8, head_dim=64, h_kv=4, window=16), None),
    "budget0": (synth.WORKLOADS["llama3b"].scaled(n_tokens=700, h_q=4, h_kv=2, window=32), 0.0),
    "budget16": (synth.WORKLOADS["llama3b"].scaled(n_tokens=700, h_q=4, h_kv=2, window=32), 16.0),
    "all_window": (synth.WORKLOADS["llama3b"].scaled(n_tokens=96, h_q=4, h_kv=2, window=96), None),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _inputs(w):
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    return (q, k, v), (qd, kd, vd), shape, sc


def _step_by_step(shape, sc, kd, vd, avg, cap, per_head):
    if per_head:
        al = rdkv.rdkv_allocate_mode(shape, rdkv.RDKV_ALLOC_PER_HEAD, sc["w_tok"], sc["g_tok"], sc["w_chan"], kd, avg,
                                     avg)
    else:
        al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg, avg)
    bounds = rdkv.rdkv_zone_bounds(shape, avg, avg)
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], cap, sizes=bounds)
    return al, cache


def _same_cache(c1, c2, shape, window):
    s1 = rdkv.rdkv_plan_sizes(c1.plan)
    s2 = rdkv.rdkv_plan_sizes(c2.plan)
    for f in ("zone_a_bytes", "zone_b_rows", "index_slots", "kept_tokens", "max_tile_bytes", "max_stage_bytes"):
        assert getattr(s1, f) == getattr(s2, f), f
    assert list(s1.head_cost) == list(s2.head_cost)
    na, nb, ns = s1.zone_a_bytes, s1.zone_b_rows, s1.index_slots
    assert torch.equal(c1.zone_a[:na], c2.zone_a[:na])
    assert torch.equal(c1.zone_b[:nb], c2.zone_b[:nb])
    assert torch.equal(c1.index_map[:ns], c2.index_map[:ns])
    assert torch.equal(c1.zone_c_k[:, :, :window], c2.zone_c_k[:, :, :window])
    assert torch.equal(c1.zone_c_v[:, :, :window], c2.zone_c_v[:, :, :window])
    assert int(c1.len_dev.item()) == int(c2.len_dev.item()) == window
    return s1


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_allocate_pack_equals_step_by_step_and_oracle(case, per_head):
    w, budget = CASES[case]
    avg = w.budgets[0] if budget is None else budget
    (q, k, v), (qd, kd, vd), shape, sc = _inputs(w)
    cap = w.window + 4
    al, ref = _step_by_step(shape, sc, kd, vd, avg, cap, per_head)
    out, cache = rdkv.rdkv_allocate_pack(shape, sc["g_tok"], sc["w_chan"], kd, vd, avg, avg, cap, per_head=per_head)
    torch.cuda.synchronize()
    for key in ("bits_tok", "sigma_chan", "g_chan", "bits_chan", "plan"):
        assert torch.equal(out[key], al[key]), key
    assert cache.len_c == w.window
    sizes = _same_cache(cache, ref, shape, w.window)
    # the packed bytes against the oracle's pack of the same widths
    bits_tok, bits_chan = out["bits_tok"].cpu().numpy(), out["bits_chan"].cpu().numpy()
    opack = O.pack(k.numpy(), v.numpy(), bits_tok, bits_chan, w.window, cap_c=cap)
    assert sizes.zone_a_bytes == opack["zone_a"].size
    assert np.array_equal(cache.zone_a[:sizes.zone_a_bytes].cpu().numpy(), opack["zone_a"])
    assert np.array_equal(cache.index_map[:sizes.index_slots].cpu().numpy(), opack["index"])
    # the V widths against the oracle's water-filling of the library's gains (one level per
    # sequence, or per head)
    g_tok = sc["g_tok"].cpu().numpy()
    for b in range(w.batch):
        if per_head:
            for j in range(w.h_kv):
                rb, _ = O.waterfill(g_tok[b, j], avg)
                assert np.array_equal(bits_tok[b, j], rb)
        else:
            rb, _ = O.waterfill(g_tok[b], avg)
            assert np.array_equal(bits_tok[b].ravel(), rb)


def test_allocate_pack_capacity_refused():
    """Zones smaller than the plan needs: the plan status says so and nothing is packed."""
    w, _ = CASES["small_f16_b2"]
    avg = w.budgets[0]
    _, (qd, kd, vd), shape, sc = _inputs(w)
    bounds = rdkv.rdkv_zone_bounds(shape, avg, avg)
    small = rdkv.Sizes(64, bounds.zone_b_rows, bounds.index_slots, 0, 0, 0, 0, bounds.n_heads)
    out = None
    plan = torch.zeros(rdkv.lib().rdkv_plan_bytes(rdkv.ctypes.byref(shape)), dtype=torch.uint8, device=DEV)
    cache = rdkv.Cache(shape, plan, small, w.window + 4, DEV)
    out = dict(bits_tok=torch.empty(w.batch, w.h_kv, w.n_prefix, dtype=torch.uint8, device=DEV),
               sigma_chan=torch.empty(w.batch, w.h_kv, w.head_dim, dtype=torch.float32, device=DEV),
               g_chan=torch.empty(w.batch, w.h_kv, w.head_dim, dtype=torch.float32, device=DEV),
               bits_chan=torch.empty(w.batch, w.h_kv, w.head_dim, dtype=torch.uint8, device=DEV), plan=plan)
    rdkv.rdkv_allocate_pack(shape, sc["g_tok"], sc["w_chan"], kd, vd, avg, avg, w.window + 4, out=out, cache=cache)
    with pytest.raises(rdkv.RDKVError) as e:
        rdkv.rdkv_plan_sizes(plan)
    assert e.value.code == rdkv.RDKV_ERR_CAPACITY
    assert int(cache.zone_a.count_nonzero().item()) == 0
    assert int(cache.index_map.count_nonzero().item()) == 0


def test_compression_in_one_graph_with_one_allocate_pack_launch():
    """Score, then allocation and pack as one launch, captured in one CUDA graph: after a replay the
    cache equals the step-by-step path's, and the decode over it matches the oracle."""
    w, _ = CASES["small_f16_b2"]
    w = w.scaled(decode_steps=4)
    avg = w.budgets[0]
    (q, k, v), (qd, kd, vd), shape, sc = _inputs(w)
    cap = w.window + 4
    comp = rdkv.Compressor(shape, avg, avg, cap, DEV, fused=True)
    comp.run(qd, kd, vd)  # once eagerly (kernel attributes are set outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        comp.run(qd, kd, vd)
    comp.cache.zone_a.zero_()
    comp.cache.zone_b.zero_()
    comp.cache.index_map.zero_()
    g.replay()
    cache = comp.finish()
    al, ref = _step_by_step(shape, sc, kd, vd, avg, cap, False)
    torch.cuda.synchronize()
    for key in ("bits_tok", "bits_chan", "plan"):
        assert torch.equal(comp.alloc_out[key], al[key]), key
    _same_cache(cache, ref, shape, w.window)
    opack = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                   cap_c=cap)
    qn, kn, vn = synth.decode_step(w, 0)
    out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
    O.append(opack, kn.numpy(), vn.numpy())
    assert np.abs(out.cpu().numpy() - O.decode(opack, qn.numpy())).max() <= 2e-3
    assert rdkv.rdkv_decode_status(cache) == 0
