"""The whole compression (weights, allocation, pack) captured in one CUDA graph: zones sized from
rdkv_zone_bounds, no host synchronisation inside.  After a replay the zones are bit-exact with the
step-by-step path (which reads the plan sizes back in between), and the decode over the cache matches
the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

CASES = {
    "small_f16": synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2,
                                                   decode_steps=6),
    "zipf_f16": synth.WORKLOADS["llama8b"].scaled(n_tokens=1500, h_q=8, h_kv=2, window=128, batch=1),
    "tiny_f32": synth.WORKLOADS["tiny"],
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("case", list(CASES))
def test_compression_in_one_graph(case):
    w = CASES[case]
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    avg = w.budgets[0]
    cap = w.window + 4
    comp = rdkv.Compressor(shape, avg, avg, cap, DEV)
    comp.run(qd, kd, vd)            # once eagerly (kernel attributes are set outside the capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        comp.run(qd, kd, vd)
    comp.cache.zone_a.zero_()
    comp.cache.zone_b.zero_()
    g.replay()
    cache = comp.finish()
    # the step-by-step path
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg, avg)
    ref_cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], cap)
    sizes = ref_cache.sizes
    assert cache.sizes.zone_a_bytes == sizes.zone_a_bytes and cache.sizes.index_slots == sizes.index_slots
    assert sizes.zone_a_bytes <= comp.bounds.zone_a_bytes and sizes.zone_b_rows <= comp.bounds.zone_b_rows
    na, nb = sizes.zone_a_bytes, sizes.zone_b_rows
    assert torch.equal(cache.zone_a[:na], ref_cache.zone_a[:na])
    assert torch.equal(cache.zone_b[:nb], ref_cache.zone_b[:nb])
    assert torch.equal(cache.index_map[:sizes.index_slots], ref_cache.index_map[:sizes.index_slots])
    assert torch.equal(comp.alloc_out["bits_tok"], al["bits_tok"])
    # decode over the graph-built cache against the oracle
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=cap)
    qn, kn, vn = synth.decode_step(w, 0)
    out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
    O.append(ref, kn.numpy(), vn.numpy())
    assert np.abs(out.cpu().numpy() - O.decode(ref, qn.numpy())).max() <= 2e-3
    assert rdkv.rdkv_decode_status(cache) == 0
