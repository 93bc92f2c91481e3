"""GPU parity of the paged zone C (block-table indirection): the same cache with its zone C in
16-row pages of a pool, in a shuffled order, against the contiguous cache and the oracle.  Rows
are bit-exact (the indirection moves fp16 rows, it computes nothing); attention within 2e-3 of
the oracle."""
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
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _two_caches(w, cap_extra, seed):
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, w.budgets[0], w.budgets[0])
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    cap = w.window + cap_extra
    flat = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], cap, sizes=sizes)
    pool = rdkv.page_pool(shape, cap, DEV, extra_pages=5, seed=seed)
    paged = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], cap, sizes=sizes, pages=pool)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=cap)
    return sc, al, flat, paged, ref


def _rows_equal(flat, paged, n):
    fk, fv = flat.zone_c_rows()
    pk, pv = paged.zone_c_rows()
    return torch.equal(fk[:, :, :n], pk[:, :, :n]) and torch.equal(fv[:, :, :n], pv[:, :, :n])


@pytest.mark.parametrize("case", list(CASES))
def test_paged_zone_c_steps_match_contiguous_and_oracle(case):
    w = CASES[case]
    steps = 20
    sc, al, flat, paged, ref = _two_caches(w, steps + 2, seed=3)
    assert _rows_equal(flat, paged, w.window)
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        if step % 2:  # fused step on both
            o_flat = rdkv.rdkv_decode_step(flat, qn.to(DEV), kn.to(DEV), vn.to(DEV))
            o_paged = rdkv.rdkv_decode_step(paged, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        else:  # append, then attend
            for c in (flat, paged):
                rdkv.rdkv_append(c, kn.to(DEV), vn.to(DEV))
            o_flat = rdkv.rdkv_decode_attn(flat, qn.to(DEV))
            o_paged = rdkv.rdkv_decode_attn(paged, qn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        exp = O.decode(ref, qn.numpy())
        assert np.abs(o_paged.cpu().numpy() - exp).max() <= 2e-3, step
        # the same attention up to the order in which warps take tiles (both are held to the oracle)
        assert (o_paged - o_flat).abs().max().item() <= 2e-3
    assert paged.len_c == flat.len_c == w.window + steps and int(paged.len_dev.item()) == w.window + steps
    assert _rows_equal(flat, paged, w.window + steps)
    rk, rv = paged.zone_c_rows()
    L = w.window + steps
    assert np.array_equal(rk[:, :, :L].cpu().numpy(), ref["zone_c_k"][:, :, :L])
    assert rdkv.rdkv_decode_status(paged) == 0


def test_paged_live_cache_recompression_and_one_launch_decode():
    """Rows moved out of a paged zone C equal those of the contiguous cache; the decode over
    segment and paged live cache in one launch matches the oracle."""
    w = CASES["small_f16"]
    steps = w.window + 8
    sc, al, flat, paged, ref = _two_caches(w, steps, seed=9)
    qs, ls = [], []
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        rdkv.rdkv_decode_step(flat, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        _, lse = rdkv.rdkv_decode_step_lse(paged, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        qs.append(qn.to(DEV))
        ls.append(lse.clone())
    n_move = paged.len_c - w.window
    kf, vf = rdkv.rdkv_zone_c_take(flat, n_move)
    kp, vp = rdkv.rdkv_zone_c_take(paged, n_move)
    assert torch.equal(kf, kp) and torch.equal(vf, vp)
    assert _rows_equal(flat, paged, w.window)
    rk, rv = O.take_zone_c(ref, n_move)
    assert np.array_equal(kp.cpu().numpy(), rk)
    seg = rdkv.recompress_from_rows(paged, kp, vp, al["plan"], sc["w_chan"], torch.stack(qs, 1).contiguous(),
                                    torch.stack(ls, 1).contiguous())
    al_seg = seg._keep[1]
    seg_ref = O.pack(rk, rv, al_seg["bits_tok"].cpu().numpy(), al_seg["bits_chan"].cpu().numpy(), 0, cap_c=0)
    qn = synth.decode_step(w, steps)[0]
    out, lse = rdkv.MultiDecode([seg, paged]).attn(qn.to(DEV))
    parts = [O.decode_lse(seg_ref, qn.numpy()), O.decode_lse(ref, qn.numpy())]
    exp, exp_lse = O.merge_attention(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - exp_lse).max() <= 2e-3
