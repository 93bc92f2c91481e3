"""Paged zones A and B, and one decode launch over a ragged batch (sequences of different prompt
lengths whose zones share one pool): the block-table idea of "Matematika KV Cache Compression"
("Solusi 1") applied to the TriZone zones the pack writes.

Paging moves bytes and computes nothing, so the oracle keeps the logical zones: the pages are gathered
back through the tables and compared byte for byte with the oracle's pack, and every sequence of a
ragged launch is compared with the oracle's decode of that sequence alone.
"""
import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    if DEV is None:
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _compress(w, seq, avg, cap_extra, pool=None):
    """One sequence (batch 1) of workload w: the library's cache (zones A and B in `pool` when given)
    and the oracle's pack of the same widths."""
    q, k, v = synth.prefill(w, seq, 0)
    qd, kd, vd = (t[None].to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg, avg)
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + cap_extra,
                           ab_pool=pool)
    cache._keep = (al, kd, vd)
    ref = O.pack(k.numpy()[None], v.numpy()[None], al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(),
                 w.window, cap_c=w.window + cap_extra)
    return cache, ref


def _pool(w, a_pages, b_pages, seed):
    return rdkv.ZonePool(w.head_dim, a_pages, b_pages, DEV, seed=seed)


@pytest.mark.parametrize("case", ["g3_d128", "g8_d128", "g4_d64_f32"])
def test_paged_zones_pack_bytes_and_decode(case):
    w = {"g3_d128": synth.WORKLOADS["llama3b"].scaled(n_tokens=2600, h_q=6, h_kv=2, window=40),
         "g8_d128": synth.WORKLOADS["qwen72b"].scaled(n_tokens=2100, h_q=16, h_kv=2, window=64),
         "g4_d64_f32": synth.WORKLOADS["tiny"].scaled(n_tokens=3000)}[case]
    pool = _pool(w, 16, 64, seed=11)
    cache, ref = _compress(w, 0, w.budgets[0], 2, pool)
    torch.cuda.synchronize()
    assert cache.sizes.zone_a_bytes > rdkv.A_PAGE_BYTES  # tiles cross page boundaries
    # zone A and zone B gathered through the tables equal the oracle's contiguous zones
    za = cache.zone_a_bytes().cpu().numpy()
    assert za.size == ref["zone_a"].size and np.array_equal(za, ref["zone_a"])
    zb = cache.zone_b_rows().cpu().numpy()
    assert np.array_equal(zb.view(np.uint16)[: ref["zone_b"].shape[0]], ref["zone_b"].view(np.uint16))
    for step in range(2):
        qn, kn, vn = synth.decode_step(w, step)
        out = rdkv.rdkv_decode_step(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        exp = O.decode(ref, qn.numpy())
        assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3, (case, step)
    assert rdkv.rdkv_decode_status(cache) == rdkv.RDKV_OK


@pytest.mark.parametrize("case", ["g4", "g8"])
def test_ragged_batch_in_one_launch(case):
    """Sequences of 2500, 700, 1900 and 333 prompt tokens, zones A and B in one shuffled pool (the third
    sequence contiguous), each with its own appended token; one launch; every sequence's output and
    log-sum-exp against the oracle's decode of that sequence alone."""
    base = {"g4": synth.WORKLOADS["llama3b"].scaled(h_q=8, h_kv=2, window=32),
            "g8": synth.WORKLOADS["qwen72b"].scaled(h_q=16, h_kv=2, window=32)}[case]
    lengths = (2500, 700, 1900, 333)
    pool = _pool(base, 24, 96, seed=5)
    caches, refs, qs = [], [], []
    for i, n in enumerate(lengths):
        w = base.scaled(n_tokens=n)
        cache, ref = _compress(w, i, w.budgets[0], 4, None if i == 2 else pool)
        qn, kn, vn = synth.decode_step(w, 0)
        rdkv.rdkv_append(cache, kn.to(DEV), vn.to(DEV))
        O.append(ref, kn.numpy(), vn.numpy())
        caches.append(cache)
        refs.append(ref)
        qs.append(qn[0])
    q = torch.stack(qs).to(DEV)
    rd = rdkv.RaggedDecode(caches)
    lse = torch.empty(len(lengths), base.h_q, dtype=torch.float32, device=DEV)
    out = rd.attn(q, lse=lse)
    assert rd.status() == rdkv.RDKV_OK
    for i, ref in enumerate(refs):
        exp, exp_lse = O.decode_lse(ref, qs[i][None].numpy())
        assert np.abs(out[i].cpu().numpy() - exp[0]).max() <= 2e-3, (case, i)
        assert np.abs(lse[i].cpu().numpy() - exp_lse[0]).max() <= 2e-3, (case, i)
    # a second launch on the same workspace (tickets back at zero) gives the same outputs (up to the
    # order in which the warps happened to take the tiles)
    out2 = rd.attn(q)
    assert torch.allclose(out, out2, rtol=0, atol=1e-5)
    for c in caches:
        c.release()


def test_ragged_batch_with_an_empty_sequence():
    """A sequence whose budget keeps no prefix token (zone C only) beside ones that keep many."""
    base = synth.WORKLOADS["llama3b"].scaled(h_q=6, h_kv=2, window=16)
    caches, refs, qs = [], [], []
    for i, (n, avg) in enumerate(((900, 2.5), (500, 0.0), (1300, 4.0))):
        w = base.scaled(n_tokens=n)
        cache, ref = _compress(w, i, avg, 2)
        qn, _, _ = synth.decode_step(w, 0)
        caches.append(cache)
        refs.append(ref)
        qs.append(qn[0])
    q = torch.stack(qs).to(DEV)
    out = rdkv.RaggedDecode(caches).attn(q)
    for i, ref in enumerate(refs):
        exp = O.decode(ref, qs[i][None].numpy())
        assert np.abs(out[i].cpu().numpy() - exp[0]).max() <= 2e-3, i
