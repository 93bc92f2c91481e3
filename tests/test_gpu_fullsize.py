"""GPU parity at the full sizes of the configured workloads, in the launch configuration
bench.py times (one fused decode step per layer and decode step), against the CPU oracle on
what it can compute at that size: every output of the allocation and the pack, the decode of
every head (or of sampled sequences and heads), and the weights of the last query rows' columns
plus the properties that hold at any size.

Inputs come from the seeded generators on the device (the same module serves both sides) and
are copied to the host for the oracle.
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


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-30)


def _compress(w, avg, steps):
    q, k, v = synth.prefill_batch(w, device=DEV)
    shape = rdkv.shape_of(q, k, w.window)
    sc = rdkv.rdkv_score(shape, q, k, v)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg)
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    cache = rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], w.window + steps, sizes=sizes)
    torch.cuda.synchronize()
    return (q, k, v), shape, sc, al, sizes, cache


def _check_weights(w, q, k, v, sc, b, tail_rows):
    """Sequence b: sum of w_t, the last columns' w_t, channel weights and spreads."""
    qb, kb, vb = (t[b].float().cpu().numpy() for t in (q, k, v))
    w_tok = sc["w_tok"][b].cpu().numpy()
    N = w.n_tokens
    # every softmax row sums to 1 over the G heads of a group
    assert np.all(np.abs(w_tok.astype(np.float64).sum(axis=1) - N * w.group) <= 1e-3 * N * w.group)
    # columns t >= N - R only receive rows tau >= t: exact from the last R rows
    ref = O.token_weights(qb, kb, first_row=N - tail_rows)[:, N - tail_rows:]
    assert _rel(w_tok[:, N - tail_rows:], ref).max() <= 1e-3
    assert _rel(sc["w_chan"][b].cpu().numpy(), O.channel_weights(qb, kb)).max() <= 1e-3
    assert _rel(sc["sigma_tok"][b].cpu().numpy(), O.value_spread(vb)).max() <= 1e-3


def _check_interior_columns(w, q, k, sc, b, j, t0, width):
    """w_t of KV head j for the interior columns [t0, t0 + width), element by element: those
    columns receive attention only from rows tau >= t0, so the oracle over those rows of the
    group's G query heads (each row normalised over all its keys) is exact for them."""
    G = w.group
    qb = q[b, :, j * G:(j + 1) * G].float().cpu().numpy()
    kb = k[b, :, j:j + 1].float().cpu().numpy()
    ref = O.token_weights(qb, kb, first_row=t0)[0, t0:t0 + width]
    got = sc["w_tok"][b, j, t0:t0 + width].cpu().numpy()
    assert _rel(got, ref).max() <= 1e-3, (j, t0, _rel(got, ref).max())


def _check_alloc_and_plan(w, k, sc, al, avg, seqs):
    g_tok = sc["g_tok"].cpu().numpy()
    bits_tok = al["bits_tok"].cpu().numpy()
    g_chan = al["g_chan"].cpu().numpy()
    bits_chan = al["bits_chan"].cpu().numpy()
    hdr, heads, slots, lam = rdkv.read_plan(al["plan"])
    for b in range(w.batch):
        rb, rl = O.waterfill(g_tok[b], avg)                 # identical gains -> identical widths
        assert np.array_equal(bits_tok[b].ravel(), rb), b
        assert float(lam[b]) == float(rl)
        rb, rl = O.waterfill(g_chan[b], avg)
        assert np.array_equal(bits_chan[b].ravel(), rb), b
    for b in seqs:
        sig = O.kept_channel_spread(k[b].float().cpu().numpy(), bits_tok[b])
        got = al["sigma_chan"][b].cpu().numpy()
        assert _rel(got, sig)[sig > 0].max() <= 1e-5
    plan = O.make_plan(bits_tok, bits_chan, w.head_dim)
    for key in ("zone_a_bytes", "zone_b_rows", "index_slots", "kept_tokens", "max_tile_bytes", "max_stage_bytes"):
        assert int(hdr[key]) == plan[key], key
    return bits_tok, bits_chan, heads


def _oracle_cache(w, k, v, bits_tok, bits_chan, b, heads_of_b, cap_c):
    """Oracle pack of sequence b (its KV heads), and the GPU's zone-A byte range of those heads."""
    ref = O.pack(k[b:b + 1].float().cpu().numpy(), v[b:b + 1].float().cpu().numpy(), bits_tok[b:b + 1],
                 bits_chan[b:b + 1], w.window, cap_c=cap_c)
    a0 = int(heads_of_b[0]["a_off"])
    a1 = int(heads_of_b[-1]["a_off"]) + int(heads_of_b[-1]["a_bytes"])
    return ref, a0, a1


def _check_pack_and_decode(w, cache, ref, a0, a1, b, steps):
    za = cache.zone_a.cpu().numpy()[a0:a1]
    assert za.size == ref["zone_a"].size and np.array_equal(za, ref["zone_a"]), b
    un = O.unpack(ref, w.head_dim)
    return un


def _decode_steps(w, cache, steps, check):
    """Fused steps in the benchmark's launch configuration; check(step, out, qn, kn, vn) per step."""
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step, device=DEV)
        out = rdkv.rdkv_decode_step(cache, qn, kn, vn)
        check(step, out.cpu().numpy(), qn.cpu().numpy(), kn.cpu().numpy(), vn.cpu().numpy())
    assert rdkv.rdkv_decode_status(cache) == 0


def test_llama3b_layer_full_size():
    """The benchmark's workload: Llama-3.2-3B-shaped layer, N = 32768, 2.5 bits, every head checked."""
    w = synth.WORKLOADS["llama3b"]
    steps = 3
    (q, k, v), shape, sc, al, sizes, cache = _compress(w, w.budgets[0], steps)
    _check_weights(w, q, k, v, sc, 0, tail_rows=16)
    # a block of 64 interior columns of one KV head at N/2: 64 key tiles of 256 precede it and 128
    # query blocks of 128 rows contribute to it
    _check_interior_columns(w, q, k, sc, 0, 5, w.n_tokens // 2, 64)
    bits_tok, bits_chan, heads = _check_alloc_and_plan(w, k, sc, al, w.budgets[0], seqs=[0])
    ref, a0, a1 = _oracle_cache(w, k, v, bits_tok, bits_chan, 0, heads[: w.h_kv], w.window + steps)
    un = _check_pack_and_decode(w, cache, ref, a0, a1, 0, steps)
    assert np.array_equal(cache.zone_b.cpu().numpy()[: ref["zone_b"].shape[0]].view(np.uint16),
                          ref["zone_b"].view(np.uint16))

    def check(step, out, qn, kn, vn):
        O.append(ref, kn, vn)
        exp = O.decode(ref, qn, unpacked=un)
        assert np.abs(out - exp).max() <= 2e-3, (step, np.abs(out - exp).max())

    _decode_steps(w, cache, steps, check)


def test_batched_decode_sampled_sequences():
    """8 sequences x N = 32768 with independent allocations (2 bits): allocations of all, pack and
    decode of sequences 0 and 5."""
    w = synth.WORKLOADS["batched"]
    steps = 2
    (q, k, v), shape, sc, al, sizes, cache = _compress(w, w.budgets[0], steps)
    for b in (0, 7):
        assert np.all(np.abs(sc["w_tok"][b].double().sum(dim=1).cpu().numpy() - w.n_tokens * w.group)
                      <= 1e-3 * w.n_tokens * w.group)
    bits_tok, bits_chan, heads = _check_alloc_and_plan(w, k, sc, al, w.budgets[0], seqs=[0, 5])
    refs = {}
    for b in (0, 5):
        ref, a0, a1 = _oracle_cache(w, k, v, bits_tok, bits_chan, b, heads[b * w.h_kv:(b + 1) * w.h_kv],
                                    w.window + steps)
        refs[b] = (ref, _check_pack_and_decode(w, cache, ref, a0, a1, b, steps))

    def check(step, out, qn, kn, vn):
        for b, (ref, un) in refs.items():
            O.append(ref, kn[b:b + 1], vn[b:b + 1])
            exp = O.decode(ref, qn[b:b + 1], unpacked=un)
            assert np.abs(out[b:b + 1] - exp).max() <= 2e-3, (step, b)

    _decode_steps(w, cache, steps, check)


@pytest.mark.parametrize("budget", [0.4, 1.0, 2.0, 4.0])
def test_llama8b_budget_sweep(budget):
    """Llama-3.1-8B-shaped layer, N = 131072, Zipf salience: allocation of every unit at each budget;
    the pack and decode of KV head 0 at the 2.5 %-retention and 2-bit budgets."""
    w = synth.WORKLOADS["llama8b"]
    steps = 1
    (q, k, v), shape, sc, al, sizes, cache = _compress(w, budget, steps)
    if budget == 0.4:
        _check_weights(w, q, k, v, sc, 0, tail_rows=8)
    bits_tok, bits_chan, heads = _check_alloc_and_plan(w, k, sc, al, budget, seqs=[0])
    if budget not in (0.4, 2.0):
        return
    # KV head 0 alone: its layout depends only on its own widths
    k0, v0 = k[:, :, :1], v[:, :, :1]
    ref = O.pack(k0.float().cpu().numpy(), v0.float().cpu().numpy(), bits_tok[:, :1], bits_chan[:, :1], w.window,
                 cap_c=w.window + steps)
    hp = heads[0]
    za = cache.zone_a.cpu().numpy()[int(hp["a_off"]):int(hp["a_off"]) + int(hp["a_bytes"])]
    assert np.array_equal(za, ref["zone_a"])
    un = O.unpack(ref, w.head_dim)

    def check(step, out, qn, kn, vn):
        O.append(ref, kn[:, :1], vn[:, :1])
        exp = O.decode(ref, qn[:, : w.group], unpacked=un)
        assert np.abs(out[:, : w.group] - exp).max() <= 2e-3

    _decode_steps(w, cache, steps, check)


def test_qwen72b_layer_sampled_head():
    """Qwen2.5-72B-shaped layer, N = 262144 (one of the stack's layers): allocation of every unit,
    pack and decode of KV head 5."""
    w = synth.WORKLOADS["qwen72b"]
    steps = 1
    (q, k, v), shape, sc, al, sizes, cache = _compress(w, w.budgets[0], steps)
    assert np.all(np.abs(sc["w_tok"][0].double().sum(dim=1).cpu().numpy() - w.n_tokens * w.group)
                  <= 1e-3 * w.n_tokens * w.group)
    bits_tok, bits_chan, heads = _check_alloc_and_plan(w, k, sc, al, w.budgets[0], seqs=[])
    j = 5
    kj, vj = k[:, :, j:j + 1], v[:, :, j:j + 1]
    ref = O.pack(kj.float().cpu().numpy(), vj.float().cpu().numpy(), bits_tok[:, j:j + 1], bits_chan[:, j:j + 1],
                 w.window, cap_c=w.window + steps)
    hp = heads[j]
    za = cache.zone_a.cpu().numpy()[int(hp["a_off"]):int(hp["a_off"]) + int(hp["a_bytes"])]
    assert np.array_equal(za, ref["zone_a"])
    un = O.unpack(ref, w.head_dim)
    G = w.group

    def check(step, out, qn, kn, vn):
        O.append(ref, kn[:, j:j + 1], vn[:, j:j + 1])
        exp = O.decode(ref, qn[:, j * G:(j + 1) * G], unpacked=un)
        assert np.abs(out[:, j * G:(j + 1) * G] - exp).max() <= 2e-3

    _decode_steps(w, cache, steps, check)


def test_llama3b_layer_recompression_full_size():
    """Llama-3.2-3B-shaped layer at N = 32768, as the benchmark's re-compression measurement runs it:
    W + 8 fused decode steps with lse, the rows beyond the window moved into a segment from the last
    32 queries, then one decode launch over segment and cache.  Checked for a sampled KV head against
    the oracle: the rows, the widths at the prefill's levels (given the library's gains), the
    segment's bytes and the merged attention of the head's query heads."""
    w = synth.WORKLOADS["llama3b"]
    steps = w.window + 8
    (q, k, v), shape, sc, al, sizes, cache = _compress(w, w.budgets[0], steps)
    G, j = w.group, 3
    qs, ls = [], []
    for step in range(steps):
        qn, kn, vn = synth.decode_step(w, step)
        _, lse = rdkv.rdkv_decode_step_lse(cache, qn.to(DEV), kn.to(DEV), vn.to(DEV))
        qs.append(qn.to(DEV))
        ls.append(lse.clone())
    assert rdkv.rdkv_decode_status(cache) == 0
    R = 32
    q_rec, lse_rec = torch.stack(qs[-R:], 1).contiguous(), torch.stack(ls[-R:], 1).contiguous()
    n_move = cache.len_c - w.window
    zk_before, zv_before = (t.cpu().numpy().copy() for t in cache.zone_c_rows())
    seg = rdkv.recompress(cache, al["plan"], sc["w_chan"], q_rec, lse_rec, n_move)
    sc_seg, al_seg = seg._keep
    rk = zk_before[0, :, :n_move].transpose(1, 0, 2)  # [n, H_kv, D]
    rv = zv_before[0, :, :n_move].transpose(1, 0, 2)
    # weights of head j from the oracle on the same recent queries and lse
    eg = O.recompress_gains(rk, rv, q_rec[0].cpu().numpy(), lse_rec[0].cpu().numpy(), w.n_tokens / R)
    assert _rel(sc_seg["w_tok"][0, j].cpu().numpy(), eg["w_tok"][j]).max() <= 1e-3
    lam = rdkv.plan_levels(al["plan"]).cpu().numpy()
    g_tok = sc_seg["g_tok"][0].cpu().numpy()
    bits_tok = al_seg["bits_tok"][0].cpu().numpy()
    assert np.array_equal(bits_tok.ravel(), O.widths_at(O.breakpoints(g_tok), lam[0]))
    g_chan = al_seg["g_chan"][0].cpu().numpy()
    bits_chan = al_seg["bits_chan"][0].cpu().numpy()
    assert np.array_equal(bits_chan.ravel(), O.widths_at(O.breakpoints(g_chan), lam[1]))
    # the segment's bytes of head j
    ref_seg = O.pack(rk[None, :, j:j + 1], rv[None, :, j:j + 1], bits_tok[None, j:j + 1], bits_chan[None, j:j + 1], 0,
                     cap_c=0)
    _, heads_seg, _, _ = rdkv.read_plan(al_seg["plan"])
    hp = heads_seg[j]
    za = seg.zone_a.cpu().numpy()[int(hp["a_off"]):int(hp["a_off"]) + int(hp["a_bytes"])]
    assert np.array_equal(za, ref_seg["zone_a"])
    # one launch over segment and cache, head j's query heads against the oracle
    bits_pre = al["bits_tok"].cpu().numpy()[:, j:j + 1]
    chan_pre = al["bits_chan"].cpu().numpy()[:, j:j + 1]
    ref = O.pack(k[:, :, j:j + 1].float().cpu().numpy(), v[:, :, j:j + 1].float().cpu().numpy(), bits_pre, chan_pre,
                 w.window, cap_c=w.window)
    zk, zv = (t.cpu().numpy() for t in cache.zone_c_rows())
    ref["zone_c_k"][:, :, :w.window] = zk[:, j:j + 1, :w.window]
    ref["zone_c_v"][:, :, :w.window] = zv[:, j:j + 1, :w.window]
    ref["len_c"] = w.window
    qn = synth.decode_step(w, steps)[0]
    out, lse = rdkv.MultiDecode([seg, cache]).attn(qn.to(DEV))
    qh = qn.numpy()[:, j * G:(j + 1) * G]
    o1, l1 = O.decode_lse(ref_seg, qh)
    o2, l2 = O.decode_lse(ref, qh)
    exp, exp_lse = O.merge_attention(np.stack([o1, o2]), np.stack([l1, l2]))
    assert np.abs(out.cpu().numpy()[:, j * G:(j + 1) * G] - exp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy()[:, j * G:(j + 1) * G] - exp_lse).max() <= 2e-3


def test_early_columns_token_weights():
    """w_t of the early columns [256, 320) of one KV head on a 3B-shaped layer of N = 8192, element
    by element against the oracle over the rows tau >= 256 (exact for those columns): the 62
    query blocks of 128 rows from row 256 on contribute to every one of its columns."""
    w = synth.WORKLOADS["llama3b"].scaled(n_tokens=8192)
    q, k, v = synth.prefill_batch(w, device=DEV)
    shape = rdkv.shape_of(q, k, w.window)
    sc = rdkv.rdkv_score(shape, q, k, v)
    torch.cuda.synchronize()
    _check_interior_columns(w, q, k, sc, 0, 2, 256, 64)


def test_ragged_batch_full_size_sampled_sequences():
    """The benchmark's ragged batch: eight Llama-3.2-3B-shaped sequences of 32768 down to 4096 prompt
    tokens, each compressed on its own at 2.5 bits, zones A and B in one shuffled page pool, one
    rdkv_decode_ragged launch.  Sequences 0, 4 and 7 (32768, 16384 and 4096 tokens): their zones
    gathered back through the page tables equal the oracle's pack byte for byte, and their outputs
    and log-sum-exps match the oracle's decode of each sequence alone."""
    base = synth.WORKLOADS["llama3b"]
    lengths = (32768, 28672, 24576, 20480, 16384, 12288, 8192, 4096)
    avg, D = base.budgets[0], base.head_dim
    packs = []
    for i, n in enumerate(lengths):
        w = base.scaled(n_tokens=n)
        q, k, v = (t[None].to(DEV) for t in synth.prefill(w, i, 0))
        shape = rdkv.shape_of(q, k, w.window)
        sc = rdkv.rdkv_score(shape, q, k, v)
        al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg)
        packs.append((shape, al, k, v, rdkv.rdkv_plan_sizes(al["plan"])))
        del q, sc
    a_pages = sum(-(-int(p[4].zone_a_bytes) // rdkv.A_PAGE_BYTES) for p in packs)
    b_pages = sum(max(1, -(-int(p[4].zone_b_rows) // rdkv.B_PAGE_ROWS)) for p in packs)
    pool = rdkv.ZonePool(D, a_pages, b_pages, DEV, seed=3)
    caches = [rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], base.window, sizes=sizes,
                             ab_pool=pool) for shape, al, k, v, sizes in packs]
    qs = [synth.decode_step(base.scaled(n_tokens=n), 0, 0)[0][0] for n in lengths]
    lse = torch.empty(len(lengths), base.h_q, dtype=torch.float32, device=DEV)
    rd = rdkv.RaggedDecode(caches)
    out = rd.attn(torch.stack(qs).to(DEV), lse=lse).cpu().numpy()
    assert rd.status() == rdkv.RDKV_OK
    lse = lse.cpu().numpy()
    for i in (0, 4, 7):
        shape, al, k, v, sizes = packs[i]
        ref = O.pack(k.float().cpu().numpy(), v.float().cpu().numpy(), al["bits_tok"].cpu().numpy(),
                     al["bits_chan"].cpu().numpy(), base.window, cap_c=base.window)
        za = caches[i].zone_a_bytes().cpu().numpy()
        assert za.size == ref["zone_a"].size and np.array_equal(za, ref["zone_a"]), i
        zb = caches[i].zone_b_rows().cpu().numpy()
        assert np.array_equal(zb.view(np.uint16)[: ref["zone_b"].shape[0]], ref["zone_b"].view(np.uint16)), i
        exp, exp_lse = O.decode_lse(ref, qs[i][None].numpy())
        assert np.abs(out[i] - exp[0]).max() <= 2e-3, i
        assert np.abs(lse[i] - exp_lse[0]).max() <= 2e-3, i
