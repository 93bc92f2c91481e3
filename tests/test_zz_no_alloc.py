"""The decode entry point that allocates nothing.

Callers that cannot allocate device memory (a plugin inside an engine that
owns all device allocations, or a serving path where allocation is not
allowed) use rdkv_decode_attn_noalloc, which keeps its scratch in a fixed
array built into the library.  It must give the oracle's output (and the same
output as rdkv_decode_attn with a caller workspace), call after call, also
when calls on caches of other shapes used the shared scratch in between, and
refuse caches whose scratch would not fit.  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu

CASES = {"small_f16": lambda: synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2),
         "tiny_f32": lambda: synth.WORKLOADS["tiny"],
         "g8_f16": lambda: synth.WORKLOADS["qwen72b"].scaled(n_tokens=1500, h_q=16, h_kv=2, window=64, batch=1)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _packed(w, steps):
    """The library's cache and the oracle's cache of the same widths, both with room for `steps` rows."""
    dev = torch.device("cuda:0")
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, w.budgets[0], w.budgets[0])
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + steps)
    cache._keep = (al, kd, vd)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + steps)
    return cache, ref


@pytest.mark.parametrize("case", ["small_f16", "tiny_f32"])
def test_noalloc_decode_matches_oracle_on_consecutive_calls(case):
    w = CASES[case]()
    dev = torch.device("cuda:0")
    cache, ref = _packed(w, steps=2)
    for step in range(2):                       # two calls in a row, the scratch keeps the last call's contents
        qn, kn, vn = synth.decode_step(w, step)
        rdkv.rdkv_append(cache, kn.to(dev), vn.to(dev))
        O.append(ref, kn.numpy(), vn.numpy())
        expect = O.decode(ref, qn.numpy())
        with_ws = rdkv.rdkv_decode_attn(cache, qn.to(dev))
        out = torch.full_like(with_ws, float("nan"))
        rdkv.rdkv_decode_attn_noalloc(cache, qn.to(dev), out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.abs(got - expect).max() <= 2e-3, (case, step)            # the oracle
        assert np.abs(got - with_ws.cpu().numpy()).max() <= 2e-3, (case, step)   # the workspace path


def test_noalloc_calls_on_different_caches_share_the_scratch():
    """Calls alternate between caches of three shapes (other head counts, group sizes and split
    counts, so the partials and tickets of one call overlap what the previous call left in the
    scratch); a bounded-wait self-test on its own workspace runs in between.  Every call matches
    the oracle."""
    dev = torch.device("cuda:0")
    items = []
    for name in ("small_f16", "g8_f16", "tiny_f32"):
        w = CASES[name]()
        cache, ref = _packed(w, steps=1)
        qn, kn, vn = synth.decode_step(w, 0)
        rdkv.rdkv_append(cache, kn.to(dev), vn.to(dev))
        O.append(ref, kn.numpy(), vn.numpy())
        items.append((name, cache, qn, O.decode(ref, qn.numpy())))
    rdkv.rdkv_decode_timeout_selftest(items[0][1], items[0][2].to(dev), wait_cycles=2_000_000)
    assert rdkv.rdkv_decode_status(items[0][1]) == rdkv.RDKV_ERR_TIMEOUT
    for rnd in range(2):
        for name, cache, qn, expect in items:
            out = torch.full((qn.shape[0], qn.shape[1], qn.shape[2]), float("nan"), device=dev)
            rdkv.rdkv_decode_attn_noalloc(cache, qn.to(dev), out)
            torch.cuda.synchronize()
            assert np.abs(out.cpu().numpy() - expect).max() <= 2e-3, (name, rnd)


def test_noalloc_rejects_caches_beyond_its_scratch():
    L = rdkv.lib()
    s = rdkv.make_shape(64, 262144, 512, 64, 128, 128, "f16")
    sizes = rdkv.Sizes(1 << 36, 0, 1 << 30, 1 << 30, 4096, 4096, 0, 64 * 64)
    fake = 256
    c = rdkv.CacheStruct(s, fake, fake, fake, fake, fake, fake, fake, 1024, 128, sizes)
    assert L.rdkv_decode_workspace_bytes(ctypes.byref(c)) > (4 << 20)
    r = L.rdkv_decode_attn_noalloc(ctypes.byref(c), ctypes.c_void_p(fake), ctypes.c_void_p(fake), None)
    assert r == rdkv.RDKV_ERR_WORKSPACE
    assert b"built-in scratch" in L.rdkv_last_error_string()
