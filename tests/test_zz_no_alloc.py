"""The decode entry point that allocates nothing.

Callers that cannot allocate device memory (a plugin inside an engine that
owns all device allocations, or a serving path where allocation is not
allowed) use rdkv_decode_attn_noalloc, which keeps its scratch in a fixed
array built into the library.  It must give the same output as
rdkv_decode_attn with a caller workspace, call after call, and refuse caches
whose scratch would not fit.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixed_bit_kv_gb300 import rdkv, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _packed_cache(w, steps):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in synth.prefill_batch(w))
    shape = rdkv.shape_of(q, k, w.window)
    sc = rdkv.rdkv_score(shape, q, k, v)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, w.budgets[0], w.budgets[0])
    return rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], w.window + steps)


@pytest.mark.parametrize("case", ["small_f16", "tiny_f32"])
def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls(case):
    w = {"small_f16": synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2),
         "tiny_f32": synth.WORKLOADS["tiny"]}[case]
    dev = torch.device("cuda:0")
    cache = _packed_cache(w, steps=2)
    for step in range(2):                       # two calls in a row, the scratch keeps the last call's contents
        qn, kn, vn = (t.to(dev) for t in synth.decode_step(w, step))
        rdkv.rdkv_append(cache, kn, vn)
        ref = rdkv.rdkv_decode_attn(cache, qn)
        out = torch.full_like(ref, float("nan"))
        rdkv.rdkv_decode_attn_noalloc(cache, qn, out)
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= 2e-3, (case, step, err)


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
