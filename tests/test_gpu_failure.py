"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The decode's every wait on a tile copy is bounded; when one runs out the kernel
records RDKV_ERR_TIMEOUT in the call's status word and returns, so the context
stays usable.  `rdkv_decode_timeout_selftest` runs the decode kernel with every
stage armed for bytes that no copy delivers (and no copy issued), so each
warp's first wait runs out after a short limit.  Checked: the host reads
TIMEOUT with its message, the word is cleared by the read, and a normal call on
the same cache, workspace and context right after matches the oracle.
"""
import time

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


def _cache(w, avg):
    q, k, v = synth.prefill_batch(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    shape = rdkv.shape_of(qd, kd, w.window)
    sc = rdkv.rdkv_score(shape, qd, kd, vd)
    al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], kd, avg, avg)
    cache = rdkv.rdkv_pack(shape, al["plan"], kd, vd, al["bits_tok"], al["bits_chan"], w.window + 4)
    ref = O.pack(k.numpy(), v.numpy(), al["bits_tok"].cpu().numpy(), al["bits_chan"].cpu().numpy(), w.window,
                 cap_c=w.window + 4)
    cache._keep = (al, kd, vd)
    return cache, ref


@pytest.mark.parametrize("case", ["small_f16", "tiny_f32"])
def test_decode_wait_that_runs_out_reports_timeout(case):
    w = (synth.WORKLOADS["llama3b"].scaled(n_tokens=1000, h_q=6, h_kv=2, window=40, batch=2)
         if case == "small_f16" else synth.WORKLOADS["tiny"])
    cache, ref = _cache(w, w.budgets[0])
    qn, _, _ = synth.decode_step(w, 0)
    qd = qn.to(DEV)
    assert rdkv.rdkv_decode_status(cache) == rdkv.RDKV_OK
    t0 = time.perf_counter()
    rdkv.rdkv_decode_timeout_selftest(cache, qd, wait_cycles=2_000_000)  # about 1 ms per wait
    status = rdkv.rdkv_decode_status(cache)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == rdkv.RDKV_ERR_TIMEOUT
    assert b"bounded wait" in rdkv.lib().rdkv_last_error_string()
    assert elapsed < 10.0  # the waits are bounded: two limits per warp, far below a second
    # the read cleared the word; the context, the cache and the workspace (tickets back at zero) still serve
    assert rdkv.rdkv_decode_status(cache) == rdkv.RDKV_OK
    out = rdkv.rdkv_decode_attn(cache, qd)
    assert rdkv.rdkv_decode_status(cache) == rdkv.RDKV_OK
    exp = O.decode(ref, qn.numpy())
    assert np.abs(out.cpu().numpy() - exp).max() <= 2e-3


def test_selftest_argument_check():
    w = synth.WORKLOADS["tiny"]
    cache, _ = _cache(w, w.budgets[0])
    qn, _, _ = synth.decode_step(w, 0)
    with pytest.raises(rdkv.RDKVError):
        rdkv.rdkv_decode_timeout_selftest(cache, qn.to(DEV), wait_cycles=0)
