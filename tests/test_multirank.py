"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2).

Each rank compresses and decodes its own sequences; the only collective is the
max-over-ranks reduction of the timings.  These tests run that host logic with
the gloo backend, and the reference arm under torchrun (rank 0 alone prints).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    from mixed_bit_kv_gb300 import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        w = synth.WORKLOADS["tiny"]
        first, last = bench.rank_sequences(rank, w.batch)
        # this rank's inputs come from its own sequences' seeds
        q, k, v = synth.prefill(w, first, 0)
        digest = float(q.double().sum() + 3 * k.double().sum() + 7 * v.double().sum())
        digests = [None] * ws
        dist.all_gather_object(digests, digest)
        # per-rank totals: the reduction keeps the slowest rank's
        mine = [10.0 + rank, 5.0 - rank, 2.5 * (rank + 1)]
        got = bench.max_over_ranks(mine, ws, torch.device("cpu"))
        rate = bench.whole_job_rate(ws, 1000.0, got[1] * 1e-3)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"first": first, "last": last, "digests": digests, "max": got, "rate": rate}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_sequences_and_take_the_max(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    # disjoint, adjacent sequence ranges
    assert res[0]["last"] == res[1]["first"] and res[0]["first"] < res[0]["last"] < res[1]["last"]
    # the ranks drew different inputs, and agree on what each drew
    assert res[0]["digests"] == res[1]["digests"] and res[0]["digests"][0] != res[0]["digests"][1]
    # element-wise max over ranks, the same on every rank
    for r in res:
        assert r["max"] == [11.0, 5.0, 5.0]
        assert r["rate"] == pytest.approx(2 * 1000.0 / 5.0e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.0, 2.0], 1, torch.device("cpu")) == [1.0, 2.0]
    assert bench.rank_sequences(0, 8) == (0, 8)
    assert bench.whole_job_rate(1, 10.0, 2.0) == 5.0


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
