#!/usr/bin/env python
"""Benchmark of the RDKV hot path (score -> allocate -> TriZone pack -> append + decode) on GB300.

One step = compress every layer of a stack of independently generated layers
of the chosen workload (default: the Qwen2.5-72B-shaped layer, N = 262144,
H_q = 64, H_kv = 8, 2 bits, window 128; 4 layers of the 80-layer stack, so the
packed zones the decode rotates through, about 0.6 GB, exceed the 129 MB L2
several times), then run the workload's decode steps over all layers (append
the new token, attend).  Inputs are resident in HBM when the timed region
starts; the decode phase is replayed from a captured CUDA graph.  Per-step
times are medians over the timed steps.

Rank 0 prints one JSON line.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import resource
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TriZone decode attn HBM GB/s (decode us/step and scoring TFLOP/s alongside)"
UNIT = "GB/s"

# layers of each workload's stack in one benchmark step: enough independently packed layers that
# the zones one decode step reads exceed the L2 several times
DEFAULT_LAYERS = {"qwen72b": 4, "llama3b": 28, "batched": 4, "llama8b": 4, "tiny": 8}
# decode-only measurements of other workloads added to the line: (layers, decode steps)
EXTRA_DECODE = {"batched": (3, 64), "llama3b": (16, 64)}
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------- environment
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_sequences(rank, batch):
    """First and one-past-last sequence of this rank: every rank compresses and decodes its own
    `batch` sequences (weak scaling, no data-path exchange)."""
    return rank * batch, (rank + 1) * batch


def max_over_ranks(values, ws, device):
    """Element-wise maximum over ranks of per-rank totals: the slowest rank sets the step time."""
    if ws <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(ws, units_per_rank, seconds):
    """Units all ranks processed per second (each rank processes the same amount)."""
    return ws * units_per_rank / seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, sm_max_mhz=2070.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi samples every 200 ms while running (SM clock, max clock, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def captured_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, or None when
    there is no record for that workload or the kernel's source has changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p))[kernel][workload]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except (OSError, KeyError, ValueError, TypeError):
        return None
    if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec["bytes_per_launch"]


# ---------------------------------------------------------------- algorithmic work
def pack_bytes_per_layer(w, sizes):
    """Bytes the pack must move for one layer (from the plan's totals): K and V rows of the kept
    prefix tokens and of the window read, zones A and B, the index map and the window rows of zone
    C written."""
    P = 2 if w.dtype == "f16" else 4
    win = 2 * w.batch * w.h_kv * w.window * w.head_dim
    read = 2 * int(sizes.kept_tokens) * w.head_dim * P + win * P
    written = int(sizes.zone_a_bytes) + int(sizes.zone_b_rows) * w.head_dim * 2 + int(sizes.index_slots) * 4 + win * 2
    return read + written


def decode_bytes_per_call(heads, D, h_q, batch, len_c):
    """Bytes one decode call must move: zone-A payload of real tokens and channels with the K
    metadata of each head's quantised channels (once per head) and the V metadata of each token,
    zone-B rows of real tokens, len_c zone-C rows per head, q in and out.  Padding excluded."""
    total = 0.0
    for hp in heads:
        n16k, n8k, n4k, n2k, _ = (int(x) for x in hp["n_k"])
        ntok = int(np.sum(hp["n_v"]))
        kq = n8k + n4k + n2k
        total += ntok * (2 * n16k + (8 * n8k + 4 * n4k + 2 * n2k) / 8) + (4 * kq if ntok else 0)
        for n, b in zip(hp["n_v"], (2, 4, 8, 16)):
            total += int(n) * (D * b / 8 + (4 * D / 32 if b < 16 else 0))
        total += len_c * 4 * D
    return total + batch * h_q * D * (2 + 4)


def scorer_flops(w):
    """2 passes x 2*D flops per causal (query head, row, key) pair."""
    return 2 * 2 * w.head_dim * w.h_q * w.batch * w.n_tokens * (w.n_tokens + 1) / 2


def scorer_exps(w):
    """The scorer's second ceiling: one base-2 exponential per causal pair in each of the two passes."""
    return 2 * w.h_q * w.batch * w.n_tokens * (w.n_tokens + 1) / 2


def median(xs):
    return float(statistics.median(xs))


def decode_roofline(dec_bytes_per_launch, value_per_gpu, peaks, workload, time_share=None):
    roof = {"bound": "hbm", "achieved": round(value_per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(value_per_gpu / peaks["hbm_gbs"], 4),
            "traffic": captured_traffic("decode_kernel", workload),
            "algorithmic_bytes_per_launch": int(dec_bytes_per_launch),
            "kernel": "rdkv::decode_kernel (fused append + attend, one launch per layer step)",
            "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    if time_share is not None:
        roof["time_share"] = round(time_share, 3)
    return roof


# ---------------------------------------------------------------- our arm
def run_ours(args, ws, rank, local):
    import torch
    from mixed_bit_kv_gb300 import rdkv, synth

    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    if args.tokens is not None:  # reduced prompt length (profiling captures); the description says so
        w = w.scaled(n_tokens=args.tokens,
                     description=w.description + f" (prompt reduced to N={args.tokens})")
    L = args.layers if args.layers is not None else DEFAULT_LAYERS.get(w.name, 4)
    S = args.decode_steps if args.decode_steps is not None else w.decode_steps
    avg = w.budgets[0] if args.budget is None else args.budget
    first_seq, _ = rank_sequences(rank, w.batch)
    shape = rdkv.make_shape(w.batch, w.n_tokens, w.h_q, w.h_kv, w.head_dim, w.window, w.dtype)
    cap_c = w.window + S

    # inputs resident in HBM
    pre = []
    for layer in range(L):
        qs, ks, vs = zip(*(synth.prefill(w, first_seq + b, layer, device=dev) for b in range(w.batch)))
        pre.append(tuple(torch.stack(t).contiguous() for t in (qs, ks, vs)))
    dq, dk, dv = synth.decode_stream(w, S, L, first_seq, device=dev)
    outs = torch.empty(S, L, w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=dev)

    score_out = [None] * L
    alloc_out = [None] * L
    caches = [None] * L
    lib = rdkv.lib()

    def compress(timing):
        for layer in range(L):
            q, k, v = pre[layer]
            ev4 = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if timing is not None else None
            if ev4:
                ev4[0].record()
            score_out[layer] = rdkv.rdkv_score(shape, q, k, v, out=score_out[layer])
            if ev4:
                ev4[1].record()
            sc = score_out[layer]
            alloc_out[layer] = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg,
                                                  out=alloc_out[layer])
            al = alloc_out[layer]
            if ev4:
                ev4[2].record()
            sizes = rdkv.rdkv_plan_sizes(al["plan"])  # zone sizes for the buffers (synchronises)
            if ev4:
                ev4[2] = torch.cuda.Event(enable_timing=True)  # the pack interval starts after the sizes
                ev4[2].record()
            caches[layer] = rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], cap_c,
                                           into=caches[layer], sizes=sizes)
            if ev4:
                ev4[3].record()
                timing.append(ev4)

    def decode_phase():
        for s in range(S):
            for layer in range(L):
                # append the new token and attend, one launch per layer
                rdkv.rdkv_decode_step(caches[layer], dq[s, layer], dk[s, layer], dv[s, layer], out=outs[s, layer])

    # warm-up: eager once (allocates every buffer), then capture the decode phase
    compress(None)
    for c in caches:
        c.decode_workspace()
    torch.cuda.synchronize()
    n0 = lib.rdkv_launch_count()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        decode_phase()
    decode_launches = lib.rdkv_launch_count() - n0
    for _ in range(max(0, args.warmup - 1)):
        compress(None)
        g.replay()
    torch.cuda.synchronize()
    for c in caches:
        st = rdkv.rdkv_decode_status(c)
        if st != 0:
            raise RuntimeError(f"decode status {st}")

    # algorithmic decode bytes per step (all layers, all decode steps)
    heads_per_layer = [rdkv.read_plan(alloc_out[layer]["plan"])[1] for layer in range(L)]
    dec_bytes = sum(decode_bytes_per_call(h, w.head_dim, w.h_q, w.batch, w.window + s + 1)
                    for h in heads_per_layer for s in range(S))
    kept = sum(int(np.sum(h["n_v"])) for h in heads_per_layer) / (L * w.batch * w.h_kv * w.n_prefix)
    tiles_per_launch = sum(int(np.sum(h["tiles"])) for h in heads_per_layer) / L
    zone_bytes_layer = sum(int(c.c.sizes.zone_a_bytes) + int(c.c.sizes.zone_b_rows) * w.head_dim * 2
                           for c in caches) / L

    # timed region
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(torch.cuda.current_device())

    def timed_steps():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev, score_ev = [], []
        launches0 = lib.rdkv_launch_count()
        with ClockSampler(gpu_id) as clk:
            t0 = time.perf_counter()
            for _ in range(args.steps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                c = torch.cuda.Event(enable_timing=True)
                a.record()
                step_ev = []
                compress(step_ev)
                b.record()
                g.replay()
                c.record()
                ev.append((a, b, c))
                score_ev.append(step_ev)
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
        if ws > 1:
            torch.distributed.barrier()
        return ev, score_ev, clk, wall, lib.rdkv_launch_count() - launches0

    ev, score_ev, clk, wall, compress_launches = timed_steps()
    # a hardware or thermal slowdown during the timed steps: measured once more, the first reasons kept
    slowed = sorted(set(clk.summary()["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"})
    if max_over_ranks([1.0 if slowed else 0.0], ws, dev)[0] > 0:  # every rank takes the same decision
        slowed = slowed or ["on another rank"]
        ev, score_ev, clk, wall, compress_launches = timed_steps()
    gpu_launches = int(compress_launches + args.steps * decode_launches)
    # per-step times; the line reports the median step
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    dec_ms = [b.elapsed_time(c) for a, b, c in ev]
    score_ms = [sum(e[0].elapsed_time(e[1]) for e in se) for se in score_ev]
    alloc_ms = [sum(e[1].elapsed_time(e[2]) for e in se) for se in score_ev]  # incl. the sizes read-back
    pack_ms = [sum(e[2].elapsed_time(e[3]) for e in se) for se in score_ev]
    med = max_over_ranks([median(step_ms), median(dec_ms), median(score_ms), median(alloc_ms), median(pack_ms)],
                         ws, dev)
    ms_per_step, dec_ms_step, score_ms_step, alloc_ms_step, pack_ms_step = med

    value = whole_job_rate(ws, dec_bytes, dec_ms_step * 1e-3) / 1e9
    flops = scorer_flops(w) * L
    score_tflops = whole_job_rate(ws, flops, score_ms_step * 1e-3) / 1e12
    peaks = measured_peaks()
    clocks = clk.summary()
    if slowed:
        clocks["remeasured_after"] = slowed

    dec_frac_time, score_frac_time = dec_ms_step / ms_per_step, score_ms_step / ms_per_step
    decode_roof = decode_roofline(dec_bytes / (S * L), value / ws, peaks, w.name, dec_frac_time)
    # fp16 scorer on the tensor cores: measured dense bf16 peak (fp16 has the same nominal dense rate);
    # the sustained figure, since the scorer runs back to back over every layer inside the step.
    # fp32 inputs run on CUDA cores: roofline against the FP32 FMA peak instead.
    if w.dtype == "f16":
        t1 = captured_traffic("score_kernel_pass1", w.name)
        t2 = captured_traffic("score_kernel_pass2", w.name)
        score_roof = {"bound": "tensor", "achieved": round(score_tflops / ws, 2),
                      "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                      "frac": round(score_tflops / ws / peaks["bf16_tflops_sustained"], 4),
                      "traffic": (t1 + t2) if (t1 and t2) else None, "flops_per_launch_pair": scorer_flops(w),
                      "exp2_per_launch_pair": scorer_exps(w),
                      "exp2_per_s": round(score_tflops / ws * 1e12 * scorer_exps(w) / scorer_flops(w), 1),
                      "exp2_note": "the SFU's share of its peak is an ncu counter (XU pipe active 57-61 %, "
                                   "profiles/score_kernel_llama3b_layer.md)",
                      "kernel": "rdkv::tc::score_kernel (passes 1 and 2)",
                      "peak_source": f"{peaks['source']} bf16 dense sustained (fp16 nominal rate equal)",
                      "time_share": round(score_frac_time, 3)}
    else:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        score_roof = {"bound": "alu", "achieved": round(score_tflops / ws, 2), "peak": round(alu_peak, 1),
                      "unit": "TFLOP/s", "frac": round(score_tflops / ws / alu_peak, 4), "traffic": None,
                      "peak_source": "SMs x 128 FP32 lanes x 2 flops x max SM clock",
                      "time_share": round(score_frac_time, 3)}

    # context, outside the timed steps: the same decode phase replayed from its graph after a pause.
    # Inside a step it starts right after seconds of scoring at the power cap, before the SM clock
    # has recovered.
    time.sleep(0.5)
    alone = []
    for _ in range(3):
        for cch in caches:
            cch.len_dev.fill_(w.window)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        alone.append(e0.elapsed_time(e1))
    alone_ms = max_over_ranks([median(alone)], ws, dev)[0]
    decode_after_pause = {
        "us_per_layer_step": round(alone_ms * 1e3 / (S * L), 3),
        "gbs": round(whole_job_rate(ws, dec_bytes, alone_ms * 1e-3) / 1e9, 1),
        "note": "the step's decode phase replayed alone from its CUDA graph after a 0.5 s pause (median of 3), "
                "outside the timed steps; inside a step it follows the power-capped scoring directly"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, shape, L, S, avg, cap_c, pre, dq, dk, dv, dec_bytes, ws, dev)
    comparator = None
    if not args.no_comparator:
        comparator = run_fp16_comparator(w, L, pre, dq, dev)
        comparator["trizone_speedup"] = round(comparator["us_per_layer_step"] / (dec_ms_step * 1e3 / (S * L)), 2)
    paged = None
    if not args.no_recompress and rank == 0:
        paged = run_paged(w, shape, pre[L - 1], alloc_out[L - 1], cap_c, dq, dk, dv, dev)
    graph_compress = None
    if not args.no_recompress and rank == 0:
        graph_compress = run_graph_compress(w, shape, pre[L - 1], avg, cap_c, dev)
    recompress = None
    if not args.no_recompress and rank == 0:
        recompress = run_recompress(w, caches[L - 1], alloc_out[L - 1]["plan"], score_out[L - 1]["w_chan"], dq, dev)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16" if w.dtype == "f16" else "f32",
        "data": "synthetic (seeded generator, workload shapes and salience structure)",
        "config": {"workload": w.name, "description": w.description, "layers": L, "decode_steps": S,
                   "avg_bits": avg, "batch_per_gpu": w.batch, "kept_fraction": round(kept, 4),
                   "parallelism": f"replicas x{ws} (independent sequences per rank)",
                   "timing": "median over the timed steps (CUDA events on the launching stream)",
                   "l2": (f"inputs larger than L2: {sum(t.numel() * t.element_size() for p in pre for t in p) / 1e9:.1f}"
                          f" GB of prefill inputs; the decode rotates through {L} independently packed layers of "
                          f"{zone_bytes_layer / 1e6:.0f} MB each ({L * zone_bytes_layer / L2_BYTES:.1f}x L2)")},
        "decode_us_per_layer_step": round(dec_ms_step * 1e3 / (S * L), 3),
        "decode_after_pause": decode_after_pause,
        "decode_ms_per_model_step": round(dec_ms_step / S, 4),
        "decode_bytes_per_step": int(dec_bytes),
        "decode_tiles_per_launch": int(round(tiles_per_launch)),
        "scorer_tflops": round(score_tflops, 2), "scorer_ms_per_layer": round(score_ms_step / L, 3),
        "compress_ms_per_layer": round((ms_per_step - dec_ms_step) / L, 3),
        "compress_breakdown_ms_per_layer": {
            "score (weights: tensor-core passes, channel norms, V spreads)": round(score_ms_step / L, 3),
            "allocate (water-filling V and K, channel spreads, plan; sizes read back)": round(alloc_ms_step / L, 3),
            "pack (index map, tiles, zone B, window)": round(pack_ms_step / L, 3)},
        "pack_gbs": round(sum(pack_bytes_per_layer(w, c.c.sizes) for c in caches) / (pack_ms_step * 1e-3) / 1e9, 1),
        "zone_bytes_per_layer": int(zone_bytes_layer),
        "roofline": decode_roof, "rooflines": {"decode": decode_roof, "scorer": score_roof},
        "gpu_launches": gpu_launches, "clocks": clocks, "wall_s": round(wall, 3),
    }
    if w.n_layers > 1:
        fp16_model = 2 * w.n_layers * w.h_kv * w.head_dim * 2 * w.n_tokens * w.batch
        line["hbm_accounting"] = {
            "model_layers": w.n_layers, "fp16_kv_bytes": fp16_model,
            "trizone_bytes_est": int(zone_bytes_layer * w.n_layers
                                     + 2 * w.n_layers * w.batch * w.h_kv * cap_c * w.head_dim * 2),
            "note": "fp16 K+V of the whole stack by the KV-size formula 2*L*H_kv*D*P*N vs the measured zones "
                    "A and B per layer times the layers plus zone C at capacity"}
    if e2e is not None:
        line["e2e"] = e2e
    if comparator is not None:
        line["comparator"] = comparator
    if recompress is not None:
        line["recompress"] = recompress
    if paged is not None:
        line["paged_zone_c"] = paged
    if graph_compress is not None:
        line["compress_in_one_graph"] = graph_compress
    # free this workload's buffers before the other workloads' decode measurements
    del pre, dq, dk, dv, outs, score_out, alloc_out, caches, g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if not args.no_extras and rank == 0:
        line["decode_other_workloads"] = {name: run_decode_only(name, nl, ns, peaks, dev)
                                          for name, (nl, ns) in EXTRA_DECODE.items() if name != w.name}
    if not args.no_recompress and rank == 0:
        line["ragged_batch"] = run_ragged(peaks, dev)
    return line


def run_ragged(peaks, dev, steps=32):
    """A ragged batch, measured beside the path: eight Llama-3.2-3B-shaped sequences with prompt lengths
    32768 down to 4096, each compressed on its own (2.5 bits), zones A and B in pages of one shared pool
    (shuffled page order); per decode step one rdkv_decode_ragged launch over all eight, against eight
    rdkv_decode_attn launches on contiguous caches of the same plans.  CUDA graphs of `steps` steps,
    the query of each step fresh; best of 3."""
    import torch
    from mixed_bit_kv_gb300 import rdkv, synth
    base = synth.WORKLOADS["llama3b"]
    lengths = (32768, 28672, 24576, 20480, 16384, 12288, 8192, 4096)
    avg = base.budgets[0]
    pool_caches, flat, heads, D = [], [], [], base.head_dim
    packs = []
    for i, n in enumerate(lengths):
        w = base.scaled(n_tokens=n)
        q, k, v = (t[None].to(dev) for t in synth.prefill(w, i, 0))
        shape = rdkv.shape_of(q, k, w.window)
        sc = rdkv.rdkv_score(shape, q, k, v)
        al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg)
        sizes = rdkv.rdkv_plan_sizes(al["plan"])
        packs.append((shape, al, k, v, sizes))
        heads.append(rdkv.read_plan(al["plan"])[1])
        del q, sc
    a_pages = sum(-(-int(p[4].zone_a_bytes) // rdkv.A_PAGE_BYTES) for p in packs)
    b_pages = sum(max(1, -(-int(p[4].zone_b_rows) // rdkv.B_PAGE_ROWS)) for p in packs)
    pool = rdkv.ZonePool(D, a_pages, b_pages, dev, seed=3)
    for shape, al, k, v, sizes in packs:
        pool_caches.append(rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], base.window,
                                          sizes=sizes, ab_pool=pool))
        flat.append(rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], base.window,
                                   sizes=sizes))
    qs = torch.stack([torch.stack([synth.decode_step(base.scaled(n_tokens=n), s_, 0)[0][0] for n in lengths])
                      for s_ in range(steps)]).to(dev)      # [steps, 8, H_q, D]
    out = torch.empty(len(lengths), base.h_q, D, dtype=torch.float32, device=dev)
    rd = rdkv.RaggedDecode(pool_caches)
    rd.workspace()
    for c in flat:
        c.decode_workspace()
    torch.cuda.synchronize()

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s_ in range(steps):
                fn(s_)
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b) * 1e3 / steps
            best = t if best is None else min(best, t)
        return best

    us_ragged = timed(lambda s_=0: rd.attn(qs[s_], out=out))
    us_flat = timed(lambda s_=0: [rdkv.rdkv_decode_attn(c, qs[s_, i:i + 1], out=out[i:i + 1])
                                  for i, c in enumerate(flat)])
    if rd.status() != rdkv.RDKV_OK:
        raise RuntimeError("ragged decode status")
    nbytes = sum(decode_bytes_per_call(h, D, base.h_q, 1, base.window) for h in heads)
    res = {"sequences": list(lengths), "avg_bits": avg,
           "us_per_step_one_launch": round(us_ragged, 3), "us_per_step_per_sequence_launches": round(us_flat, 3),
           "gbs_one_launch": round(nbytes / (us_ragged * 1e-6) / 1e9, 1),
           "frac_of_measured_hbm": round(nbytes / (us_ragged * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
           "algorithmic_bytes_per_step": int(nbytes),
           "note": "zones A and B of the eight sequences in 64 KB / 16-row pages of one pool (shuffled); attention "
                   "only, CUDA graphs, best of 3"}
    for c in pool_caches:
        c.release()
    del pool, pool_caches, flat, packs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_decode_only(name, L, S, peaks, dev):
    """Decode of another workload, measured beside the headline: L independently packed layers
    (compressed once, untimed), then S fused decode steps over all layers from a CUDA graph, 3
    timed replays (median).  The layers' zones exceed the L2 several times."""
    import torch
    from mixed_bit_kv_gb300 import rdkv, synth
    w = synth.WORKLOADS[name]
    avg = w.budgets[0]
    shape = rdkv.make_shape(w.batch, w.n_tokens, w.h_q, w.h_kv, w.head_dim, w.window, w.dtype)
    cap_c = w.window + S
    caches, heads = [], []
    for layer in range(L):
        q, k, v = synth.prefill_batch(w, layer, device=dev)
        sc = rdkv.rdkv_score(shape, q, k, v)
        al = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg)
        caches.append(rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], cap_c))
        heads.append(rdkv.read_plan(al["plan"])[1])
        del q, k, v, sc
    dq, dk, dv = synth.decode_stream(w, S, L, 0, device=dev)
    out = torch.empty(w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=dev)
    for c in caches:
        c.decode_workspace()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(S):
            for layer in range(L):
                rdkv.rdkv_decode_step(caches[layer], dq[s, layer], dk[s, layer], dv[s, layer], out=out)
    times = []
    for _ in range(3):
        for c in caches:  # back to the window: every replay attends over the same rows
            c.len_dev.fill_(w.window)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    for c in caches:
        if rdkv.rdkv_decode_status(c) != 0:
            raise RuntimeError(f"{name}: decode status")
    dec_bytes = sum(decode_bytes_per_call(h, w.head_dim, w.h_q, w.batch, w.window + s + 1)
                    for h in heads for s in range(S))
    ms = median(times)
    gbs = dec_bytes / (ms * 1e-3) / 1e9
    zone = sum(int(c.c.sizes.zone_a_bytes) + int(c.c.sizes.zone_b_rows) * w.head_dim * 2 for c in caches) / L
    res = {"description": w.description, "layers": L, "decode_steps": S, "avg_bits": avg,
           "us_per_layer_step": round(ms * 1e3 / (S * L), 3), "gbs": round(gbs, 1),
           "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
           "algorithmic_bytes_per_launch": int(dec_bytes / (S * L)), "zone_bytes_per_layer": int(zone),
           "traffic": captured_traffic("decode_kernel", name)}
    del caches, dq, dk, dv, g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res

def run_fp16_comparator(w, L, pre, dq, dev, steps=16):
    """Context number: decode over the full fp16 cache of the same layers (all N prompt tokens, no
    compression) with torch's scaled_dot_product_attention (a library call), per layer step, replayed
    from a CUDA graph like the TriZone decode.  The caches of all layers are rotated (inputs larger
    than L2)."""
    import torch
    steps = min(steps, dq.shape[0])
    caches = [tuple(t.permute(0, 2, 1, 3).contiguous() for t in (pre[layer][1], pre[layer][2])) for layer in range(L)]
    qs = dq[:steps]  # [steps, L, B, H_q, D]
    out = torch.empty(w.batch, w.h_q, 1, w.head_dim, dtype=qs.dtype, device=dev)

    def run():
        for s in range(steps):
            for layer in range(L):
                k, v = caches[layer]
                out.copy_(torch.nn.functional.scaled_dot_product_attention(
                    qs[s, layer].unsqueeze(2), k, v, enable_gqa=True))

    run()
    torch.cuda.synchronize()
    mode = "graph"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        replay = g.replay
    except Exception:
        mode = "eager"
        replay = run
    replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (steps * L)
    nbytes = 2 * w.batch * w.n_tokens * w.h_kv * w.head_dim * 2
    del caches
    return {"kind": "fp16 full cache (all N prompt tokens), torch scaled_dot_product_attention, " + mode,
            "us_per_layer_step": round(us, 3), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}


def run_recompress(w, cache, prefill_plan, w_chan, dq, dev, recent=32, reps=20):
    """The zone-C re-compression row, measured beside the path on the last layer's cache as the
    timed steps left it (window + decode rows in zone C): the rows beyond the window move into a
    segment (weights from the last `recent` decode queries and their log-sum-exps); reported with
    the decode of the cache before (one launch) and after (segment and live cache: two launches and
    a merge)."""
    import torch
    from mixed_bit_kv_gb300 import rdkv
    S, layer = dq.shape[0], dq.shape[1] - 1
    R = min(recent, S)
    cache.c.len_c = int(cache.len_dev.item())  # graph replays advanced only the device length
    lses = torch.empty(w.batch, R, w.h_q, dtype=torch.float32, device=dev)
    for r in range(R):
        lses[:, r].copy_(rdkv.rdkv_decode_attn_lse(cache, dq[S - R + r, layer])[1])
    q_rec = dq[S - R:, layer].transpose(0, 1).contiguous()
    q = dq[S - 1, layer]
    out = torch.empty(w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=dev)

    def per_call_us(fn):
        """Per call, from a CUDA graph of `reps` calls (as the benchmark's decode phase)."""
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    us_plain = per_call_us(lambda: rdkv.rdkv_decode_attn(cache, q, out=out))
    n_move = cache.len_c - w.window
    if n_move < w.window:
        return {"skipped": f"{n_move} rows beyond the window; a move needs at least as many rows as stay"}
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    seg = rdkv.recompress(cache, prefill_plan, w_chan, q_rec, lses, n_move)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    outs = torch.empty(2, w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=dev)
    lse2 = torch.empty(2, w.batch, w.h_q, dtype=torch.float32, device=dev)
    lse_m = torch.empty(w.batch, w.h_q, dtype=torch.float32, device=dev)

    def segmented():
        rdkv.rdkv_decode_attn_lse(seg, q, out=outs[0], lse=lse2[0])
        rdkv.rdkv_decode_attn_lse(cache, q, out=outs[1], lse=lse2[1])
        rdkv.rdkv_merge_attn(outs, lse2, out=out, lse=lse_m)

    us_seg = per_call_us(segmented)
    md = rdkv.MultiDecode([seg, cache])
    us_multi = per_call_us(lambda: md.attn(q, out=out, lse=lse_m))
    st = seg.c.sizes
    seg_bytes = int(st.zone_a_bytes) + int(st.zone_b_rows) * w.head_dim * 2
    fp16_bytes = 2 * w.batch * n_move * w.h_kv * w.head_dim * 2
    return {"rows_moved": int(n_move), "recent_queries": int(R), "ms_per_layer": round(ms, 3),
            "segment_kept_fraction": round(int(st.kept_tokens) / (w.batch * w.h_kv * n_move), 4),
            "segment_bytes": seg_bytes, "fp16_bytes_of_the_rows": fp16_bytes,
            "decode_us_one_cache": round(us_plain, 3), "decode_us_segment_and_cache": round(us_seg, 3),
            "decode_us_segment_and_cache_one_launch": round(us_multi, 3),
            "note": "take rows + weights from recent queries + widths at the prefill's levels + plan "
                    "(sizes read back) + pack, CUDA events; decodes per call from CUDA graphs: one launch for the "
                    "cache; segment and cache as two launches and a merge, or as one launch over both"}


def run_paged(w, shape, layer_inputs, al, cap_c, dq, dk, dv, dev):
    """Paged zone C, measured beside the path: the last layer packed twice, with a contiguous zone C
    and with its zone C in 16-row pages of a shuffled pool; per-call time of the benchmark's fused
    decode steps (CUDA graph of every step) on each."""
    import torch
    from mixed_bit_kv_gb300 import rdkv
    _, k, v = layer_inputs
    S, layer = dq.shape[0], dq.shape[1] - 1
    sizes = rdkv.rdkv_plan_sizes(al["plan"])
    out = torch.empty(w.batch, w.h_q, w.head_dim, dtype=torch.float32, device=dev)
    res = {}
    for name, pages in (("contiguous", None), ("paged", rdkv.page_pool(shape, cap_c, dev, seed=7))):
        cache = rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], cap_c, sizes=sizes,
                               pages=pages)
        cache.decode_workspace()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in range(S):
                rdkv.rdkv_decode_step(cache, dq[s, layer], dk[s, layer], dv[s, layer], out=out)
        times = []
        for _ in range(3):
            rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], cap_c, sizes=sizes, into=cache)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / S)
        if rdkv.rdkv_decode_status(cache) != 0:
            raise RuntimeError("paged decode status")
        res[name + "_us_per_step"] = round(min(times), 3)
    res["note"] = ("one layer, every decode step of the workload (fused append + attend) from a CUDA graph, "
                   "best of 3; zone C in 16-row pages of a shuffled pool vs contiguous")
    return res


def run_graph_compress(w, shape, layer_inputs, avg, cap_c, dev, reps=3):
    """Compression without host synchronisation, measured beside the path: weights, allocation and
    pack of one layer with zones sized from rdkv_zone_bounds, captured once in a CUDA graph and
    replayed (the benchmark's own compression reads the plan sizes back between allocation and
    pack)."""
    import torch
    from mixed_bit_kv_gb300 import rdkv
    q, k, v = layer_inputs
    comp = rdkv.Compressor(shape, avg, avg, cap_c, dev)
    comp.run(q, k, v)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        comp.run(q, k, v)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    exact = comp.finish()
    res = {"ms_per_layer": round(a.elapsed_time(b) / reps, 3),
           "zone_a_bytes_bound": int(comp.bounds.zone_a_bytes), "zone_a_bytes": int(exact.sizes.zone_a_bytes),
           "note": "score + allocate + pack from one CUDA graph, zones sized by rdkv_zone_bounds"}
    try:
        res["allocate_pack"] = run_allocate_pack_compare(shape, comp, q, k, v, avg, cap_c, dev)
    except Exception as e:  # a refused cooperative launch must not cost the benchmark's line
        res["allocate_pack"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return res


def run_allocate_pack_compare(shape, comp, q, k, v, avg, cap_c, dev, reps=5):
    """Allocation and pack of one layer (the scorer's outputs already in place), each way captured in
    a CUDA graph and replayed: the allocation's and the pack's own kernels (rdkv_allocate, rdkv_pack
    into zones sized by rdkv_zone_bounds) against the one persistent launch (rdkv_allocate_pack).
    Both ways leave byte-identical zones (checked here on zone A)."""
    import ctypes
    import torch
    from mixed_bit_kv_gb300 import rdkv
    L = rdkv.lib()
    so = comp.score_out
    step_out = {key: torch.zeros_like(t) for key, t in comp.alloc_out.items()}
    step_ws = rdkv._ws(L.rdkv_allocate_workspace_bytes(ctypes.byref(shape)), dev)
    step_cache = rdkv.Cache(shape, step_out["plan"], comp.bounds, cap_c, dev)
    one_out = {key: torch.zeros_like(t) for key, t in comp.alloc_out.items()}
    one_ws = rdkv._ws(L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(shape), 0), dev)
    one_cache = rdkv.Cache(shape, one_out["plan"], comp.bounds, cap_c, dev)

    def step_by_step():
        rdkv.rdkv_allocate(shape, so["g_tok"], so["w_chan"], k, avg, avg, out=step_out, ws=step_ws)
        step_cache.c.sizes = comp.bounds
        rdkv._check(L.rdkv_pack(ctypes.byref(step_cache.c), rdkv._ptr(k), rdkv._ptr(v), rdkv._ptr(step_out["bits_tok"]),
                                rdkv._ptr(step_out["bits_chan"]), rdkv._stream()))

    def one_launch():
        rdkv.rdkv_allocate_pack(shape, so["g_tok"], so["w_chan"], k, v, avg, avg, cap_c, out=one_out, ws=one_ws,
                                cache=one_cache)

    def graph_ms(fn):
        n0 = L.rdkv_launch_count()
        fn()
        torch.cuda.synchronize()
        launches = int(L.rdkv_launch_count() - n0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return median(times), launches

    step_ms, step_n = graph_ms(step_by_step)
    one_ms, one_n = graph_ms(one_launch)
    n = int(rdkv.rdkv_plan_sizes(one_out["plan"]).zone_a_bytes)
    same = bool(torch.equal(step_cache.zone_a[:n], one_cache.zone_a[:n])
                and torch.equal(step_out["plan"], one_out["plan"]))
    return {"step_by_step_ms": round(step_ms, 4), "step_by_step_launches": step_n,
            "one_launch_ms": round(one_ms, 4), "one_launch_launches": one_n, "identical_zone_a_and_plan": same,
            "note": "allocation + pack of one layer from CUDA graphs (median of 5 replays): the stage kernels "
                    "against one cooperative persistent kernel"}


def run_e2e(args, w, shape, L, S, avg, cap_c, pre, dq, dk, dv, dec_bytes, ws, dev):
    """The whole step end to end through the public API with pinned host buffers: every layer's
    prefill inputs copied host->device (on a copy stream, so that the next layer's copy overlaps this
    layer's compression), scored, allocated, its plan sizes read back, packed; then
    every decode step's q, k, v copied host->device, the fused append + attend of every layer, and
    the step's outputs copied device->host.  Wall time per step (median); the value is the same
    metric as the line's (decode algorithmic bytes per second), over the whole step's time."""
    import torch
    from mixed_bit_kv_gb300 import rdkv

    h_pre = [tuple(t.cpu().pin_memory() for t in trip) for trip in pre]
    h_dq, h_dk, h_dv = (t.cpu().pin_memory() for t in (dq, dk, dv))
    h_out = torch.empty((S, L, w.batch, w.h_q, w.head_dim), dtype=torch.float32).pin_memory()
    d_pre = [tuple(torch.empty_like(t) for t in trip) for trip in pre]
    d_dq, d_dk, d_dv = (torch.empty_like(t[0]) for t in (dq, dk, dv))   # one decode step, all layers
    d_out = torch.empty((L, w.batch, w.h_q, w.head_dim), dtype=torch.float32, device=dev)
    score_out, alloc_out, caches = [None] * L, [None] * L, [None] * L

    copy_stream = torch.cuda.Stream(device=dev)

    def step_compress():
        # every layer's prefill inputs go host->device on a copy stream, each layer's compression
        # waiting only for its own inputs: the copies of layer l + 1 overlap the compression of layer l
        cur = torch.cuda.current_stream(dev)
        copy_stream.wait_stream(cur)  # the previous step's readers of the device buffers are done
        landed = []
        with torch.cuda.stream(copy_stream):
            for layer in range(L):
                for dst, src in zip(d_pre[layer], h_pre[layer]):
                    dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                landed.append(ev)
        for layer in range(L):
            cur.wait_event(landed[layer])
            q, k, v = d_pre[layer]
            score_out[layer] = rdkv.rdkv_score(shape, q, k, v, out=score_out[layer])
            sc = score_out[layer]
            alloc_out[layer] = rdkv.rdkv_allocate(shape, sc["g_tok"], sc["w_chan"], k, avg, avg,
                                                  out=alloc_out[layer])
            al = alloc_out[layer]
            caches[layer] = rdkv.rdkv_pack(shape, al["plan"], k, v, al["bits_tok"], al["bits_chan"], cap_c,
                                           into=caches[layer])

    def decode_phase():
        for s in range(S):
            d_dq.copy_(h_dq[s], non_blocking=True)
            d_dk.copy_(h_dk[s], non_blocking=True)
            d_dv.copy_(h_dv[s], non_blocking=True)
            for layer in range(L):
                rdkv.rdkv_decode_step(caches[layer], d_dq[layer], d_dk[layer], d_dv[layer], out=d_out[layer])
            h_out[s].copy_(d_out, non_blocking=True)

    step_compress()
    for c in caches:
        c.decode_workspace()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        decode_phase()
    step_compress()
    g.replay()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 3))
    times, t_dec = [], []
    for _ in range(steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step_compress()
        t1 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        times.append(t2 - t0)
        t_dec.append(t2 - t1)   # the decode phase, from its launch (the compress phase may still run on the GPU)
    h2d = sum(t.numel() * t.element_size() for trip in h_pre for t in trip) + \
        sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv))
    d2h = h_out.numel() * 4 + L * 96   # outputs, plus the plan totals each rdkv_plan_sizes reads back
    step_s = max_over_ranks([median(times)], ws, dev)[0]  # the slowest rank sets the whole job's step
    del h_pre, d_pre, caches, score_out, alloc_out, g
    return {"value": round(ws * dec_bytes / step_s / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "step_ms": round(step_s * 1e3, 2),
            "note": "whole step, median wall time: per layer the prefill inputs' H2D (copy stream, overlapping "
                    "the previous layer's compression), score, allocate, plan sizes (read back), pack; then per "
                    "decode step the H2D of q/k/v, every layer's fused append + attend and the D2H of the "
                    "outputs; value = decode algorithmic bytes / step time"}


# ---------------------------------------------------------------- CPU oracle (baseline and reference arm)
ORACLE_SAMPLE_TOKENS = {"tiny": 512, "llama3b": 2048, "llama8b": 2048, "qwen72b": 2048, "batched": 2048}


def _oracle_job(job):
    """One oracle call in a worker process (one thread): returns its seconds."""
    import oracle as O
    kind, a = job
    t0 = time.perf_counter()
    if kind == "score":
        O.score(a["q"], a["k"], a["v"], a["window"])
    elif kind == "allocate":
        O.allocate(a["g_tok"], a["w_chan"], a["k"], a["avg"], a["avg"])
    elif kind == "pack":
        O.pack(a["k"], a["v"], a["bits_tok"], a["bits_chan"], a["window"], cap_c=a["cap_c"])
    elif kind == "decode":
        O.decode(a["cache"], a["q"])
    return time.perf_counter() - t0


def _oracle_setup(name, n_tokens):
    """A bounded sample of a workload for the oracle: one sequence, one layer, N = n_tokens; its
    weights, allocation and pack by the oracle (untimed), and the jobs of each step with their
    units of work."""
    import oracle as O
    from mixed_bit_kv_gb300 import synth
    w = synth.WORKLOADS[name].scaled(n_tokens=n_tokens, batch=1)
    avg = w.budgets[0]
    q, k, v = (t.numpy() for t in synth.prefill(w, 0, 0))
    sc = O.score(q, k, v, w.window)
    al = O.allocate(sc["g_tok"], sc["w_chan"], k, avg, avg)
    cache = O.pack(k[None], v[None], al["bits_tok"][None], al["bits_chan"][None], w.window, cap_c=w.window + 1)
    qn, kn, vn = (t.numpy() for t in synth.decode_step(w, 0))
    O.append(cache, kn, vn)
    P = 2 if w.dtype == "f16" else 4
    plan = cache["plan"]
    pack_bytes = (2 * plan["kept_tokens"] * w.head_dim * P + 2 * w.h_kv * w.window * w.head_dim * (P + 2)
                  + plan["zone_a_bytes"] + plan["zone_b_rows"] * w.head_dim * 2 + plan["index_slots"] * 4)
    jobs = {
        "score": (("score", dict(q=q, k=k, v=v, window=w.window)), scorer_flops(w), "flop"),
        "allocate": (("allocate", dict(g_tok=sc["g_tok"], w_chan=sc["w_chan"], k=k, avg=avg)), 1, "call"),
        "pack": (("pack", dict(k=k[None], v=v[None], bits_tok=al["bits_tok"][None], bits_chan=al["bits_chan"][None],
                               window=w.window, cap_c=w.window + 1)), pack_bytes, "byte"),
        "decode": (("decode", dict(cache=cache, q=qn)),
                   O.decode_bytes(plan, w.head_dim, w.h_q, w.h_kv, cache["len_c"], 1), "byte"),
    }
    return w, jobs


def _spawn_pool(n):
    """A pool of n single-threaded worker processes, started with spawn (safe after CUDA use)."""
    import multiprocessing as mp
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        pool = mp.get_context("spawn").Pool(n)
        pool.map(math.sqrt, range(n))   # workers up before anything is timed
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
    return pool


def oracle_baseline(headline):
    """The oracle as it stands, timed on this host's cores: each step on one core (one worker, one
    thread) and on all cores (one single-threaded worker per core, each running the same call),
    on bounded samples of the workloads (one sequence, one layer, reduced N).  Steps: decode,
    allocate and pack on the 3B-shaped layer and the headline workload, the scorer on the tiny,
    3B- and 8B-shaped layers.  Returns the cpu_baseline object (value: headline decode GB/s on all
    cores)."""
    nproc = os.cpu_count() or 1
    t_all0 = time.perf_counter()
    plan = [("decode", "llama3b"), ("allocate", "llama3b"), ("pack", "llama3b"),
            ("score", "tiny"), ("score", "llama3b"), ("score", "llama8b")]
    if headline not in ("llama3b",):
        plan = [("decode", headline), ("allocate", headline), ("pack", headline)] + plan
    setups = {}
    for _, name in plan:
        if name not in setups:
            setups[name] = _oracle_setup(name, ORACLE_SAMPLE_TOKENS.get(name, 2048))
    steps = {}
    one = _spawn_pool(1)
    try:
        for kind, name in plan:
            job, units, unit = setups[name][1][kind]
            steps.setdefault(kind, {})[name] = {"one_core_s": one.map(_oracle_job, [job])[0]}
    finally:
        one.close()
        one.join()
    allp = _spawn_pool(nproc)
    try:
        for kind, name in plan:
            job, units, unit = setups[name][1][kind]
            t0 = time.perf_counter()
            allp.map(_oracle_job, [job] * nproc, chunksize=1)
            steps[kind][name]["all_cores_s"] = time.perf_counter() - t0
    finally:
        allp.close()
        allp.join()
    for kind, name in plan:
        w, jobs = setups[name]
        _, units, unit = jobs[kind]
        r = steps[kind][name]
        r["sample"] = f"one sequence, one layer, N={w.n_tokens} (workload N={ORACLE_FULL_N[name]})"
        if unit == "byte":
            r["one_core_gbs"] = units / r["one_core_s"] / 1e9
            r["all_cores_gbs"] = nproc * units / r["all_cores_s"] / 1e9
        elif unit == "flop":
            r["one_core_gflops"] = units / r["one_core_s"] / 1e9
            r["all_cores_gflops"] = nproc * units / r["all_cores_s"] / 1e9
        else:
            r["one_core_us_per_call"] = r["one_core_s"] * 1e6
            r["all_cores_calls_per_s"] = nproc / r["all_cores_s"]
    head = steps["decode"][headline]
    return {"value": head["all_cores_gbs"], "unit": UNIT, "cores": nproc, "kind": "oracle",
            "one_core_value": head["one_core_gbs"],
            "sample": (f"oracle decode (unpack + float64 attention) of one {headline}-shaped layer at "
                       f"N={setups[headline][0].n_tokens}; value on all {nproc} cores ({nproc} single-threaded "
                       f"workers, each one call), one_core_value on one; steps below: one core and all cores"),
            "steps": steps, "wall_s": round(time.perf_counter() - t_all0, 1)}


ORACLE_FULL_N = {"tiny": 512, "llama3b": 32768, "llama8b": 131072, "qwen72b": 262144, "batched": 32768}


def run_reference(args):
    """The reference arm: the CPU oracle's decode on a bounded sample of the workload (one
    sequence, one layer, reduced N), on all host cores (one single-threaded worker per core, each
    one decode call per step)."""
    name = args.workload
    nproc = os.cpu_count() or 1
    t_all = time.perf_counter()
    w, jobs = _oracle_setup(name, ORACLE_SAMPLE_TOKENS.get(name, 2048))
    job, units, _ = jobs["decode"]
    pool = _spawn_pool(nproc)
    vals, secs = [], []
    try:
        for _ in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            pool.map(_oracle_job, [job] * nproc, chunksize=1)
            dt = time.perf_counter() - t0
            secs.append(dt)
            vals.append(nproc * units / dt / 1e9)
    finally:
        pool.close()
        pool.join()
    value = median(vals[args.warmup:])
    desc = (f"oracle decode (unpack + float64 attention) of one {name}-shaped layer at N={w.n_tokens} "
            f"(workload N={ORACLE_FULL_N[name]}); {nproc} single-threaded workers, one call each per step")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(median(secs[args.warmup:]) * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)",
            "config": {"workload": name, "avg_bits": w.budgets[0], "oracle_tokens": w.n_tokens},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nproc, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t_all, 1)}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen72b")
    ap.add_argument("--layers", type=int, default=None, help="layers of the stack (default: per workload)")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--budget", type=float, default=None)
    ap.add_argument("--tokens", type=int, default=None,
                    help="prompt length N (default: the workload's; shorter for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-comparator", action="store_true", help="skip the fp16 full-cache SDPA context number")
    ap.add_argument("--no-recompress", action="store_true", help="skip the zone-C re-compression and paged zone-C measurements")
    ap.add_argument("--no-extras", action="store_true", help="skip the decode measurements of the other workloads")
    args = ap.parse_args()
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if ws > 1:
        torch.distributed.barrier()
    line = run_ours(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_baseline(args.workload)
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
