#!/usr/bin/env python
"""Benchmark of the RDKV hot path (score -> allocate -> TriZone pack -> append + decode) on GB300.

One step = compress every layer of a stack of independently generated layers
of the chosen workload (default: the Llama-3.2-3B-shaped layer, N = 32768,
28 layers like the model), then run the workload's decode steps over all
layers (append the new token, attend).  Inputs are resident in HBM when the
timed region starts; the decode phase is replayed from a captured CUDA graph.
The working set (prefill inputs ~9 GB, packed caches ~0.7 GB) is larger than
L2, and each decode call reads a cache last touched 27 calls earlier.

Rank 0 prints one JSON line.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import resource
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TriZone decode attn HBM GB/s (scoring TFLOP/s, decode us/step alongside)"
UNIT = "GB/s"


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


def captured_traffic(kernel):
    """DRAM bytes per launch from the committed ncu record, or None when the kernel's
    source has changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p))[kernel]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except (OSError, KeyError, ValueError):
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
    """Bytes one decode call must move: zone-A payload and metadata of real tokens
    and channels, zone-B rows of real tokens, len_c zone-C rows per head, q in and
    out.  Padding excluded."""
    total = 0.0
    for hp in heads:
        n16k, n8k, n4k, n2k, _ = (int(x) for x in hp["n_k"])
        ntok = int(np.sum(hp["n_v"]))
        kq = n8k + n4k + n2k
        total += ntok * (2 * n16k + (8 * n8k + 4 * n4k + 2 * n2k) / 8) + 4 * kq * ntok / 32
        for n, b in zip(hp["n_v"], (2, 4, 8, 16)):
            total += int(n) * (D * b / 8 + (4 * D / 32 if b < 16 else 0))
        total += len_c * 4 * D
    return total + batch * h_q * D * (2 + 4)


def scorer_flops(w):
    """2 passes x 2*D flops per causal (query head, row, key) pair."""
    return 2 * 2 * w.head_dim * w.h_q * w.batch * w.n_tokens * (w.n_tokens + 1) / 2


# ---------------------------------------------------------------- our arm
def run_ours(args, ws, rank, local):
    from mixed_bit_kv_gb300 import rdkv, synth

    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    L = args.layers
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
    stream = torch.cuda.current_stream()

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

    # timed region
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = []
    score_ev = []
    launches0 = lib.rdkv_launch_count()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(torch.cuda.current_device())
    with ClockSampler(gpu_id) as clk:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            c = torch.cuda.Event(enable_timing=True)
            a.record()
            compress(score_ev)
            b.record()
            g.replay()
            c.record()
            ev.append((a, b, c))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    compress_launches = lib.rdkv_launch_count() - launches0
    gpu_launches = int(compress_launches + args.steps * decode_launches)
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    dec_ms = [b.elapsed_time(c) for a, b, c in ev]
    score_ms = sum(e[0].elapsed_time(e[1]) for e in score_ev) / args.steps
    alloc_ms = sum(e[1].elapsed_time(e[2]) for e in score_ev) / args.steps  # incl. the sizes read-back
    pack_ms = sum(e[2].elapsed_time(e[3]) for e in score_ev) / args.steps
    tot_ms, tot_dec, tot_score = sum(step_ms), sum(dec_ms), score_ms * args.steps
    tot_ms, tot_dec, tot_score = max_over_ranks([tot_ms, tot_dec, tot_score], ws, dev)
    score_ms = tot_score / args.steps

    ms_per_step = tot_ms / args.steps
    dec_ms_step = tot_dec / args.steps
    value = whole_job_rate(ws, dec_bytes, dec_ms_step * 1e-3) / 1e9
    flops = scorer_flops(w) * L
    score_tflops = whole_job_rate(ws, flops, score_ms * 1e-3) / 1e12
    peaks = measured_peaks()
    clocks = clk.summary()

    # roofline of the dominant kernel by time share in the step
    dec_frac_time, score_frac_time = dec_ms_step / ms_per_step, score_ms / ms_per_step
    decode_roof = {"bound": "hbm", "achieved": round(value / ws, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": round(value / ws / peaks["hbm_gbs"], 4), "traffic": captured_traffic("decode_kernel"),
                   "algorithmic_bytes_per_launch": int(dec_bytes / (S * L)),
                   "peak_source": peaks["source"], "time_share": round(dec_frac_time, 3)}
    # fp16 scorer on the tensor cores: measured dense bf16 peak (fp16 has the same nominal dense rate);
    # the sustained figure, since the scorer runs back to back over every layer inside the step.
    # fp32 inputs run on CUDA cores: roofline against the FP32 FMA peak instead.
    if w.dtype == "f16":
        t1, t2 = captured_traffic("score_kernel_pass1"), captured_traffic("score_kernel_pass2")
        score_roof = {"bound": "tensor", "achieved": round(score_tflops / ws, 2),
                      "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                      "frac": round(score_tflops / ws / peaks["bf16_tflops_sustained"], 4),
                      "traffic": (t1 + t2) if (t1 and t2) else None, "flops_per_launch_pair": scorer_flops(w),
                      "peak_source": f"{peaks['source']} bf16 dense sustained (fp16 nominal rate equal)",
                      "time_share": round(score_frac_time, 3)}
    else:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        score_roof = {"bound": "alu", "achieved": round(score_tflops / ws, 2), "peak": round(alu_peak, 1),
                      "unit": "TFLOP/s", "frac": round(score_tflops / ws / alu_peak, 4), "traffic": None,
                      "peak_source": "SMs x 128 FP32 lanes x 2 flops x max SM clock",
                      "time_share": round(score_frac_time, 3)}
    dominant = score_roof if score_frac_time >= dec_frac_time else decode_roof

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
                   "l2": "inputs larger than L2: 9 GB prefill, ~0.7 GB of packed caches rotated across layers"},
        "decode_us_per_layer_step": round(dec_ms_step * 1e3 / (S * L), 3),
        "decode_ms_per_model_step": round(dec_ms_step / S, 4),
        "decode_bytes_per_step": int(dec_bytes),
        "scorer_tflops": round(score_tflops, 2), "scorer_ms_per_layer": round(score_ms / L, 3),
        "compress_ms_per_layer": round((ms_per_step - dec_ms_step) / L, 3),
        "compress_breakdown_ms_per_layer": {
            "score (weights: tensor-core passes, channel norms, V spreads)": round(score_ms / L, 3),
            "allocate (water-filling V and K, channel spreads, plan; sizes read back)": round(alloc_ms / L, 3),
            "pack (index map, tiles, zone B, window)": round(pack_ms / L, 3)},
        "pack_gbs": round(sum(pack_bytes_per_layer(w, c.c.sizes) for c in caches) / (pack_ms * 1e-3) / 1e9, 1),
        "roofline": dominant, "rooflines": {"decode": decode_roof, "scorer": score_roof},
        "gpu_launches": gpu_launches, "clocks": clocks, "wall_s": round(wall, 3),
    }
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
    return line


def run_fp16_comparator(w, L, pre, dq, dev, steps=16):
    """Context number: decode over the full fp16 cache of the same layers (all N prompt tokens, no
    compression) with torch's scaled_dot_product_attention (a library call), per layer step, replayed
    from a CUDA graph like the TriZone decode.  The caches of all layers are rotated (inputs larger
    than L2)."""
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
    return {"ms_per_layer": round(a.elapsed_time(b) / reps, 3),
            "zone_a_bytes_bound": int(comp.bounds.zone_a_bytes), "zone_a_bytes": int(exact.sizes.zone_a_bytes),
            "note": "score + allocate + pack from one CUDA graph, zones sized by rdkv_zone_bounds"}


def run_e2e(args, w, shape, L, S, avg, cap_c, pre, dq, dk, dv, dec_bytes, ws, dev):
    """Same metric through the public API with pinned host inputs: every step copies the
    prefill inputs and every decode step's inputs host->device and reads each output back."""
    from mixed_bit_kv_gb300 import rdkv

    h_pre = [tuple(t.cpu().pin_memory() for t in trip) for trip in pre]
    h_dq, h_dk, h_dv = (t.cpu().pin_memory() for t in (dq, dk, dv))
    h_out = torch.empty((S, L, w.batch, w.h_q, w.head_dim), dtype=torch.float32).pin_memory()
    d_pre = [tuple(torch.empty_like(t) for t in trip) for trip in pre]
    d_dq, d_dk, d_dv = (torch.empty_like(t[0]) for t in (dq, dk, dv))   # one decode step, all layers
    d_out = torch.empty((L, w.batch, w.h_q, w.head_dim), dtype=torch.float32, device=dev)
    score_out, alloc_out, caches = [None] * L, [None] * L, [None] * L

    def step_compress():
        for layer in range(L):
            for dst, src in zip(d_pre[layer], h_pre[layer]):
                dst.copy_(src, non_blocking=True)
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
    steps = max(1, min(args.steps, 2))
    t_dec = 0.0
    for _ in range(steps):
        step_compress()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        t_dec += time.perf_counter() - t0
    h2d = sum(t.numel() * t.element_size() for trip in h_pre for t in trip) + \
        sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv))
    d2h = h_out.numel() * 4 + L * 96
    return {"value": round(ws * dec_bytes / (t_dec / steps) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "decode phase wall time incl. per-decode-step H2D of q/k/v and D2H of outputs; "
                    "the prefill H2D copies run in the compress phase of the same step"}


# ---------------------------------------------------------------- CPU oracle (baseline and reference arm)
def oracle_sample(w, avg, n_tokens, layers_sample=1, decode_calls=2):
    """Times the CPU oracle's decode (unpack + float64 attention) on a reduced-length
    sample of the workload; returns (GB/s of algorithmic decode bytes, cores used, description)."""
    import oracle as O
    from mixed_bit_kv_gb300 import synth
    ws_ = w.scaled(n_tokens=n_tokens, batch=1)
    q, k, v = (t.numpy() for t in synth.prefill(ws_, 0, 0))
    sc = O.score(q, k, v, ws_.window)
    al = O.allocate(sc["g_tok"], sc["w_chan"], k, avg, avg)
    cache = O.pack(k[None], v[None], al["bits_tok"][None], al["bits_chan"][None], ws_.window,
                   cap_c=ws_.window + decode_calls)
    qn, kn, vn = (t.numpy() for t in synth.decode_step(ws_, 0))
    O.append(cache, kn, vn)
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    nbytes = 0.0
    for _ in range(decode_calls):
        O.decode(cache, qn)
        nbytes += O.decode_bytes(cache["plan"], ws_.head_dim, ws_.h_q, ws_.h_kv, cache["len_c"], 1)
    dt = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    cores = max(1, int(round(cpu / dt)))
    desc = (f"oracle decode (unpack + float64 attention) of one {w.name}-shaped layer at N={n_tokens} "
            f"(full workload N={w.n_tokens}), {decode_calls} calls, {dt:.1f} s")
    return nbytes / dt / 1e9, cores, desc


def run_reference(args):
    from mixed_bit_kv_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    avg = w.budgets[0] if args.budget is None else args.budget
    n = min(w.n_tokens, args.oracle_tokens)
    vals, t_all = [], time.perf_counter()
    for _ in range(args.warmup + args.steps):
        gbs, cores, desc = oracle_sample(w, avg, n, decode_calls=1)
        vals.append(gbs)
    value = float(np.mean(vals[args.warmup:]))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round((time.perf_counter() - t_all) * 1e3 / (args.warmup + args.steps), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)", "config": {"workload": w.name, "avg_bits": avg,
                                                               "oracle_tokens": n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3b")
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--budget", type=float, default=None)
    ap.add_argument("--oracle-tokens", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-comparator", action="store_true", help="skip the fp16 full-cache SDPA context number")
    ap.add_argument("--no-recompress", action="store_true", help="skip the zone-C re-compression and paged zone-C measurements")
    args = ap.parse_args()
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

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
            from mixed_bit_kv_gb300 import synth
            w = synth.WORKLOADS[args.workload]
            avg = w.budgets[0] if args.budget is None else args.budget
            gbs, cores, desc = oracle_sample(w, avg, min(w.n_tokens, args.oracle_tokens))
            line["cpu_baseline"] = {"value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
