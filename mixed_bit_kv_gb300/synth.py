"""Seeded synthetic prefill and decode inputs for the RDKV workloads.

This module only draws random tensors with the structure of the workloads the
RDKV summary evaluates on (gist.science/ko/paper/2605.08317, section 4: long
contexts on LLaMA/Qwen-shaped layers) and of the attention picture on the
aistudio.id KV-cache page ("Solusi 2": attention sinks, heavy hitters, a
recent window).  It holds none of the compression arithmetic: no weights, no
allocation, no quantisation.  Both the CPU oracle and the CUDA path receive
the tensors made here.

Recipe (every constant below is a choice of this project; the pages print
none of them):

* base values z ~ N(0, 1) for Q, K and V;
* each KV head j gets a random unit direction u_j; queries are
  q = z + MU * u_j, so a key k = z + alpha * u_j with alpha = delta*sqrt(D)/MU
  receives a logit boost of about delta from every query of its group;
* sinks: the first ``n_sinks`` tokens get delta = ``sink_delta``;
* heavy hitters: a random ``hh_frac`` of the allocatable prefix gets
  delta = ``hh_delta``;
* Zipf salience: a random permutation ranks the prefix tokens r = 1..N_p and
  token rank r gets delta = ln(1 + (N/10) * r**-s), so the excess attention
  mass falls off as a Zipf law of exponent s;
* outlier key channels: ``n_outlier`` random channels per KV head are scaled
  by ``outlier_scale`` (applied after the alignment boost);
* decode steps draw fresh q (with the same u_j), k and v (with the same
  outlier channels) from a per-step seed.

Seeds: prefill of (workload id c, sequence s, layer l) uses
1_000_000*c + 1000*s + l; decode step i uses that value * 2**20 + i + 1, and the
bulk decode stream of a (sequence, layer) uses that value * 2**20.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

MU = 2.0


@dataclass(frozen=True)
class Workload:
    name: str
    workload_id: int
    batch: int
    n_tokens: int
    h_q: int
    h_kv: int
    head_dim: int
    window: int
    dtype: str                       # "f16" or "f32"
    budgets: tuple                   # average bits per unit (V and K alike)
    decode_steps: int
    n_outlier: int = 0
    outlier_scale: float = 1.0
    n_sinks: int = 0
    sink_delta: float = 0.0
    hh_frac: float = 0.0
    hh_delta: float = 0.0
    zipf_s: float = 0.0
    n_layers: int = 1
    description: str = field(default="", compare=False)

    @property
    def n_prefix(self) -> int:
        return self.n_tokens - self.window

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "f16" else torch.float32

    def scaled(self, **kw) -> "Workload":
        """Same generator, other sizes (parity cases at reduced length)."""
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, 1, 512, 4, 1, 64, 32, "f32", (3.0,), 16,
        n_outlier=2, outlier_scale=8.0, n_sinks=3, sink_delta=8.0,
        description="tiny single layer, batch 1: H_q=4, H_kv=1, D=64, N=512, fp32, "
                    "2 outlier K channels x8, 3 sink tokens; 3 bits; window 32; 16 decode steps"),
    "llama3b": Workload(
        "llama3b", 2, 1, 32768, 24, 8, 128, 128, "f16", (2.5,), 256,
        n_outlier=4, outlier_scale=10.0, hh_frac=0.01, hh_delta=4.0,
        description="Llama-3.2-3B-shaped layer: H_q=24, H_kv=8, D=128, fp16, batch 1, N=32768, "
                    "4 outlier K channels per head x10, 1% heavy hitters; 2.5 bits; window 128; 256 decode steps"),
    "llama8b": Workload(
        "llama8b", 3, 1, 131072, 32, 8, 128, 128, "f16", (0.4, 1.0, 2.0, 4.0), 256,
        zipf_s=1.1,
        description="Llama-3.1-8B-shaped layer: H_q=32, H_kv=8, D=128, fp16, batch 1, N=131072, "
                    "Zipf(1.1) token salience; budgets 0.4 (~2.5% retention), 1, 2, 4 bits; window 128"),
    "batched": Workload(
        "batched", 4, 8, 32768, 32, 8, 128, 128, "f16", (2.0,), 512,
        n_outlier=4, outlier_scale=10.0, hh_frac=0.01, hh_delta=4.0,
        description="batched decode: 8 sequences x N=32768, H_q=32, H_kv=8, D=128, fp16, "
                    "independent allocations; 2 bits; 512 decode steps with append"),
    "qwen72b": Workload(
        "qwen72b", 5, 1, 262144, 64, 8, 128, 128, "f16", (2.0,), 256,
        n_outlier=4, outlier_scale=10.0, hh_frac=0.01, hh_delta=4.0, n_layers=80,
        description="Qwen2.5-72B-shaped layer stack: H_q=64, H_kv=8, D=128, fp16, N=262144, "
                    "80 layers (kernels timed per layer); 2 bits; window 128"),
}


def prefill_seed(w: Workload, seq: int = 0, layer: int = 0) -> int:
    return 1_000_000 * w.workload_id + 1000 * seq + layer


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _directions(g, w: Workload, device):
    u = torch.randn(w.h_kv, w.head_dim, generator=g, device=device, dtype=torch.float32)
    return u / u.norm(dim=-1, keepdim=True)


def _outlier_channels(g, w: Workload, device):
    """[h_kv, n_outlier] channel indices (drawn even when n_outlier == 0 to keep streams aligned)."""
    rows = [torch.randperm(w.head_dim, generator=g, device=device)[: w.n_outlier] for _ in range(w.h_kv)]
    return torch.stack(rows) if w.n_outlier > 0 else torch.zeros(w.h_kv, 0, dtype=torch.long, device=device)


def prefill(w: Workload, seq: int = 0, layer: int = 0, device="cpu"):
    """Q [N, H_q, D], K [N, H_kv, D], V [N, H_kv, D] of one sequence, in the workload's dtype."""
    g = _gen(prefill_seed(w, seq, layer), device)
    N, D, Hq, Hkv = w.n_tokens, w.head_dim, w.h_q, w.h_kv
    Np = w.n_prefix
    u = _directions(g, w, device)
    outl = _outlier_channels(g, w, device)
    kv_of_q = torch.arange(Hq, device=device) // w.group

    q = torch.randn(N, Hq, D, generator=g, device=device, dtype=torch.float32)
    q += MU * u[kv_of_q][None]
    k = torch.randn(N, Hkv, D, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(N, Hkv, D, generator=g, device=device, dtype=torch.float32)

    delta = torch.zeros(Hkv, N, device=device, dtype=torch.float32)
    if w.n_sinks:
        delta[:, : w.n_sinks] = w.sink_delta
    if w.hh_frac > 0 and Np > 0:
        n_hh = max(1, int(round(w.hh_frac * Np)))
        for j in range(Hkv):
            idx = torch.randperm(Np, generator=g, device=device)[:n_hh]
            delta[j, idx] = w.hh_delta
    if w.zipf_s > 0 and Np > 0:
        for j in range(Hkv):
            rank = torch.randperm(Np, generator=g, device=device).to(torch.float32) + 1.0
            delta[j, :Np] = torch.log1p((N / 10.0) * rank.pow(-w.zipf_s))
    alpha = delta * (math.sqrt(D) / MU)                      # [Hkv, N]
    k += alpha.t()[..., None] * u[None]
    for j in range(Hkv):
        if outl.shape[1]:
            k[:, j, outl[j]] *= w.outlier_scale
    dt = w.torch_dtype
    return q.to(dt), k.to(dt), v.to(dt)


def prefill_batch(w: Workload, layer: int = 0, device="cpu"):
    """Stacked [B, N, H, D] tensors, each sequence from its own seed."""
    qs, ks, vs = zip(*(prefill(w, s, layer, device) for s in range(w.batch)))
    return torch.stack(qs), torch.stack(ks), torch.stack(vs)


def decode_step(w: Workload, step: int, layer: int = 0, device="cpu"):
    """q_new [B, H_q, D], k_new [B, H_kv, D], v_new [B, H_kv, D] for decode step ``step``."""
    qs, ks, vs = [], [], []
    for s in range(w.batch):
        base = prefill_seed(w, s, layer)
        g0 = _gen(base, device)
        u = _directions(g0, w, device)
        outl = _outlier_channels(g0, w, device)
        g = _gen((base << 20) + step + 1, device)
        kv_of_q = torch.arange(w.h_q, device=device) // w.group
        q = torch.randn(w.h_q, w.head_dim, generator=g, device=device) + MU * u[kv_of_q]
        k = torch.randn(w.h_kv, w.head_dim, generator=g, device=device)
        v = torch.randn(w.h_kv, w.head_dim, generator=g, device=device)
        for j in range(w.h_kv):
            if outl.shape[1]:
                k[j, outl[j]] *= w.outlier_scale
        qs.append(q); ks.append(k); vs.append(v)
    dt = w.torch_dtype
    return torch.stack(qs).to(dt), torch.stack(ks).to(dt), torch.stack(vs).to(dt)


def decode_stream(w: Workload, steps: int, layers: int, first_seq: int = 0, device="cpu"):
    """Decode inputs of `steps` steps for `layers` layers of sequences first_seq.. (batch w.batch):
    q [steps, layers, B, H_q, D], k and v [steps, layers, B, H_kv, D], drawn per (sequence, layer)
    with that prefill's query direction and outlier channels."""
    B = w.batch
    qs = torch.empty(steps, layers, B, w.h_q, w.head_dim, device=device)
    ks = torch.empty(steps, layers, B, w.h_kv, w.head_dim, device=device)
    vs = torch.empty(steps, layers, B, w.h_kv, w.head_dim, device=device)
    kv_of_q = torch.arange(w.h_q, device=device) // w.group
    for layer in range(layers):
        for b in range(B):
            base = prefill_seed(w, first_seq + b, layer)
            g0 = _gen(base, device)
            u = _directions(g0, w, device)
            outl = _outlier_channels(g0, w, device)
            g = _gen(base << 20, device)
            qs[:, layer, b] = torch.randn(steps, w.h_q, w.head_dim, generator=g, device=device) + MU * u[kv_of_q]
            k = torch.randn(steps, w.h_kv, w.head_dim, generator=g, device=device)
            for j in range(w.h_kv):
                if outl.shape[1]:
                    k[:, j, outl[j]] *= w.outlier_scale
            ks[:, layer, b] = k
            vs[:, layer, b] = torch.randn(steps, w.h_kv, w.head_dim, generator=g, device=device)
    dt = w.torch_dtype
    return qs.to(dt), ks.to(dt), vs.to(dt)
