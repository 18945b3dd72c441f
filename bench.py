"""Throughput of fused causal GQA attention, forward + backward, on GB300.

One step = one forward (O, LSE) and one backward (dQ, dK, dV) of the whole
workload through the C ABI, inputs resident in HBM. The default workload is
long-context training: B=2, Hq=32, Hkv=8, S=16384, D=128, causal, seeded
synthetic bf16 inputs (Q, K, V ~ N(0,1), dO ~ N(0, 1e-2)).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line. Under torchrun (N > 1) every rank runs its own replica
of the workload (independent problems, no data-path collective: weak
scaling); the reported time is the max over ranks.

Throughput is algorithmic: forward 4*D flops per visible (query, key) pair
per query head, backward 10*D (five contractions, including the recompute of
Q K^T), i.e. fwd = 4*B*Hq*D*S(S+1)/2 and bwd = 2.5 * fwd. Masked halves of
diagonal tiles are not counted.

``--impl reference`` times the f64 CPU oracle (the only reference there is)
on a bounded sample of the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal GQA attention fwd+bwd TFLOP/s and % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops(B, Hq, S, D):
    pairs = S * (S + 1) / 2.0
    fwd = 4.0 * B * Hq * D * pairs
    return fwd, 2.5 * fwd


# ---- replicas over ranks (the path does not shard: every rank solves its own seeded problem)

def replica_seed(seed, rank):
    """Seed of rank `rank`'s replica of a workload: distinct inputs per rank, rank 0 = the workload's."""
    return seed + 1000 * rank


def max_over_ranks_of(x, world, device):
    """The largest of every rank's x (the job's step time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops_per_rank, world, ms_per_step):
    """Whole-job throughput: every rank's work over the slowest rank's step time."""
    return world * step_flops_per_rank / (ms_per_step / 1e3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {"bwd_main": ("bwd.cu", "ptx.cuh", "common.h"), "fwd": ("fwd.cu", "ptx.cuh", "common.h"),
                  "decode_split": ("decode.cu", "ptx.cuh", "common.h"),
                  "bwd_dq": ("bwd_dq.cu", "ptx.cuh", "common.h")}


def kernel_source_hash(kernel_name):
    """sha256 over the source files a kernel is built from (its .cu file and the shared headers)."""
    src = os.path.join(ROOT, "causal_gqa_attention_flash_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel_name]:
        h.update(open(os.path.join(src, f), "rb").read())
    return h.hexdigest()


def profiled_traffic(kernel_name, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_name}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m_bytes or not m_hash or kernel_source_hash(kernel_name) != m_hash.group(1):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(w, budget_s=12.0, prefix=4096):
    """Time the f64 oracle on causal prefixes of the workload: all G query heads of one KV group over
    positions [0, prefix) (a self-contained causal sub-problem), forward + backward, repeated over
    KV groups until budget_s of wall time has passed. Returns (TFLOP/s, description, cores)."""
    import numpy as np

    import oracle
    from gqa_inputs import make_inputs, to_f64

    S = min(prefix, w.S)
    q, k, v, dO = make_inputs(1, w.G, 1, S, w.D, seed=w.seed, do_std=w.do_std)
    qf, kf, vf, dOf = (to_f64(t) for t in (q, k, v, dO))
    fwd1, bwd1 = flops(1, w.G, S, w.D)
    done, t0, units = 0.0, time.perf_counter(), 0
    while True:
        oracle.forward(qf, kf, vf, causal=True, scale=w.scale)
        oracle.backward(qf, kf, vf, dOf, causal=True, scale=w.scale)
        done += fwd1 + bwd1
        units += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    desc = (f"{units} x (1 KV group = {w.G} query heads, causal prefix S={S}, D={w.D}) fwd+bwd in f64 numpy, "
            f"{el:.1f} s")
    return done / el / 1e12, desc, os.cpu_count()


def reference_arm(args, w, rank, world):
    if rank != 0:
        return
    val, desc, cores = cpu_oracle_sample(w, budget_s=max(5.0, min(30.0, 3.0 * args.steps)))
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, shapes of the workload)",
        "config": config_of(w),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


DECODE = dict(B=8, Hq=32, Hkv=8, Sq=1, Sk=16384, D=128, seed=5)


def decode_measurement(g, torch, peaks, peak_src, steps=20, warmup=3):
    """Split-KV decode (one new token per sequence against a 16k-token cache): HBM-bound, so the
    metric is the cache bytes read per second against the measured HBM peak."""
    from gqa_inputs import make_inputs
    c = DECODE
    _, k, v, _ = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sk"], c["D"], c["seed"], with_do=False)
    q = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["D"], c["seed"] + 1, with_do=False)[0]
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((c["B"], c["Hq"], c["Sq"]), device="cuda", dtype=torch.float32)
    ws = torch.empty(g.gqa_attn_decode_workspace_size(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"], 0),
                     device="cuda", dtype=torch.uint8)
    # a buffer larger than L2, written between timed calls so that every call reads the cache from HBM
    flush = torch.empty(256 << 20, device="cuda", dtype=torch.uint8)
    for _ in range(warmup):
        g.gqa_attn_decode_fwd(q, k, v, o=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    total = 0.0
    g.gqa_attn_trace_arm()
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gqa_attn_decode_fwd(q, k, v, o=o, lse=lse, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    tr = g.gqa_attn_trace_collect()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("decode failed")
    ms = total / steps
    cache_bytes = 2 * k.numel() * k.element_size()
    algo = cache_bytes + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
    n, t = tr["decode_split"]
    split_ms = t / max(n, 1)
    gbs = algo / (ms * 1e-3) / 1e9
    split_gbs = cache_bytes / (split_ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"workload": "decode: B=8 Hq=32 Hkv=8 Sq=1 Sk=16384 D=128 (one new token against a 16k cache)",
            "value": gbs, "unit": "GB/s", "us_per_call": ms * 1e3, "l2": "256 MB buffer written between calls",
            "kernels": {k_: {"launches": n_, "avg_ms": (t_ / n_ if n_ else None)} for k_, (n_, t_) in tr.items() if n_},
            "roofline": {"kernel": "decode_split", "bound": "hbm", "achieved": split_gbs, "peak": peak, "unit": "GB/s",
                         "frac": split_gbs / peak, "traffic": profiled_traffic("decode_split", "decode16k"),
                         "peak_source": f"{peak_src} HBM copy"}}


PREFILL = dict(B=2, Hq=32, Hkv=8, Sq=512, Sk=16384, D=128, seed=6)
PREFILL_B1 = dict(B=1, Hq=32, Hkv=8, Sq=512, Sk=16384, D=128, seed=7)


def prefill_measurement(g, torch, peaks, peak_src, c=PREFILL, steps=20, warmup=3):
    """Tensor-core forward of Sq new tokens per sequence over an Sk-token cache (bottom-right
    causal) through gqa_attn_fwd_splitkv, which splits the key ranges when the grid is small (then
    the forward and the merge kernel both run): FLOPs are 4 D per visible (query, key) pair,
    against the measured bf16 burst peak."""
    from gqa_inputs import make_inputs
    _, k, v, _ = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sk"], c["D"], c["seed"], with_do=False)
    q = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["D"], c["seed"] + 1, with_do=False)[0]
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((c["B"], c["Hq"], c["Sq"]), device="cuda", dtype=torch.float32)
    nws = g.gqa_attn_fwd_splitkv_workspace_size(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"])
    ws = torch.empty(max(nws, 256), device="cuda", dtype=torch.uint8)
    flush = torch.empty(256 << 20, device="cuda", dtype=torch.uint8)
    for _ in range(warmup):
        g.gqa_attn_fwd_splitkv(q, k, v, o=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    total = 0.0
    g.gqa_attn_trace_arm()
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gqa_attn_fwd_splitkv(q, k, v, o=o, lse=lse, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    tr = g.gqa_attn_trace_collect()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("prefill failed")
    ms = total / steps
    koff = c["Sk"] - c["Sq"]
    pairs = c["Sq"] * koff + c["Sq"] * (c["Sq"] + 1) // 2
    fl = 4.0 * c["D"] * pairs * c["B"] * c["Hq"]
    n, t = tr["fwd"]
    kern_ms = t / max(n, 1)
    nc, tc = tr["fwd_combine"]
    comb_ms = tc / max(nc, 1) if nc else 0.0
    achieved = fl / ((kern_ms + comb_ms) * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": (f"prefill: B={c['B']} Hq={c['Hq']} Hkv={c['Hkv']} Sq={c['Sq']} Sk={c['Sk']} D={c['D']} "
                         f"({c['Sq']} new tokens over a {c['Sk'] // 1024}k cache, causal)"),
            "value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "us_per_call": ms * 1e3,
            "split": {"workspace_bytes": nws, "fwd_us": kern_ms * 1e3, "combine_us": comb_ms * 1e3,
                      "combine_launches_per_call": nc / steps},
            "l2": "256 MB buffer written between calls",
            "roofline": {"kernel": "fwd + fwd_combine" if nc else "fwd", "bound": "tensor", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                         "peak_source": f"{peak_src} bf16 dense, burst (kernel timed alone)"}}


PACKED = dict(Hq=32, Hkv=8, D=128, n=16, lo=512, hi=3584, seed=8)


def packed_measurement(g, torch, peaks, peak_src, steps=20, warmup=3):
    """Forward + backward of a packed batch of 16 causal sequences of mixed length (uniform on
    [512, 3584] tokens, laid end to end): FLOPs are 4 D (forward) + 10 D (backward) per visible
    pair of each sequence, against the measured bf16 burst peak (each step timed alone)."""
    from gqa_inputs import draw_lengths, make_packed_inputs
    c = PACKED
    lens = draw_lengths(c["n"], c["lo"], c["hi"], c["seed"])
    q, k, v, dO, cu, _ = make_packed_inputs(c["Hq"], c["Hkv"], lens, lens, c["D"], c["seed"])
    q, k, v, dO, cu = q.cuda(), k.cuda(), v.cuda(), dO.cuda(), cu.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(g.gqa_attn_bwd_varlen_workspace_size(c["Hq"], c["Hkv"], q.shape[1], c["D"]),
                     device="cuda", dtype=torch.uint8)
    flush = torch.empty(256 << 20, device="cuda", dtype=torch.uint8)
    m = max(lens)

    def step():
        g.gqa_attn_fwd_varlen(q, k, v, cu, cu, m, o=o, lse=lse)
        g.gqa_attn_bwd_varlen(q, k, v, o, dO, lse, cu, m, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    total = 0.0
    g.gqa_attn_trace_arm()
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    tr = g.gqa_attn_trace_collect()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("packed forward/backward failed")
    ms = total / steps
    pairs = c["Hq"] * sum(n * (n + 1) // 2 for n in lens)
    fwd_fl, bwd_fl = 4.0 * c["D"] * pairs, 10.0 * c["D"] * pairs
    avg = {name: (t_ / n_ if n_ else None) for name, (n_, t_) in tr.items()}
    fwd_tf = fwd_fl / (avg["fwd"] * 1e-3) / 1e12
    bwd_tf = bwd_fl / (avg["bwd_main"] * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": (f"packed: Hq=32 Hkv=8 D=128, {c['n']} causal sequences of {min(lens)}..{max(lens)} tokens "
                         f"({sum(lens)} in all, lengths uniform on [{c['lo']}, {c['hi']}], seed {c['seed']}), "
                         "forward + backward"),
            "value": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "l2": "256 MB buffer written between steps",
            "kernels": {k_: {"launches": n_, "avg_ms": avg[k_]} for k_, (n_, _) in tr.items() if n_},
            "roofline": {"kernel": "bwd_main", "bound": "tensor", "achieved": bwd_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": bwd_tf / peak, "traffic": None,
                         "peak_source": f"{peak_src} bf16 dense, burst (each step timed alone)",
                         "fwd_kernel": {"achieved": fwd_tf, "frac": fwd_tf / peak}}}


def deterministic_measurement(g, torch, w, peaks, peak_src, steps, warmup, bufs, peak_kind="sustained"):
    """The same fwd+bwd step with the deterministic backward (query-major dQ kernel, KV-major dK/dV
    kernel), timed back to back like the main line. `value` counts the same algorithmic flops as
    the main line (4 D + 10 D per visible pair), so the two compare by time; the kernels' rooflines
    count the work they execute (dK/dV kernel 8 D per pair, dQ kernel 6 D per pair)."""
    q, k, v, dO, o, lse, dq, dk, dv, ws = bufs

    def step():
        g.gqa_attn_fwd(q, k, v, causal=True, scale=w.scale, o=o, lse=lse)
        g.gqa_attn_bwd(q, k, v, o, dO, lse, causal=True, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                       deterministic=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    g.gqa_attn_trace_arm()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    tr = g.gqa_attn_trace_collect()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("deterministic backward failed")
    ms = e0.elapsed_time(e1) / steps
    fwd_fl, bwd_fl = flops(w.B, w.Hq, w.S, w.D)
    pairs_fl = bwd_fl / 10.0  # D flops per visible pair, all heads
    avg = {name: (t_ / n_ if n_ else None) for name, (n_, t_) in tr.items()}
    peak = peaks["bf16_tflops" if peak_kind == "burst" else "bf16_tflops_sustained"]
    dq_tf = 6.0 * pairs_fl / (avg["bwd_dq"] * 1e-3) / 1e12
    dkdv_tf = 8.0 * pairs_fl / (avg["bwd_dkdv"] * 1e-3) / 1e12
    return {"workload": config_of(w)["workload"] + ", deterministic backward",
            "value": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "kernels": {k_: {"launches": n_, "avg_ms": avg[k_]} for k_, (n_, _) in tr.items() if n_},
            "roofline": {"kernel": "bwd_dq", "bound": "tensor", "achieved": dq_tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": dq_tf / peak, "traffic": profiled_traffic("bwd_dq", w.name),
                         "peak_source": f"{peak_src} bf16 dense, {peak_kind} (as the main line's clock record)",
                         "bwd_dkdv_kernel": {"achieved": dkdv_tf, "frac": dkdv_tf / peak}}}


def rope_measurement(g, torch, w, peaks, peak_src, steps, warmup, bufs, peak_kind="sustained"):
    """The same fwd+bwd step with the rotary embedding fused in (tables for base 10000): `value`
    counts the same algorithmic attention flops as the main line, so the two compare by time; the
    rotation passes (keys once in the forward, queries once in the backward) are listed."""
    from gqa_inputs import rope_tables
    q, k, v, dO, o, lse, dq, dk, dv, _ = bufs
    cos, sin = (t.cuda() for t in rope_tables(w.S, w.D))
    ws_f = torch.empty(g.gqa_attn_fwd_rope_workspace_size(w.B, w.Hkv, w.S, w.D), device="cuda", dtype=torch.uint8)
    ws_b = torch.empty(g.gqa_attn_bwd_rope_workspace_size(w.B, w.Hq, w.Hkv, w.S, w.D), device="cuda",
                       dtype=torch.uint8)

    def step():
        g.gqa_attn_fwd_rope(q, k, v, cos, sin, scale=w.scale, o=o, lse=lse, workspace=ws_f)
        g.gqa_attn_bwd_rope(q, k, v, o, dO, lse, cos, sin, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws_b)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    g.gqa_attn_trace_arm()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    tr = g.gqa_attn_trace_collect()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("rotary-embedding step failed")
    ms = e0.elapsed_time(e1) / steps
    fwd_fl, bwd_fl = flops(w.B, w.Hq, w.S, w.D)
    avg = {name: (t_ / n_ if n_ else None) for name, (n_, t_) in tr.items()}
    peak = peaks["bf16_tflops" if peak_kind == "burst" else "bf16_tflops_sustained"]
    main_tf = bwd_fl / (avg["bwd_main"] * 1e-3) / 1e12
    fwd_tf = fwd_fl / (avg["fwd"] * 1e-3) / 1e12
    return {"workload": config_of(w)["workload"] + ", rotary embedding (rotate-half, base 10000)",
            "value": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "kernels": {k_: {"launches": n_, "avg_ms": avg[k_]} for k_, (n_, _) in tr.items() if n_},
            "roofline": {"kernel": "bwd_main", "bound": "tensor", "achieved": main_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": main_tf / peak, "traffic": None,
                         "peak_source": f"{peak_src} bf16 dense, {peak_kind} (as the main line's clock record)",
                         "fwd_kernel": {"achieved": fwd_tf, "frac": fwd_tf / peak}}}


def peak_choice(peaks, clock_summary):
    """The bf16 denominator the clock record supports: the sustained (power-capped) figure when
    any sample of the timed region shows sw_power_cap, else the burst figure."""
    capped = "sw_power_cap" in (clock_summary or {}).get("reasons", [])
    return ("sustained", peaks["bf16_tflops_sustained"]) if capped else ("burst", peaks["bf16_tflops"])


CONFIG_NAMES = ("tiny", "lm101m", "block512", "qwen3_8b", "long16k")


def config_measurement(g, torch, w, peaks, reps=20, warmup=3):
    """fwd, bwd and fwd+bwd of one workload, each timed alone: TFLOP/s (algorithmic flops), the
    per-kernel averages from the library's own CUDA events (a second, traced pass), the gap between
    the measured time and the sum of kernel times (launch cost; negative where consecutive kernels
    overlap under programmatic dependent launch), and the host time one call takes to enqueue.
    Inputs smaller than L2 get a 256 MB buffer written between timed iterations (each iteration is
    timed on its own); larger ones run back to back."""
    from gqa_inputs import make_inputs
    q, k, v, dO = (t.cuda() for t in make_inputs(w.B, w.Hq, w.Hkv, w.S, w.D, w.seed, do_std=w.do_std))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.S), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(g.gqa_attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.S, w.D), device="cuda", dtype=torch.uint8)
    stream = torch.cuda.current_stream()
    small = w.B * w.Hq * w.S * w.D * 2 <= 129e6
    flush = torch.empty(256 << 20, device="cuda", dtype=torch.uint8) if small else None

    def fwd():
        g.gqa_attn_fwd(q, k, v, causal=True, scale=w.scale, o=o, lse=lse, stream=stream)

    def bwd():
        g.gqa_attn_bwd(q, k, v, o, dO, lse, causal=True, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                       stream=stream)

    def both():
        fwd()
        bwd()

    fwd_fl, bwd_fl = flops(w.B, w.Hq, w.S, w.D)
    out = {"shape": config_of(w)["workload"],
           "l2": "256 MB buffer written between timed iterations" if small else "inputs larger than L2"}

    def timed(fn, traced):
        """Mean ms per call over `reps` calls (and host seconds spent enqueueing them); with
        `traced`, the library's per-kernel events are armed as well (they sit between the
        kernels, so the call times come from a pass without them)."""
        torch.cuda.synchronize()
        host_s = 0.0
        if traced:
            g.gqa_attn_trace_arm()
        if small:
            total = 0.0
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                t0 = time.perf_counter()
                fn()
                host_s += time.perf_counter() - t0
                e1.record(stream)
                torch.cuda.synchronize()
                total += e0.elapsed_time(e1)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                t0 = time.perf_counter()
                fn()
                host_s += time.perf_counter() - t0
            e1.record(stream)
            torch.cuda.synchronize()
            total = e0.elapsed_time(e1)
        tr = g.gqa_attn_trace_collect() if traced else None
        return total / reps, host_s / reps, tr

    for label, fn, fl in (("fwd", fwd, fwd_fl), ("bwd", bwd, bwd_fl), ("fwd_bwd", both, fwd_fl + bwd_fl)):
        for _ in range(warmup):
            fn()
        ms, host_s, _ = timed(fn, False)
        _, _, tr = timed(fn, True)
        rc = g.gqa_attn_get_error()
        if rc != 0:
            raise RuntimeError(f"{w.name} {label} failed: {g.gqa_attn_strerror(rc)}")
        kern = {name: t_ / reps for name, (n_, t_) in tr.items() if n_}  # kernel ms per call
        out[label] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                      "kernel_ms": kern, "gap_ms": ms - sum(kern.values()),
                      "host_us_per_call": host_s * 1e6}
    # the two contraction kernels alone, by their own events
    kf = out["fwd_bwd"]["kernel_ms"]
    out["fwd_kernel_tflops"] = fwd_fl / (kf["fwd"] * 1e-3) / 1e12
    out["bwd_main_tflops"] = bwd_fl / (kf["bwd_main"] * 1e-3) / 1e12
    return out


def configs_measurement(g, torch, peaks, peak_src, local_rank, reps=20, warmup=3):
    """Every workload of the pages' shapes: fwd, bwd and fwd+bwd TFLOP/s and fractions of both the
    burst and the sustained bf16 peaks; `peak_used` names the one the clock record supports."""
    from gqa_inputs import WORKLOADS
    res = {}
    with ClockSampler(local_rank) as clk:
        for name in CONFIG_NAMES:
            res[name] = config_measurement(g, torch, WORKLOADS[name], peaks, reps, warmup)
    clocks = clk.summary()
    which, peak = peak_choice(peaks, clocks)
    for r in res.values():
        for label in ("fwd", "bwd", "fwd_bwd"):
            r[label]["frac"] = r[label]["tflops"] / peak
            r[label]["frac_burst"] = r[label]["tflops"] / peaks["bf16_tflops"]
            r[label]["frac_sustained"] = r[label]["tflops"] / peaks["bf16_tflops_sustained"]
        for kk in ("fwd_kernel", "bwd_main"):
            r[kk + "_frac"] = r[kk + "_tflops"] / peak
    return {"peak_used": which, "peak": peak, "peak_source": f"{peak_src} bf16 dense, {which}",
            "burst": peaks["bf16_tflops"], "sustained": peaks["bf16_tflops_sustained"],
            "clocks": clocks, "workloads": res}


def config_of(w):
    return {"workload": f"{w.name}: causal GQA B={w.B} Hq={w.Hq} Hkv={w.Hkv} S={w.S} D={w.D}",
            "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": True, "scale": w.scale,
            "seed": w.seed, "l2": "inputs larger than L2 (Q and dO are each > 129 MB)"
            if w.B * w.Hq * w.S * w.D * 2 > 129e6 else "inputs smaller than L2 (L2 not flushed)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="long16k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--shape", default=None,
                    help="B,Hq,Hkv,S,D: override the workload's shape (same seed and value distributions); "
                         "for profiling smaller cases")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the deterministic-backward, rotary-embedding, decode, prefill-over-cache and packed-batch measurements")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload fwd / bwd / fwd+bwd table")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from gqa_inputs import WORKLOADS, Workload
    w = WORKLOADS[args.workload]
    if args.shape:
        B, Hq, Hkv, S, D = (int(x) for x in args.shape.split(","))
        w = Workload(f"{w.name}-shape{B}x{Hq}x{Hkv}x{S}x{D}", B, Hq, Hkv, S, D, seed=w.seed, do_std=w.do_std)

    if args.impl == "reference":
        reference_arm(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist

    import causal_gqa_attention_flash_gb300 as g
    from gqa_inputs import make_inputs

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x):
        return max_over_ranks_of(x, world, "cuda")

    # Each rank: its own seeded replica of the workload (independent problems).
    q_h, k_h, v_h, dO_h = make_inputs(w.B, w.Hq, w.Hkv, w.S, w.D, replica_seed(w.seed, rank), do_std=w.do_std)
    q_h, k_h, v_h, dO_h = (t.pin_memory() for t in (q_h, k_h, v_h, dO_h))
    q, k, v, dO = (t.cuda() for t in (q_h, k_h, v_h, dO_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.S), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(g.gqa_attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.S, w.D), device="cuda", dtype=torch.uint8)
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
    stream = torch.cuda.current_stream()

    def step():
        g.gqa_attn_fwd(q, k, v, causal=True, scale=w.scale, o=o, lse=lse, stream=stream)
        g.gqa_attn_bwd(q, k, v, o, dO, lse, causal=True, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                       stream=stream)

    # End to end: every step uploads its inputs from pinned host memory and reads its results
    # back. Two device buffer sets and two copy streams (host-to-device, device-to-host): step
    # i+1's inputs go up and step i's results come down while step i computes.
    sets = [(q, k, v, dO, o, lse, dq, dk, dv)]
    sets.append(tuple(torch.empty_like(t) for t in sets[0]))
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def run_e2e(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_read = [torch.cuda.Event() for _ in range(2)]
        start = torch.cuda.Event()
        start.record(stream)

        def upload(i):
            bq, bk, bv, bdo = sets[i % 2][:4]
            h2d_s.wait_event(start)
            if i >= 2:  # set i % 2 last served step i - 2
                h2d_s.wait_event(comp_done[i % 2])
            with torch.cuda.stream(h2d_s):
                for dst, src in ((bq, q_h), (bk, k_h), (bv, v_h), (bdo, dO_h)):
                    dst.copy_(src, non_blocking=True)
            in_ready[i % 2].record(h2d_s)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            bq, bk, bv, bdo, bo, blse, bdq, bdk, bdv = sets[i % 2]
            stream.wait_event(in_ready[i % 2])
            if i >= 2:  # the results of step i - 2 have been read from this set
                stream.wait_event(out_read[i % 2])
            g.gqa_attn_fwd(bq, bk, bv, causal=True, scale=w.scale, o=bo, lse=blse, stream=stream)
            g.gqa_attn_bwd(bq, bk, bv, bo, bdo, blse, causal=True, scale=w.scale, dq=bdq, dk=bdk, dv=bdv,
                           workspace=ws, stream=stream)
            comp_done[i % 2].record(stream)
            d2h_s.wait_event(comp_done[i % 2])
            with torch.cuda.stream(d2h_s):
                for dst, src in zip(outs_h, (bo, blse, bdq, bdk, bdv)):
                    dst.copy_(src, non_blocking=True)
            out_read[i % 2].record(d2h_s)
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)

    fwd_fl, bwd_fl = flops(w.B, w.Hq, w.S, w.D)
    step_fl = fwd_fl + bwd_fl

    # ---- device-resident timing
    g.gqa_attn_trace_arm()  # creates the trace events during warm-up
    for _ in range(args.warmup):
        step()
    g.gqa_attn_trace_collect()
    rc = g.gqa_attn_get_error()
    if rc != 0:
        raise RuntimeError(f"warm-up failed: {g.gqa_attn_strerror(rc)}")
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        g.gqa_attn_trace_arm()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        trace = g.gqa_attn_trace_collect()
    barrier()
    rc = g.gqa_attn_get_error()
    if rc != 0:
        raise RuntimeError(f"timed steps failed: {g.gqa_attn_strerror(rc)}")
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)

    # ---- end to end: pinned host buffers in, results back to pinned host buffers, every step
    run_e2e(max(2, args.warmup))
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_e2e(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    if g.gqa_attn_get_error() != 0:
        raise RuntimeError("end-to-end steps failed")
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h, dO_h))
    d2h = sum(t.numel() * t.element_size() for t in outs_h)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    launches = sum(n for n, _ in trace.values())
    main_n, main_ms = trace["bwd_main"]
    fwd_n, fwd_ms = trace["fwd"]
    main_avg = main_ms / max(main_n, 1)
    fwd_avg = fwd_ms / max(fwd_n, 1)
    clocks = clk.summary()
    peak_kind, peak_tf = peak_choice(peaks, clocks)
    achieved = bwd_fl / (main_avg / 1e3) / 1e12
    fwd_achieved = fwd_fl / (fwd_avg / 1e3) / 1e12
    traffic = profiled_traffic("bwd_main", w.name)
    kernels = {name: {"launches": n, "avg_ms": (t / n if n else None), "share": (t / max(sum(
        tt for _, tt in trace.values()), 1e-12))} for name, (n, t) in trace.items()}

    line = {
        "metric": METRIC,
        "value": job_tflops(step_fl, world, ms),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, N(0,1e-2) dO)",
        "config": config_of(w),
        "fwd_tflops": fwd_achieved,
        "bwd_tflops": bwd_fl / ((ms - fwd_avg) / 1e3) / 1e12,
        "frac_of_peak": job_tflops(step_fl, world, ms) / (world * peak_tf),
        "kernels": kernels,
        "host_gap_ms": ms - sum(t for _, t in trace.values()) / args.steps,
        "roofline": {"kernel": "bwd_main", "bound": "tensor", "achieved": achieved, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 dense, {peak_kind} (the clock record of the timed "
                                    f"region {'shows' if peak_kind == 'sustained' else 'shows no'} sw_power_cap)",
                     "frac_burst": achieved / peaks["bf16_tflops"],
                     "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "fwd_kernel": {"achieved": fwd_achieved, "frac": fwd_achieved / peak_tf,
                                    "frac_burst": fwd_achieved / peaks["bf16_tflops"],
                                    "frac_sustained": fwd_achieved / peaks["bf16_tflops_sustained"],
                                    "traffic": profiled_traffic("fwd", w.name)}},
        "e2e": {"value": job_tflops(step_fl, world, ms_e2e), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "copies": "every step: Q, K, V, dO up from pinned host memory, O, LSE, dQ, dK, dV back; "
                          "double-buffered on two copy streams, overlapping the neighbouring steps' compute"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if world == 1 and not args.no_configs:
        line["configs"] = configs_measurement(g, torch, peaks, peak_src, local_rank)
    if world == 1 and not args.no_decode:
        line["deterministic"] = deterministic_measurement(g, torch, w, peaks, peak_src, args.steps, args.warmup,
                                                          (q, k, v, dO, o, lse, dq, dk, dv, ws), peak_kind)
        line["rope"] = rope_measurement(g, torch, w, peaks, peak_src, args.steps, args.warmup,
                                        (q, k, v, dO, o, lse, dq, dk, dv, ws), peak_kind)
        line["decode"] = decode_measurement(g, torch, peaks, peak_src)
        line["prefill"] = prefill_measurement(g, torch, peaks, peak_src, PREFILL)
        line["prefill_b1"] = prefill_measurement(g, torch, peaks, peak_src, PREFILL_B1)
        line["packed"] = packed_measurement(g, torch, peaks, peak_src)
    if world == 1 and not args.no_cpu_baseline:
        val, desc, cores = cpu_oracle_sample(w)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
