#!/usr/bin/env python3
"""Benchmark of the fused attention forward hot path on one GB300 (or N, as
independent weak-scaled replicas under torchrun).

One step = one pass of the whole hot path over one batch of synthetic input:
  1. prefill: dense diffusion-transformer self-attention, B=2, S=4096,
     24 heads, D=128, non-causal (attn_fwd_dense, tcgen05 kernel);
  2. paged decode: 64 sequences, contexts U[1024, 32768], 32 query / 8 KV
     heads, D=128, cache (2, nb, 128, 8, 128) (attn_fwd_paged: split-K kernel
     + LSE-merge combine).
The headline `value` is the prefill's TFLOP/s (4*B*H*S^2*D algorithmic
flops over the kernel's CUDA-event time); the decode's HBM GB/s sits in
`paged_decode`.  Between steps a 512 MiB buffer is rewritten so that L2
(129 MB) holds nothing of the previous step.

`--impl reference` times the float64 CPU oracle on a bounded sample of the
same workload on this machine's host cores (there is no other reference
implementation of this path).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--only all|prefill|decode|kv_write|paged_prefill|masked|vsa] [--prefill WORKLOAD]
                       [--paged-prefill chunked_prefill|spec_decode] [--no-cpu]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attn fwd TFLOP/s & % bf16 TC peak; paged-decode HBM GB/s & % of HBM peak"
# Prefill workloads the step can run (--prefill); the default is the headline one.
PREFILL_WORKLOADS = {
    "dit_self": workloads.dit_self,
    "cross_attn": workloads.cross_attn,
    "varlen_causal_gqa": workloads.varlen_causal_gqa,
    "self_d64": lambda: workloads.head_sweep(64),
    "self_d96": lambda: workloads.head_sweep(96),
    "self_d192": lambda: workloads.head_sweep(192),
    "self_d256": lambda: workloads.head_sweep(256),
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_for(key: str, source_file: str):
    """DRAM bytes per call from a committed ncu summary (key "kernel@workload"),
    only while the kernel source still matches the one the counters were
    taken on."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(key)
    if not d:
        return None
    with open(os.path.join(ROOT, "attention_forward_09_gb300", "csrc", source_file), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return d["bytes_per_launch"] if d.get("source_sha") == sha else None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.text = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.text = self.proc.communicate(timeout=5)[0]
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "text", "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over the ranks (timing only; no data moves)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle

def oracle_prefill_sample(w: workloads.Dense, budget_s: float, inputs=None, rows_per_unit: int = 1024):
    """Time the float64 oracle on the dense workload, unit by unit (one
    (batch, head) and `rows_per_unit` query rows against all keys), until
    budget_s has passed; returns (TFLOP/s, description, seconds)."""
    import oracle

    q, k, v = inputs if inputs is not None else w.make()
    g = w.Hq // w.Hkv
    per_bh = -(-w.Sq // rows_per_unit)
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    while True:
        bh, chunk = divmod(done % (w.B * w.Hq * per_bh), per_bh)
        b, h = divmod(bh, w.Hq)
        rows = list(range(chunk * rows_per_unit, min(w.Sq, (chunk + 1) * rows_per_unit)))
        kv = h // g
        oracle.attention_single(q[b, :, h:h + 1], k[b, :, kv:kv + 1], v[b, :, kv:kv + 1], w.scale, w.causal,
                                rows=rows)
        flops += 4.0 * w.D * len(rows) * w.Sk
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= w.B * w.Hq * per_bh:  # never past the whole workload
            break
    desc = (f"{done} units of {rows_per_unit} query rows x all {w.Sk} keys, one (batch, head) each, "
            f"of {w.name} ({w.B * w.Hq * per_bh} units in the full workload)")
    return flops / el / 1e12, desc, el


def oracle_paged_sample(w: workloads.Paged, q, cache, bt, sl, budget_s: float):
    import oracle

    done, nbytes = 0, 0
    t0 = time.perf_counter()
    order = np.argsort(w.seq_lens)
    while True:
        s = int(order[done % len(order)])
        oracle.attention_paged(q[s:s + 1], cache, bt[s:s + 1], sl[s:s + 1], w.scale)
        nbytes += 2 * w.seq_lens[s] * w.Hkv * w.D * 2
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= len(order):
            break
    return nbytes / el / 1e9, f"{done} of {len(order)} sequences of {w.name} (shortest first)", el


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.dit_self()
    inputs = w.make()
    steps = []
    per_step = min(2.0, 120.0 / max(1, args.steps + args.warmup))  # whole run ~2 minutes at most
    for i in range(args.warmup + args.steps):
        tf, desc, el = oracle_prefill_sample(w, per_step, inputs)
        if i >= args.warmup:
            steps.append((tf, el))
    value = statistics.median(t for t, _ in steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(e for _, e in steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "seq_len": w.Sq, "heads": w.Hq, "head_dim": w.D},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": desc + f"; {per_step:.0f} s of oracle work per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_for(kernel_prefix: str, workload: str):
    """The committed ncu summary of a kernel on a workload, if there is one."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    for f in sorted(os.listdir(d)):
        if f.startswith(kernel_prefix) and f.endswith(f"__{workload}.md"):
            return f"profiles/{f}"
    return None


def time_calls(fn, steps, warmup, flush, stream):
    """Mean CUDA-event time (ms) of fn() over `steps` calls after `warmup`,
    L2 flushed before every call (outside the events)."""
    for _ in range(warmup):
        flush.fill_(1.0)
        fn()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def measure_configs(gb, dev, stream, status, flush, steps, warmup, pk, peak_kind):
    """Every workload of the headline metric, each timed on its own (inputs
    resident, L2 flushed between calls): prefill TFLOP/s against the measured
    bf16 burst peak, decode GB/s against the measured HBM copy bandwidth."""
    peak_tf, peak_bw = float(pk["bf16_tflops"]), float(pk["hbm_gbs"])
    res = {}

    def prefill_entry(w, fn, launches, kernel):
        ms = time_calls(fn, steps, warmup, flush, stream)
        tf = w.flops() / (ms * 1e-3) / 1e12
        return {"workload": w.name, "ms": ms, "value": tf, "unit": "TFLOP/s", "bound": "tensor", "peak": peak_tf,
                "frac": tf / peak_tf, "peak_kind": f"{peak_kind} bf16 burst", "flops_per_call": w.flops(),
                "launches_per_call": launches, "kernel": kernel,
                "profile": profile_for(kernel.split("<")[0], w.name)}

    def kernel_name(d):
        return f"fmha2_fwd_sm103a<Prefill2Cfg<{d}>>" if d <= 128 else f"fmha_fwd_sm103a<PrefillCfg<{d}>>"

    # 1: tiny packed documents (parity is checked in the tests; timed here for completeness)
    w = workloads.tiny_varlen()
    q, k, v, cq, ck = (x.to(dev) for x in w.make())
    o = torch.empty(w.Tq, w.Hq, w.D, dtype=torch.float32, device=dev)
    l = torch.empty(w.Hq, w.Tq, dtype=torch.float32, device=dev)
    e = prefill_entry(w, lambda: gb.attn_fwd_varlen(q, k, v, cq, ck, max(w.lens_q), max(w.lens_k), w.scale, w.causal,
                                                    out=o, lse=l, dev_status=status, stream=stream),
                      gb.attn_fwd_varlen_plan(w.lens_q, w.D, w.causal, w.Hq, w.Hkv, w.lens_k), kernel_name(w.D))
    e["note"] = "parity-only workload (a few microseconds of work); its fraction says nothing about the kernel"
    res["1_tiny_varlen"] = e

    # 2, 5a, 5b: dense
    for key, w in (("2_dit_self", workloads.dit_self()), ("5a_cross", workloads.cross_attn()),
                   ("5b_d64", workloads.head_sweep(64)), ("5b_d96", workloads.head_sweep(96)),
                   ("5b_d192", workloads.head_sweep(192)), ("5b_d256", workloads.head_sweep(256))):
        q, k, v = (x.to(dev) for x in w.make())
        o = torch.empty(w.B, w.Sq, w.Hq, w.D, dtype=torch.float32, device=dev)
        l = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
        launches = gb.attn_fwd_dense_plan(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, w.causal)[0]
        res[key] = prefill_entry(w, lambda: gb.attn_fwd_dense(q, k, v, w.scale, w.causal, out=o, lse=l,
                                                              dev_status=status, stream=stream),
                                 launches, kernel_name(w.D))
        del q, k, v, o, l

    # 3: packed causal prefill with GQA
    w = workloads.varlen_causal_gqa()
    q, k, v, cq, ck = (x.to(dev) for x in w.make())
    o = torch.empty(w.Tq, w.Hq, w.D, dtype=torch.float32, device=dev)
    l = torch.empty(w.Hq, w.Tq, dtype=torch.float32, device=dev)
    res["3_varlen_causal_gqa"] = prefill_entry(
        w, lambda: gb.attn_fwd_varlen(q, k, v, cq, ck, max(w.lens_q), max(w.lens_k), w.scale, w.causal, out=o,
                                      lse=l, dev_status=status, stream=stream),
        gb.attn_fwd_varlen_plan(w.lens_q, w.D, w.causal, w.Hq, w.Hkv, w.lens_k), kernel_name(w.D))
    res["3_varlen_causal_gqa"]["doc_lengths"] = list(w.lens_q)
    del q, k, v, o, l

    # 4: paged decode
    w = workloads.paged_decode()
    pq, cache, bt, sl = (x.to(dev) for x in w.make(chunk_rows=256))
    mx = max(w.seq_lens)
    ws = torch.empty(gb.attn_fwd_paged_workspace_size(len(w.seq_lens), w.Hq, w.Hkv, w.D, mx), dtype=torch.uint8,
                     device=dev)
    o = torch.empty(len(w.seq_lens), w.Hq, w.D, dtype=torch.float32, device=dev)
    l = torch.empty(len(w.seq_lens), w.Hq, dtype=torch.float32, device=dev)
    ms = time_calls(lambda: gb.attn_fwd_paged(pq, cache, bt, sl, mx, w.scale, out=o, lse=l, workspace=ws,
                                              dev_status=status, stream=stream), steps, warmup, flush, stream)
    nbytes = w.algorithmic_bytes(out_bytes_per_elem=4, with_lse=True)
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["4_paged_decode"] = {"workload": w.name, "ms": ms, "value": gbs, "unit": "GB/s", "bound": "hbm",
                             "peak": peak_bw, "frac": gbs / peak_bw, "peak_kind": f"{peak_kind} HBM copy",
                             "bytes_per_call": nbytes, "launches_per_call": 3,
                             "kernel": "paged_schedule + paged_decode_sm103a + paged_combine",
                             "profile": profile_for("paged_decode_sm103a", w.name + "_first16")}
    del pq, cache, bt, sl, ws, o, l
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} while timing the workloads")
    return res


def sustained_prefill(gb, dev, stream, status, seconds, pk, peak_kind, clock_gpu):
    """The headline prefill back to back for `seconds` (no flush: a serving
    loop's steady state), against the measured sustained bf16 peak, with its
    own clock record."""
    w = workloads.dit_self()
    q, k, v = (x.to(dev) for x in w.make())
    o = torch.empty(w.B, w.Sq, w.Hq, w.D, dtype=torch.float32, device=dev)
    l = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)

    def call():
        gb.attn_fwd_dense(q, k, v, w.scale, w.causal, out=o, lse=l, dev_status=status, stream=stream)

    for _ in range(20):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    call()
    e1.record(stream)
    torch.cuda.synchronize()
    n = max(50, int(seconds / (e0.elapsed_time(e1) * 1e-3)))
    with ClockSampler(clock_gpu) as clk:
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    tf = w.flops() / (ms * 1e-3) / 1e12
    peak = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the sustained leg")
    return {"workload": w.name, "calls": n, "seconds": n * ms * 1e-3, "ms_per_call": ms, "value": tf,
            "unit": "TFLOP/s", "peak": peak, "frac": tf / peak, "peak_kind": f"{peak_kind} bf16 sustained",
            "frac_of_burst_peak": tf / float(pk["bf16_tflops"]), "clocks": clk.summary()}


def run_ours(args, world, rank, local):
    import attention_forward_09_gb300 as gb
    from attention_forward_09_gb300 import _build

    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    gb.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, peak_kind = peaks()

    # ---- inputs (CPU, seeded), then resident in HBM
    do_pre, do_dec = args.only in ("all", "prefill"), args.only in ("all", "decode")
    wp = PREFILL_WORKLOADS[args.prefill]()
    varlen = isinstance(wp, workloads.Varlen)
    if varlen:
        q, k, v, cq, ck = wp.make()
    else:
        q, k, v = wp.make()
    if do_pre:
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        if varlen:
            cqd, ckd = cq.to(dev), ck.to(dev)
            outd = torch.empty(wp.Tq, wp.Hq, wp.D, dtype=torch.float32, device=dev)
            lsed = torch.empty(wp.Hq, wp.Tq, dtype=torch.float32, device=dev)
        else:
            outd = torch.empty(wp.B, wp.Sq, wp.Hq, wp.D, dtype=torch.float32, device=dev)
            lsed = torch.empty(wp.B, wp.Hq, wp.Sq, dtype=torch.float32, device=dev)
    wd = workloads.paged_decode()
    if args.decode_seqs:
        wd = workloads.Paged(wd.name + f"_first{args.decode_seqs}", wd.seq_lens[:args.decode_seqs], wd.Hq, wd.Hkv,
                             wd.D, seed=wd.seed, max_blocks_per_seq=wd.max_blocks_per_seq)
    max_len = max(wd.seq_lens)
    if do_dec:
        pq, cache, bt, sl = wd.make(chunk_rows=256)
        pqd, cached, btd, sld = pq.to(dev), cache.to(dev), bt.to(dev), sl.to(dev)
        ws = torch.empty(gb.attn_fwd_paged_workspace_size(len(wd.seq_lens), wd.Hq, wd.Hkv, wd.D, max_len),
                         dtype=torch.uint8, device=dev)
        pout = torch.empty(len(wd.seq_lens), wd.Hq, wd.D, dtype=torch.float32, device=dev)
        plse = torch.empty(len(wd.seq_lens), wd.Hq, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if not do_pre:
        pre_launches = 0
    elif varlen:
        pre_launches = 1
    else:
        pre_launches = gb.attn_fwd_dense_plan(wp.B, wp.Sq, wp.Sk, wp.Hq, wp.Hkv, wp.D, wp.causal)[0]

    def prefill():
        if do_pre and varlen:
            gb.attn_fwd_varlen(qd, kd, vd, cqd, ckd, max(wp.lens_q), max(wp.lens_k), wp.scale, wp.causal, out=outd,
                               lse=lsed, dev_status=status, stream=stream)
        elif do_pre:
            gb.attn_fwd_dense(qd, kd, vd, wp.scale, wp.causal, out=outd, lse=lsed, dev_status=status, stream=stream)

    def decode():
        if do_dec:
            gb.attn_fwd_paged(pqd, cached, btd, sld, max_len, wd.scale, out=pout, lse=plse, workspace=ws,
                              dev_status=status, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        prefill()
        decode()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            decode()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    pre_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    pre_avg = max_over_ranks(statistics.mean(pre_ms), world)
    dec_avg = max_over_ranks(statistics.mean(dec_ms), world)
    step_ms = max_over_ranks(statistics.mean(p + d for p, d in zip(pre_ms, dec_ms)), world)

    flops = wp.flops()
    tflops_rank = flops / (pre_avg * 1e-3) / 1e12 if do_pre else None
    value = sum_over_ranks(flops, world) / (pre_avg * 1e-3) / 1e12 if do_pre else None
    dec_bytes = wd.algorithmic_bytes(out_bytes_per_elem=4, with_lse=True)
    dec_gbs_rank = dec_bytes / (dec_avg * 1e-3) / 1e9 if do_dec else None
    dec_value = sum_over_ranks(dec_bytes, world) / (dec_avg * 1e-3) / 1e9 if do_dec else None
    peak_tf = float(pk["bf16_tflops"])
    peak_bw = float(pk["hbm_gbs"])

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if do_pre:
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        if varlen:  # the cu_seqlens travel too
            hcq, hck = cq.pin_memory(), ck.pin_memory()
        hout = torch.empty(outd.shape, dtype=torch.float32).pin_memory()
        hlse = torch.empty(lsed.shape, dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        for _ in range(e2e_steps):
            qd.copy_(hq, non_blocking=True)
            kd.copy_(hk, non_blocking=True)
            vd.copy_(hv, non_blocking=True)
            if varlen:
                cqd.copy_(hcq, non_blocking=True)
                ckd.copy_(hck, non_blocking=True)
            prefill()
            hout.copy_(outd, non_blocking=True)
            hlse.copy_(lsed, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

        # The same steps as a pipeline, as a serving loop would run them: two
        # sets of device buffers; step i+1's inputs go up and step i-1's
        # results come down on their own streams while step i computes.
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        sets = [{"q": qd, "k": kd, "v": vd, "out": outd, "lse": lsed},
                {"q": torch.empty_like(qd), "k": torch.empty_like(kd), "v": torch.empty_like(vd),
                 "out": torch.empty_like(outd), "lse": torch.empty_like(lsed)}]
        if varlen:
            sets[0].update(cq=cqd, ck=ckd)
            sets[1].update(cq=torch.empty_like(cqd), ck=torch.empty_like(ckd))
        hosts = [(hout, hlse), (torch.empty_like(hout).pin_memory(), torch.empty_like(hlse).pin_memory())]
        ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("inp", "cmp", "out")}

        def call(b, st):
            if varlen:
                gb.attn_fwd_varlen(b["q"], b["k"], b["v"], b["cq"], b["ck"], max(wp.lens_q), max(wp.lens_k), wp.scale,
                                   wp.causal, out=b["out"], lse=b["lse"], dev_status=status, stream=st)
            else:
                gb.attn_fwd_dense(b["q"], b["k"], b["v"], wp.scale, wp.causal, out=b["out"], lse=b["lse"],
                                  dev_status=status, stream=st)

        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        p0.record(s_in)
        for i in range(e2e_steps):
            b, (ho, hl), k2 = sets[i % 2], hosts[i % 2], i % 2
            if i >= 2:
                s_in.wait_event(ev["cmp"][k2])   # step i-2 has read these inputs
            with torch.cuda.stream(s_in):
                b["q"].copy_(hq, non_blocking=True)
                b["k"].copy_(hk, non_blocking=True)
                b["v"].copy_(hv, non_blocking=True)
                if varlen:
                    b["cq"].copy_(hcq, non_blocking=True)
                    b["ck"].copy_(hck, non_blocking=True)
            ev["inp"][k2].record(s_in)
            s_cmp.wait_event(ev["inp"][k2])
            if i >= 2:
                s_cmp.wait_event(ev["out"][k2])  # step i-2's results have been read back
            call(b, s_cmp)
            ev["cmp"][k2].record(s_cmp)
            s_out.wait_event(ev["cmp"][k2])
            with torch.cuda.stream(s_out):
                ho.copy_(b["out"], non_blocking=True)
                hl.copy_(b["lse"], non_blocking=True)
            ev["out"][k2].record(s_out)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_cmp)
        p1.record(s_out)
        torch.cuda.synchronize()
        pipe_ms = max_over_ranks(p0.elapsed_time(p1) / e2e_steps, world)
        # same inputs every step: the last result read back must equal the device-timed run's
        same = bool(torch.equal(hosts[(e2e_steps - 1) % 2][0], outd.cpu()))
        h2d = (q.numel() + k.numel() + v.numel()) * 2 + (8 * (len(wp.lens_q) + 1) if varlen else 0)
        d2h = hout.numel() * 4 + hlse.numel() * 4
        e2e = {"value": flops / (pipe_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "ms_per_step": pipe_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "pipelined": "inputs of step i+1 up and results of step i-1 down on their own streams during "
                            "step i (two buffer sets)",
               "sequential": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "ms_per_step": e2e_ms},
               "result_matches_device_run": same}

    # ---- every workload of the metric on its own, then the headline prefill sustained
    configs, sustained = None, None
    if args.only == "all" and not args.no_configs:
        configs = measure_configs(gb, dev, stream, status, flush, args.steps, args.warmup, pk, peak_kind)
        sustained = sustained_prefill(gb, dev, stream, status, args.sustained_s, pk, peak_kind, local)

    # ---- oracle on the host cores (rank 0, N=1 only)
    cpu, cpu_dec = None, None
    if world == 1 and not args.no_cpu:
        if do_pre and not varlen:
            tf, desc, _ = oracle_prefill_sample(wp, 10.0, (q, k, v))
            cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle", "sample": desc}
        if do_dec:
            gbs, ddesc, _ = oracle_paged_sample(wd, pq, cache, bt, sl, 8.0)
            cpu_dec = {"value": gbs, "unit": "GB/s", "cores": cores_used(), "kind": "oracle", "sample": ddesc}

    if rank != 0:
        return
    pre_kernel = (f"fmha2_fwd_sm103a<Prefill2Cfg<{wp.D}>>" if wp.D <= 128 else f"fmha_fwd_sm103a<PrefillCfg<{wp.D}>>")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{wp.name} + {wd.name}",
            "prefill": ({"docs": len(wp.lens_q), "tokens": wp.Tq, "max_doc": max(wp.lens_q), "heads": wp.Hq,
                         "kv_heads": wp.Hkv, "head_dim": wp.D, "causal": wp.causal, "out_dtype": "f32", "lse": True}
                        if varlen else
                        {"B": wp.B, "seq_len": wp.Sq, "kv_len": wp.Sk, "heads": wp.Hq, "kv_heads": wp.Hkv,
                         "head_dim": wp.D, "causal": wp.causal, "out_dtype": "f32", "lse": True}),
            "decode": {"num_seqs": len(wd.seq_lens), "context_tokens": wd.context_tokens(),
                       "max_seq_len": max_len, "heads": wd.Hq, "kv_heads": wd.Hkv, "head_dim": wd.D,
                       "block_size": 128, "num_blocks": wd.num_blocks},
            "l2": "512 MiB buffer rewritten between steps (flush); decode cache 4.4 GB > L2",
            "parallelism": f"replicas x{world}",
            "only": args.only,
        },
        "roofline": {
            "bound": "tensor", "kernel": pre_kernel, "launches_per_call": pre_launches,
            "achieved": tflops_rank, "peak": peak_tf,
            "unit": "TFLOP/s", "frac": tflops_rank / peak_tf if do_pre else None, "peak_kind": f"{peak_kind} bf16 burst",
            "traffic": traffic_for(f"{pre_kernel.split('<')[0]}@{wp.name}", "prefill.cu"),
            "flops_per_launch": flops, "launch_ms": pre_avg,
        },
        "paged_decode": {
            "value": dec_value, "unit": "GB/s", "ms": dec_avg,
            "roofline": {"bound": "hbm", "kernel": "paged_schedule + paged_decode_sm103a + paged_combine", "achieved": dec_gbs_rank,
                         "peak": peak_bw, "unit": "GB/s", "frac": dec_gbs_rank / peak_bw if do_dec else None,
                         "peak_kind": f"{peak_kind} HBM copy", "bytes_per_call": dec_bytes,
                         "traffic": traffic_for(f"paged_decode_sm103a@{wd.name}", "decode.cu")},
            "cpu_baseline": cpu_dec,
        },
        "configs": configs,
        "sustained": sustained,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: the prefill launches (full waves, then the split last wave);
        # the decode schedule, decode and combine kernels
        "gpu_launches": (pre_launches + 3 * int(do_dec)) * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


def run_kv_write(args, world, rank, local):
    """`--only kv_write`: the KV cache write of a prefill step (the packed
    causal GQA workload's K/V stored through slot_mapping), HBM GB/s."""
    import attention_forward_09_gb300 as gb
    from attention_forward_09_gb300 import _build

    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    gb.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, peak_kind = peaks()
    w = workloads.prefill_kv_write()
    k, v, slots, shape = w.make()
    kd, vd, sd = k.to(dev), v.to(dev), slots.to(dev)
    cache = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def write(kk, vv, ss):
        gb.attn_kv_cache_write(kk, vv, ss, cache, dev_status=status, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        write(kd, vd, sd)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            write(kd, vd, sd)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world)
    nbytes = w.algorithmic_bytes()
    gbs_rank = nbytes / (ms * 1e-3) / 1e9
    value = sum_over_ranks(nbytes, world) / (ms * 1e-3) / 1e9

    # end to end: K, V and slots up from pinned host memory, the status word back
    hk, hv, hs = k.pin_memory(), v.pin_memory(), slots.pin_memory()
    hst = torch.empty(1, dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        sd.copy_(hs, non_blocking=True)
        write(kd, vd, sd)
        hst.copy_(status, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = (k.numel() + v.numel()) * 2 + slots.numel() * 4

    cpu = None
    if world == 1 and not args.no_cpu:  # the oracle on one whole call (about a second)
        import oracle

        base = torch.zeros(shape, dtype=torch.bfloat16)
        t0 = time.perf_counter()
        ref = oracle.kv_cache_write(k, v, slots, base)
        el = time.perf_counter() - t0
        cpu = {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
               "sample": f"one whole call: {w.tokens} tokens of {w.name}",
               "matches": bool(torch.equal(ref.view(torch.int16), cache.cpu().view(torch.int16)))}
    if rank != 0:
        return
    line = {
        "metric": "kv cache write HBM GB/s & % of HBM peak", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "kv_heads": w.Hkv, "head_dim": w.D,
                   "block_size": w.block_size, "num_blocks": w.num_blocks,
                   "l2": "512 MiB buffer rewritten between steps (flush)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "kv_cache_write_sm103a", "achieved": gbs_rank,
                     "peak": float(pk["hbm_gbs"]), "unit": "GB/s", "frac": gbs_rank / float(pk["hbm_gbs"]),
                     "peak_kind": f"{peak_kind} HBM copy", "bytes_per_call": nbytes,
                     "traffic": traffic_for(f"kv_cache_write_sm103a@{w.name}", "cache_write.cu")},
        "cpu_baseline": cpu,
        "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


PAGED_PREFILL_WORKLOADS = {"chunked_prefill": workloads.chunked_prefill, "spec_decode": workloads.spec_decode}


def run_paged_prefill(args, world, rank, local):
    """`--only paged_prefill`: several query tokens per sequence over the
    paged cache (`--paged-prefill chunked_prefill|spec_decode`), TFLOP/s."""
    import attention_forward_09_gb300 as gb
    from attention_forward_09_gb300 import _build

    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    gb.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, peak_kind = peaks()
    w = PAGED_PREFILL_WORKLOADS[args.paged_prefill]()
    q, cache, bt, sl, cu = w.make()
    qd, cached, btd, sld, cud = q.to(dev), cache.to(dev), bt.to(dev), sl.to(dev), cu.to(dev)
    Tq = q.shape[0]
    outd = torch.empty(Tq, w.Hq, w.D, dtype=torch.float32, device=dev)
    lsed = torch.empty(w.Hq, Tq, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    mq, ml = max(w.q_lens), max(w.seq_lens)

    def run():
        gb.attn_fwd_paged_prefill(qd, cached, btd, sld, cud, mq, ml, w.scale, w.causal, out=outd, lse=lsed,
                                  dev_status=status, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        run()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world)
    flops = w.flops()
    tf_rank = flops / (ms * 1e-3) / 1e12
    value = sum_over_ranks(flops, world) / (ms * 1e-3) / 1e12
    kv_bytes = 2 * sum(w.seq_lens) * w.Hkv * w.D * 2

    # end to end: the step's new queries and metadata up (the cache is resident), out and lse back
    hq, hcu, hbt, hsl = q.pin_memory(), cu.pin_memory(), bt.pin_memory(), sl.pin_memory()
    hout, hlse = torch.empty(outd.shape).pin_memory(), torch.empty(lsed.shape).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in ((qd, hq), (cud, hcu), (btd, hbt), (sld, hsl)):
            d_.copy_(h_, non_blocking=True)
        run()
        hout.copy_(outd, non_blocking=True)
        hlse.copy_(lsed, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = q.numel() * 2 + (cu.numel() + bt.numel() + sl.numel()) * 4

    cpu = None
    if world == 1 and not args.no_cpu:  # the oracle on the shortest sequences, about 10 s
        import oracle

        t0, done, fl = time.perf_counter(), 0, 0.0
        order = sorted(range(len(w.seq_lens)), key=lambda s: w.seq_lens[s])
        for s in order:
            a, b = int(cu[s]), int(cu[s + 1])
            oracle.attention_paged_prefill(q[a:b], cache, bt[s:s + 1], sl[s:s + 1], torch.tensor([0, b - a]),
                                           w.scale, w.causal)
            fl += 4.0 * w.D * w.Hq * sum(max(0, min(w.seq_lens[s], i + w.seq_lens[s] - (b - a) + 1))
                                           for i in range(b - a))
            done += 1
            if time.perf_counter() - t0 > 10.0:
                break
        el = time.perf_counter() - t0
        cpu = {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": f"{done} of {len(order)} sequences of {w.name} (shortest first)"}
    if rank != 0:
        return
    peak_tf = float(pk["bf16_tflops"])
    line = {
        "metric": "paged prefill TFLOP/s & % bf16 TC peak", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": len(w.seq_lens), "q_len": mq, "context_tokens": sum(w.seq_lens),
                   "heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D, "causal": w.causal, "block_size": 128,
                   "l2": "512 MiB buffer rewritten between steps (flush)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": f"fmha2_fwd_sm103a<Prefill2Cfg<{w.D}>> (paged)",
                     "achieved": tf_rank, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf_rank / peak_tf,
                     "peak_kind": f"{peak_kind} bf16 burst", "flops_per_launch": flops, "traffic": None},
        "kv_read": {"bytes": kv_bytes, "GB/s": kv_bytes / (ms * 1e-3) / 1e9,
                    "frac_of_hbm": kv_bytes / (ms * 1e-3) / 1e9 / float(pk["hbm_gbs"])},
        "cpu_baseline": cpu,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * 4 + hlse.numel() * 4},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


def run_masked(args, world, rank, local):
    """`--only masked`: a right-padded batch (each row keeps its first tokens)
    two ways: attn_fwd_padded, which reads the padded tensors in place with
    per-row lengths (the headline value), and attn_fwd_masked, the general
    padding-mask pipeline (mask -> cu_seqlens, pack, varlen attention,
    unpack), in `general_mask`; TFLOP/s on the kept tokens."""
    import attention_forward_09_gb300 as gb
    from attention_forward_09_gb300 import _build

    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    gb.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, peak_kind = peaks()
    w = workloads.masked_dit()
    q, k, v, mask = w.make()
    qd, kd, vd, md = q.to(dev), k.to(dev), v.to(dev), mask.to(dev)
    lens = torch.tensor(w.lens, dtype=torch.int32)
    lensd = lens.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    outd = torch.empty(w.B, w.S, w.Hq, w.D, dtype=torch.float32, device=dev)
    lsed = torch.empty(w.B, w.Hq, w.S, dtype=torch.float32, device=dev)

    def run_padded():
        return gb.attn_fwd_padded(qd, kd, vd, lensd, lensd, w.scale, w.causal, out=outd, lse=lsed,
                                  dev_status=status, stream=stream)

    def run_general():
        return gb.attn_fwd_masked(qd, kd, vd, md, w.scale, w.causal, lse=True, dev_status=status, stream=stream)

    def timed(fn):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            fn()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world)

    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        ms = timed(run_padded)
        t_wall = time.perf_counter() - t_wall
        ms_general = timed(run_general)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    # the two routes give the same result on a right-padded batch
    o1, l1 = run_padded()
    o2, l2 = run_general()
    torch.cuda.synchronize()
    max_diff = float((o1 - o2).abs().max())
    same_padding = bool(torch.equal(torch.isinf(l1), torch.isinf(l2)))
    flops = w.flops()
    tf_rank = flops / (ms * 1e-3) / 1e12
    value = sum_over_ranks(flops, world) / (ms * 1e-3) / 1e12
    tf_general = flops / (ms_general * 1e-3) / 1e12

    hq_, hk_, hv_, hl_ = q.pin_memory(), k.pin_memory(), v.pin_memory(), lens.pin_memory()
    hout, hlse = torch.empty(outd.shape).pin_memory(), torch.empty(lsed.shape).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in ((qd, hq_), (kd, hk_), (vd, hv_), (lensd, hl_)):
            d_.copy_(h_, non_blocking=True)
        o, l = run_padded()
        hout.copy_(o, non_blocking=True)
        hlse.copy_(l, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    if rank != 0:
        return
    peak_tf = float(pk["bf16_tflops"])
    launches = gb.attn_fwd_dense_plan(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, w.causal)[0]
    line = {
        "metric": "masked attention TFLOP/s & % bf16 TC peak", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "seq_len": w.S, "kept": w.lens, "heads": w.Hq, "head_dim": w.D,
                   "causal": w.causal, "route": "attn_fwd_padded (per-row lengths, tensors read in place)",
                   "l2": "512 MiB buffer rewritten between steps (flush)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": f"fmha2_fwd_sm103a<Prefill2Cfg<{w.D}>> (padded batch)",
                     "launches_per_call": launches, "achieved": tf_rank, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": tf_rank / peak_tf, "peak_kind": f"{peak_kind} bf16 burst", "flops_per_launch": flops,
                     "traffic": None},
        "general_mask": {"route": "attn_fwd_masked: mask_to_varlen + 3 x pack_rows + varlen attention + "
                                  "unpack_rows + unpack_lse", "value": tf_general, "unit": "TFLOP/s",
                         "ms": ms_general, "frac": tf_general / peak_tf, "launches_per_call": 7,
                         "max_abs_out_diff_vs_padded": max_diff, "same_padded_rows_as_padded": same_padding},
        "cpu_baseline": None,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2 + lens.numel() * 4,
                "d2h_bytes_per_step": hout.numel() * 4 + hlse.numel() * 4},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


def vsa_kept_pairs(kv_list, kv_num, nb, npre, topk, sizes):
    """Query-key pairs the block-sparse attention computes, counted from its
    per-tile lists: per entry, the key block's tokens times the tokens of
    each query block of the tile that keeps it (list placement as stated
    with attn_vsa_block_map)."""
    import attention_forward_09_gb300 as gb

    kl, kn = kv_list.cpu().numpy().astype(np.int64), kv_num.cpu().numpy()
    sz = np.asarray(sizes, dtype=np.int64)
    sz_pad = np.append(sz, 0)
    nt, keep = (nb + 1) // 2, min(topk, nb - npre)
    td = nt if keep == nb - npre else min(nt, (npre + 1) // 2)
    c2 = min(nb, npre + 2 * keep)
    per_head = gb.attn_vsa_list_size(nb, npre, topk, 1)
    pairs = 0
    for h in range(kn.shape[0]):
        for t in range(nt):
            off = h * per_head + (t * nb if t < td else td * nb + (t - td) * c2)
            e = kl[off:off + int(kn[h, t])]
            q0, q1 = sz[2 * t], sz_pad[2 * t + 1]
            pairs += int((sz[e >> 9] * (((e & 1) != 0) * q0 + ((e & 2) != 0) * q1)).sum())
    return pairs


def run_vsa(args, world, rank, local):
    """`--only vsa`: block-sparse video attention of one sequence (tile q, k,
    v; pool; block map; attention), TFLOP/s on the query-key pairs it keeps."""
    import attention_forward_09_gb300 as gb
    from attention_forward_09_gb300 import _build

    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    gb.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, peak_kind = peaks()
    w = workloads.vsa_video(args.vsa_frames)
    q, k, v = w.make()
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    plan = gb.VsaPlan(w.prefix, w.video, dev)
    nb, npre = plan.num_blocks, plan.num_prefix_blocks
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd_ev = []

    def run(time_fwd=False):
        qt, kt, vt = (gb.attn_gather_rows(x, plan.tile_index, status, stream) for x in (qd, kd, vd))
        pq = gb.attn_vsa_pool(qt, plan.block_sizes, status, stream)
        pkk = gb.attn_vsa_pool(kt, plan.block_sizes, status, stream)
        kl, kn = gb.attn_vsa_block_map(pq, pkk, plan.block_sizes, npre, w.topk, w.scale, status, stream)
        if time_fwd:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record(stream)
        out, lse = gb.attn_fwd_vsa(qt, kt, vt, kl, kn, nb, npre, w.topk, out_index=plan.tile_index,
                                   out_rows=w.tokens, softmax_scale=w.scale, lse=True, dev_status=status,
                                   stream=stream)
        if time_fwd:
            e[1].record(stream)
            fwd_ev.append(e)
        return out, lse, kl, kn

    for _ in range(args.warmup):
        _, _, kl0, kn0 = run()
    torch.cuda.synchronize()
    flops = 4.0 * w.D * vsa_kept_pairs(kl0, kn0, nb, npre, w.topk, plan.block_sizes.cpu().tolist())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            run(time_fwd=True)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev)
    value = sum_over_ranks(flops, world) / (ms * 1e-3) / 1e12
    tf_fwd = flops / (fwd_ms * 1e-3) / 1e12

    hq_, hk_, hv_ = q.pin_memory(), k.pin_memory(), v.pin_memory()
    out0, lse0, _, _ = run()
    hout, hlse = torch.empty(out0.shape).pin_memory(), torch.empty(lse0.shape).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in ((qd, hq_), (kd, hk_), (vd, hv_)):
            d_.copy_(h_, non_blocking=True)
        o, l, _, _ = run()
        hout.copy_(o, non_blocking=True)
        hlse.copy_(l, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    cpu = None
    if world == 1 and not args.no_cpu:  # the oracle: one head's block map, then query blocks for about 10 s
        import oracle

        t0 = time.perf_counter()
        blocks, n_pre = oracle.vsa_blocks(w.prefix, w.video)
        bm = oracle.vsa_block_map(q[:, :1], k[:, :1], blocks, n_pre, w.topk, w.scale)[0]
        fl, done = 0.0, 0
        for i in range(n_pre, nb):
            keys = torch.from_numpy(np.concatenate([blocks[j] for j in np.nonzero(bm[i])[0]]))
            oracle.attention_single(q[torch.from_numpy(blocks[i]), :1], k[keys, :1], v[keys, :1], w.scale, False)
            fl += 4.0 * w.D * len(blocks[i]) * len(keys)
            done += 1
            if time.perf_counter() - t0 > 10.0:
                break
        dt = time.perf_counter() - t0
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": f"head 0: the block map of all {nb} blocks, then {done} video query blocks "
                         f"({dt:.1f} s, map time included)"}
    if rank != 0:
        return
    peak_tf = float(pk["bf16_tflops"])
    line = {
        "metric": "block-sparse video attention TFLOP/s (kept pairs) & % bf16 TC peak", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "prefix": w.prefix, "video": list(w.video), "tokens": w.tokens,
                   "blocks": nb, "topk": w.topk, "heads": w.Hq, "head_dim": w.D,
                   "density": flops / (4.0 * w.D * w.Hq * w.tokens ** 2),
                   "l2": "inputs larger than L2 (3 x 780 MB, tiled copies rewritten every step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "vsa_fwd_sm103a", "achieved": tf_fwd, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": tf_fwd / peak_tf, "peak_kind": f"{peak_kind} bf16 burst",
                     "flops_per_launch": flops, "fwd_ms": fwd_ms,
                     "traffic": traffic_for("vsa_fwd_sm103a@" + w.name, "vsa.cu")},
        "cpu_baseline": cpu,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
                "d2h_bytes_per_step": hout.numel() * 4 + hlse.numel() * 4},
        "gpu_launches": 7 * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--prefill", choices=sorted(PREFILL_WORKLOADS), default="dit_self",
                    help="prefill workload of the step (default: the headline DiT self-attention)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--paged-prefill", choices=sorted(PAGED_PREFILL_WORKLOADS), default="chunked_prefill",
                    help="workload of --only paged_prefill")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "kv_write", "paged_prefill", "masked", "vsa"],
                    default="all",
                    help="run one part of the step (profiling captures), or the KV cache write alone; "
                         "the default line needs 'all'")
    ap.add_argument("--decode-seqs", type=int, default=0,
                    help="use only the first N sequences of the decode workload (profiling captures)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle timing")
    ap.add_argument("--vsa-frames", type=int, default=21,
                    help="frames of the video grid of --only vsa (fewer: a smaller profiling capture)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing every workload of the metric and the sustained leg (profiling captures)")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back headline prefill in the sustained leg")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.only == "kv_write":
        run_kv_write(args, world, rank, local)
    elif args.only == "paged_prefill":
        run_paged_prefill(args, world, rank, local)
    elif args.only == "masked":
        run_masked(args, world, rank, local)
    elif args.only == "vsa":
        run_vsa(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
