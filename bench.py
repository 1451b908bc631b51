#!/usr/bin/env python3
"""Benchmark of the KDA chunked forward pass on GB300.

Default workload: fixed-length prefill, B = 1, T = 8192, H = 96, K = V = 128, bf16
initial and final state (the H = 96 fixed-length row of the FlashKDA benchmark
tables).  One step = one kda_fwd call over the whole workload: the prep kernel (all chunks
in parallel) and the recurrence kernel (plus a one-CTA plan kernel with cu_seqlens).
Inputs (1.0 GB) exceed the 129 MB L2, so no flush is needed between steps.

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle instead (the
reference arm for this method: a deliberately plain program on the host cores).
Under torchrun each rank runs its own replica of the workload (weak scaling, no
collective on the data path); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_23_gb300.inputs import STATE_BF16, STATE_FP32, WORKLOADS, make_workload  # noqa: E402

METRIC = "KDA fwd ms & tokens·heads/s at T=8192 H=96; % of HBM/tensor roofline"
UNIT = "tokens·heads/s"
KERNEL_DIR = os.path.join(ROOT, "gated_delta_rule_23_gb300", "csrc")
PROFILE_DIR = os.path.join(ROOT, "profiles")
# device sources each kernel is compiled from (a profile summary is valid only for these)
KERNEL_SOURCES = {"kda_prep_kernel": ["kda_device.cuh", "kda_prep.cu"],
                  "kda_recur_kernel": ["kda_device.cuh", "kda_recur.cu"],
                  "kda_recurrent_kernel": ["kda_device.cuh", "kda_recurrent.cu"],
                  "kda_decode_kernel": ["kda_device.cuh", "kda_decode.cu"]}
SLOT_BYTES_PER_CHUNK_HEAD = 74240   # fp16 operands the prep kernel hands to the recurrence kernel per (64-token chunk, head)
# FlashKDA on GB200, H=96 fixed length, T=8192: 1.01 ms (guancyxx.cn FlashKDA article, section 三,
# GB200 table) -> tokens*heads per second.  Another machine: context, not the target.
PAGES_GB200_TOKHEADS_PER_S = 8192 * 96 / 1.01e-3


def workload_config(p, idx):
    st = {STATE_BF16: "bf16", STATE_FP32: "fp32"}.get(p.state_dtype, "none")
    return {
        "workload": WORKLOADS[idx], "B": p.B, "T": p.T, "H": p.H, "K": 128, "V": 128,
        "state_dtype": st, "initial_state": p.initial_state is not None, "final_state": p.want_final,
        "varlen_lengths": None if p.cu_seqlens is None else [int(x) for x in np.diff(p.cu_seqlens)],
        "l2": "inputs larger than L2 (no flush)",
    }


def algorithmic_bytes(p):
    """HBM bytes one launch must move: q, k, v, g, beta in; out; states; parameters."""
    th = p.token_heads()
    b = th * (4 * 128 * 2 + 2 + 128 * 2)
    es = {STATE_BF16: 2, STATE_FP32: 4}.get(p.state_dtype, 0)
    per_state = p.N * p.H * 128 * 128 * es
    b += per_state * ((p.initial_state is not None) + bool(p.want_final and es))
    b += p.H * 4 + p.H * 128 * 4 + (0 if p.cu_seqlens is None else 8 * (p.N + 1))
    return b


def kernel_bytes(p):
    """HBM bytes each kernel must move in this design (the workspace slots count here, not in the path)."""
    th = p.token_heads()
    es = {STATE_BF16: 2, STATE_FP32: 4}.get(p.state_dtype, 0)
    per_state = p.N * p.H * 128 * 128 * es
    states = per_state * ((p.initial_state is not None) + bool(p.want_final and es))
    lengths = p.seq_lengths()
    slots = int(sum((int(n) + 63) // 64 for n in lengths)) * p.H * SLOT_BYTES_PER_CHUNK_HEAD
    prep = th * (4 * 128 * 2 + 2) + slots + p.H * (4 + 128 * 4)
    recur = slots + th * 128 * 2 + states
    return {"kda_prep_kernel": prep, "kda_recur_kernel": recur}


def algorithmic_flops(p, chunk=64):
    """Dense FLOPs of the chunked method per token*head: 6 K V for the three state products
    (W S, Q~ S, K~^T U) plus 10 C 128 for the intra-chunk products (Akk, Aqk, W, U0, Aqk U)."""
    return p.token_heads() * (6 * 128 * 128 + 10 * chunk * 128)


def kernel_algorithmic_bytes(p):
    """The share of the call's algorithmic bytes each kernel moves: the prep kernel reads the token
    tensors and parameters, the recurrence kernel writes out and reads / writes the states."""
    th = p.token_heads()
    es = {STATE_BF16: 2, STATE_FP32: 4}.get(p.state_dtype, 0)
    per_state = p.N * p.H * 128 * 128 * es
    states = per_state * ((p.initial_state is not None) + bool(p.want_final and es))
    cu = 0 if p.cu_seqlens is None else 8 * (p.N + 1)
    return {"kda_prep_kernel": th * (4 * 128 * 2 + 2) + p.H * (4 + 128 * 4),
            "kda_recur_kernel": th * 128 * 2 + states + cu}


def kernel_source_hash(kernel):
    """Hash of the device sources `kernel` is built from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(KERNEL_DIR, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` (a workload index, or "decode") from a committed
    ncu summary under profiles/, if it was taken on that workload and on the kernel's current sources."""
    want = kernel_source_hash(kernel)
    for name in sorted(os.listdir(PROFILE_DIR)):
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(PROFILE_DIR, name)).read()
        m_src = re.search(kernel + r" source_sha256_16:\s*([0-9a-f]+)", text)
        m_tr = re.search(kernel + r" traffic_bytes_per_launch:\s*([0-9.e+]+)", text)
        m_wl = re.search(kernel + r" traffic_workload:\s*(\S+)", text)
        if m_src and m_tr and m_wl and m_src.group(1) == want and m_wl.group(1) == str(workload):
            return float(m_tr.group(1))
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms between start() and stop()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.samples = []
        self.proc = None
        self.window = None
        self.device_index = device_index

    def _gpu_id(self):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.device_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def start(self):
        gid = self._gpu_id()
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gid:
            cmd += ["-i", gid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 7:
                continue
            rows.append((ts, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if self.window and self.window[0] - 0.2 <= r[0] <= self.window[1] + 0.2]
        if not inside:   # timed region shorter than one sampling period: nearest sample
            mid = sum(self.window) / 2 if self.window else rows[-1][0]
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1][0]) for r in inside if num(r[1][0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[1][3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][1][1]), "reasons": reasons, "samples": len(inside),
                "power_w_max": max((num(r[1][2]) or 0.0) for r in inside)}


def cpu_baseline(p, idx, max_heads=24):
    """The oracle, as it stands, on a bounded sample: the first heads over every token."""
    import oracle
    from gated_delta_rule_23_gb300.inputs import subset_heads
    nh = min(p.H, max_heads)
    sub = subset_heads(p, list(range(nh)))
    threads = min(oracle.default_threads(), nh * p.N)
    t0 = time.perf_counter()
    oracle.kda_fwd_problem(sub, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": sub.token_heads() / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{nh} of {p.H} heads, all {int(p.seq_lengths().sum())} tokens of workload {idx}; "
                      f"fp64 token-by-token recurrence, {dt:.2f} s wall"}


def run_reference(args, p, idx, rank):
    """Reference arm: the CPU oracle timed per step on a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle
    from gated_delta_rule_23_gb300.inputs import subset_heads
    threads = oracle.default_threads()
    nh = min(p.H, threads)
    ntok = min(1024, p.T)
    sub = subset_heads(p, list(range(nh)))
    if sub.cu_seqlens is None:
        import dataclasses
        sub = dataclasses.replace(sub, q=sub.q[:, :ntok].copy(), k=sub.k[:, :ntok].copy(), v=sub.v[:, :ntok].copy(),
                                  g=sub.g[:, :ntok].copy(), beta=sub.beta[:, :ntok].copy())
    else:   # the first sequences up to ~ntok tokens
        import dataclasses
        cu = sub.cu_seqlens
        n_keep = max(1, int(np.searchsorted(cu, ntok, side="right")) - 1)
        end = int(cu[n_keep])
        sub = dataclasses.replace(sub, q=sub.q[:, :end].copy(), k=sub.k[:, :end].copy(), v=sub.v[:, :end].copy(),
                                  g=sub.g[:, :end].copy(), beta=sub.beta[:, :end].copy(), cu_seqlens=cu[:n_keep + 1].copy(),
                                  initial_state=None if sub.initial_state is None else sub.initial_state[:n_keep].copy())
    for _ in range(args.warmup):
        oracle.kda_fwd_problem(sub, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kda_fwd_problem(sub, nthreads=threads)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = sub.token_heads() / dt
    sample = f"{nh} heads x {int(sub.seq_lengths().sum())} tokens of workload {idx} per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, idx),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def max_over_ranks(ms, world, device):
    """The slowest rank's time: every rank passes its own measured milliseconds and gets the maximum
    (a barrier plus an all-reduce; NCCL on the GPU, gloo in the CPU tests)."""
    if world == 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    dist.barrier()
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank, world, ms):
    """Whole-job throughput of `world` replicas: the units all ranks processed over the slowest rank's
    time in milliseconds."""
    return units_per_rank * world / (ms * 1e-3)


DECODE_N, DECODE_H = 256, 96


def measure_decode(stream, steps=50, warmup=5, n_seq=DECODE_N, T=1):
    """One decode step (T = 1) for 256 sequences at 96 heads with an fp32 state updated in place,
    through the token-recurrent entry point (its decode kernel) and, for comparison, through the
    chunked one; then the same step with a bf16 state.  The states (1.6 / 0.8 GB) are larger than
    L2, so no flush is needed between steps."""
    import torch
    from gated_delta_rule_23_gb300 import kda_fwd, kda_fwd_recurrent
    from gated_delta_rule_23_gb300.inputs import make_problem
    from gated_delta_rule_23_gb300.device import to_device

    p = make_problem(B=n_seq, T=T, H=DECODE_H, seed=77)
    dev = to_device(p)
    out = torch.empty_like(dev["q"])
    st = dev["init"]
    args = (dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_rec = timed(lambda: kda_fwd_recurrent(*args, initial_state=st, final_state=st, stream=stream))
    ms_chk = timed(lambda: kda_fwd(*args, initial_state=st, final_state=st, stream=stream))
    st16 = st.to(torch.bfloat16)
    ms_rec16 = timed(lambda: kda_fwd_recurrent(*args, initial_state=st16, final_state=st16, stream=stream))
    th = n_seq * T * DECODE_H
    state_bytes = 2 * n_seq * DECODE_H * 128 * 128 * 4
    token_bytes = th * (4 * 128 * 2 + 2 + 128 * 2)
    hbm = peaks()[0]
    ach = (state_bytes + token_bytes) / (ms_rec * 1e-3) / 1e9
    kern = "kda_decode_kernel" if 2 <= T <= 4 else "kda_recurrent_kernel"   # fp32 state: T = 1 runs staged
    wkey = "decode" if (n_seq, T) == (DECODE_N, 1) else f"decode_N{n_seq}_T{T}"
    return {"entry": "kda_fwd_recurrent", "workload": f"decode step: N={n_seq} sequences x T={T}, H={DECODE_H}, "
                                                      "fp32 state in place",
            "ms": ms_rec, "value": th / (ms_rec * 1e-3), "unit": "tokens*heads/s",
            "bytes_per_step": state_bytes + token_bytes,
            "roofline": {"bound": "hbm", "kernel": kern, "achieved": ach, "peak": hbm,
                         "unit": "GB/s", "frac": ach / hbm, "traffic": measured_traffic(kern, wkey)},
            "chunked_entry_ms": ms_chk, "steps": steps, "warmup": warmup,
            "bf16_state": {"ms": ms_rec16, "kernel": "kda_decode_kernel" if T <= 4 else "kda_recurrent_kernel",
                       "bytes_per_step": state_bytes // 2 + token_bytes,
                           "achieved": (state_bytes // 2 + token_bytes) / (ms_rec16 * 1e-3) / 1e9,
                           "frac": (state_bytes // 2 + token_bytes) / (ms_rec16 * 1e-3) / 1e9 / hbm,
                           "traffic": measured_traffic("kda_decode_kernel" if T <= 4 else "kda_recurrent_kernel",
                                                       wkey + "_bf16")}}


def measure_link(h2d_bytes, d2h_bytes, reps=3):
    """Host-link bandwidth of plain pinned copies of the e2e step's byte counts: H2D alone, D2H alone, and both
    at once on two streams (best of `reps`, CUDA events on the copy streams)."""
    import torch
    hin = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device="cuda")
    dout = torch.empty(d2h_bytes, dtype=torch.uint8, device="cuda")
    hout = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(pairs):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            evs = []
            for dst, src, st in pairs:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(st):
                    e0.record(st)
                    dst.copy_(src, non_blocking=True)
                    e1.record(st)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            ms = max(e0.elapsed_time(e1) for e0, e1 in evs)
            best = ms if best is None else min(best, ms)
        return best
    h2d_ms = timed([(din, hin, s1)])
    d2h_ms = timed([(hout, dout, s2)])
    both_ms = timed([(din, hin, s1), (hout, dout, s2)])
    return {"h2d_ms": h2d_ms, "h2d_gbs": h2d_bytes / (h2d_ms * 1e-3) / 1e9, "d2h_ms": d2h_ms,
            "d2h_gbs": d2h_bytes / (d2h_ms * 1e-3) / 1e9, "both_ms": both_ms, "floor_ms": both_ms}


def run_ours(args, p, idx, rank, world):
    import torch
    import torch.distributed as dist
    from gated_delta_rule_23_gb300 import kda_fwd, kda_fwd_host
    from gated_delta_rule_23_gb300.device import to_device

    dev = to_device(p)
    out = torch.empty_like(dev["q"])
    fin = torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"], device="cuda") if dev["sdt"] is not None else None
    stream = torch.cuda.current_stream()

    def step():
        kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
                p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    if rank == 0 and not args.kernel_only:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    sampler.mark(t_host0, t_host1)
    sampler.stop()
    ms_step = ms_total / args.steps

    # per-kernel breakdown: the same calls through kda_fwd_ws_profiled, which records events at the
    # kernel boundaries on the launching stream (always the single-launch schedule: one prep launch over
    # every chunk, then the recurrence, also where the timed step runs in pieces)
    from gated_delta_rule_23_gb300 import workspace_size
    ws = torch.empty(workspace_size(p.N, p.T, p.H, p.cu_seqlens is not None), dtype=torch.uint8, device="cuda")
    n_prof = max(3, min(args.steps, 100))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_prof)]
    for trio in evs:
        for e in trio:
            e.record(stream)
    torch.cuda.synchronize()
    for trio in evs:
        kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
                p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], stream=stream,
                workspace=ws, stage_events=trio)
    torch.cuda.synchronize()
    kernel_ms = {"kda_prep_kernel": statistics.mean(t[0].elapsed_time(t[1]) for t in evs),
                 "kda_recur_kernel": statistics.mean(t[1].elapsed_time(t[2]) for t in evs)}
    # the pages' own precision choices as measurement variants of the same call (kda_fwd_ws_variant)
    variant_ms = {}
    for name, bits in (("bf16_state", 1), ("neumann_inverse", 2), ("both", 3)):
        def vstep():
            kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
                    p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], stream=stream,
                    workspace=ws, variant=bits)
        for _ in range(3):
            vstep()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record(stream)
        for _ in range(n_prof):
            vstep()
        v1.record(stream)
        torch.cuda.synchronize()
        variant_ms[name] = v0.elapsed_time(v1) / n_prof
    del ws
    if args.kernel_only:
        if rank == 0:
            print(json.dumps({"kernel_only": True, "ms_per_step": ms_step, "T": p.T, "H": p.H,
                              "pieces_per_step": pieces_per_step(p), "scan_groups_per_step": scan_groups_per_step(p),
                              "launches_per_step": launches_per_step(p),
                              "algorithmic_bytes_per_launch": algorithmic_bytes(p), "kernel_ms": kernel_ms,
                              "variant_ms": variant_ms}),
                  flush=True)
        return

    # end to end through the C-ABI host-buffer entry point (kda_fwd_host): pinned host inputs in, host
    # results out; the call copies, computes and copies back before it returns
    has_init = p.initial_state is not None
    pin = lambda t: t.cpu().pin_memory()
    host = dict(q=pin(dev["q"]), k=pin(dev["k"]), v=pin(dev["v"]), g=pin(dev["g"]), beta=pin(dev["beta"]),
                A_log=pin(dev["A_log"]), dt_bias=pin(dev["dt_bias"]),
                init=pin(dev["init"]) if has_init else None, cu=pin(dev["cu"]) if dev["cu"] is not None else None)
    out_h = torch.empty(p.q.shape, dtype=torch.bfloat16).pin_memory()
    fin_h = (torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"]).pin_memory()
             if (p.want_final and dev["sdt"] is not None) else None)

    def e2e_step():
        kda_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], p.scale, out_h, host["A_log"],
                     host["dt_bias"], p.lower_bound, initial_state=host["init"], final_state=fin_h,
                     cu_seqlens=host["cu"])

    for _ in range(3):   # the first call of a process also reserves the pool's memory
        e2e_step()
    n_e2e = max(3, min(args.steps, 50))   # a mean over 50 calls: one slow call moves it little
    if world > 1:
        dist.barrier()
    t_e0 = time.perf_counter()
    e2e_calls = []
    for _ in range(n_e2e):
        t_c = time.perf_counter()
        e2e_step()
        e2e_calls.append((time.perf_counter() - t_c) * 1e3)
    e2e_ms = max_over_ranks((time.perf_counter() - t_e0) * 1e3 / n_e2e, world, "cuda")
    e2e_calls.sort()
    e2e_median = e2e_calls[len(e2e_calls) // 2]
    h2d_bytes = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h_bytes = sum(t.numel() * t.element_size() for t in (out_h, fin_h) if t is not None)
    link = measure_link(h2d_bytes, d2h_bytes) if rank == 0 else None

    if rank != 0:
        return
    th = p.token_heads() * world   # replicas: every rank processes the whole workload
    hbm, tc, peak_src = peaks()
    abytes = algorithmic_bytes(p)
    aflops = algorithmic_flops(p)
    kbytes = kernel_bytes(p)
    kalg = kernel_algorithmic_bytes(p)
    kernels = {}
    for name, kms in kernel_ms.items():
        ach = kbytes[name] / (kms * 1e-3) / 1e9
        ach_alg = kalg[name] / (kms * 1e-3) / 1e9
        kernels[name] = {"ms": kms, "design_bytes_per_launch": kbytes[name], "design_achieved": ach,
                         "design_frac": ach / hbm, "algorithmic_bytes_per_launch": kalg[name],
                         "achieved": ach_alg, "frac": ach_alg / hbm,
                         "traffic": measured_traffic(name, idx if args.T is None else f"{idx}@T{args.T}")}
    dom = max(kernel_ms, key=kernel_ms.get)
    t_hbm = abytes / (hbm * 1e9)
    t_tc = aflops / (tc * 1e12)
    path_ach = abytes / (ms_step * 1e-3) / 1e9
    traffic = [kernels[k]["traffic"] for k in kernels]
    line = {
        "metric": METRIC, "value": aggregate_throughput(p.token_heads(), world, ms_step), "unit": UNIT,
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (th / world) / (ms_step * 1e-3) / PAGES_GB200_TOKHEADS_PER_S,
        "dtype": "bf16", "precision": "bf16 inputs/outputs; tf32 and fp16 tensor-core operands; fp32 accumulation "
                                      "and fp32 state master",
        "data": "synthetic", "config": workload_config(p, idx),
        # the whole call against its roofline: algorithmic bytes (q, k, v, g, beta in, out, states,
        # parameters) over the measured time, against the measured HBM copy bandwidth; the FLOP bound is
        # the algorithmic FLOPs over the measured bf16 dense peak, and the slower of the two is the bound
        "roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": path_ach, "peak": hbm,
                     "unit": "GB/s", "frac": path_ach / hbm,
                     "traffic": None if any(t is None for t in traffic) else float(sum(traffic)),
                     "traffic_note": "sum over the step's kernels of ncu dram__bytes_read.sum + "
                                     "dram__bytes_write.sum per launch (profiles/)",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                     "algorithmic_bytes_per_step": abytes, "algorithmic_flops_per_step": aflops,
                     "tensor_peak_tflops": tc, "t_hbm_ms": t_hbm * 1e3, "t_tensor_ms": t_tc * 1e3,
                     "roofline_ms": max(t_hbm, t_tc) * 1e3,
                     "dominant_kernel": {"name": dom, "ms": kernel_ms[dom],
                                         "algorithmic_bytes_per_launch": kalg[dom],
                                         "achieved": kernels[dom]["achieved"], "frac": kernels[dom]["frac"]},
                     "kernels": kernels},
        "cpu_baseline": cpu_baseline(p, idx),
        "e2e": {"value": aggregate_throughput(p.token_heads(), world, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "entry": "kda_fwd_host (C ABI, pinned host buffers, host wall clock)",
                # the host link as the bound of the end-to-end call: one plain copy of the step's input bytes
                # and one of its output bytes (pinned memory, CUDA events), alone and both directions at once;
                # the floor is the slower of the concurrent pair, frac = floor / e2e time
                "link": link, "link_frac": None if link is None else link["floor_ms"] / e2e_ms,
                # the per-call spread (rank 0): a mean well above the median marks slow single calls
                "median_call_ms": e2e_median, "max_call_ms": e2e_calls[-1]},
        "clocks": sampler.summary(),
        "variants_ms_per_step": variant_ms,
        "pieces_per_step": pieces_per_step(p),
        "scan_groups_per_step": scan_groups_per_step(p),
        "gpu_launches": args.steps * launches_per_step(p),
        "decode": measure_decode(stream) if world == 1 else None,
    }
    print(json.dumps(line), flush=True)


def pieces_per_step(p):
    """Pieces along T in which one call runs this workload on the current device (kda_fwd_pieces)."""
    from gated_delta_rule_23_gb300 import _native
    return int(_native.load().kda_fwd_pieces(p.N, p.T, p.H, int(p.cu_seqlens is not None)))


def scan_groups_per_step(p):
    """Groups of the chunk-transition scan along T for this workload (kda_fwd_scan_groups; 1: no scan)."""
    from gated_delta_rule_23_gb300 import _native
    return int(_native.load().kda_fwd_scan_groups(p.N, p.T, p.H, int(p.cu_seqlens is not None)))


def launches_per_step(p):
    """Kernels one call launches: the varlen plan, prep and recurrence; a decode step's single kernel; with
    the scan along T, prep, the groups' transitions, their start states and the grouped recurrence; or, in
    pieces, a prep and a recurrence launch per piece; plus, for the scan and the pieces, the bf16 state
    conversions into and out of the fp32 states they pass on."""
    if p.cu_seqlens is not None:
        return 3
    if 1 <= p.T <= 16:   # the token-recurrent kernels
        return 1
    conv = int(p.state_dtype == STATE_BF16) * (int(p.initial_state is not None) + int(p.want_final))
    if scan_groups_per_step(p) > 1:
        return 4 + conv
    pieces = pieces_per_step(p)
    if pieces > 1:
        return 2 * pieces + conv
    return 2


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, help="0-4; 2 = T=8192 H=96 fixed length")
    ap.add_argument("--T", type=int, default=None,
                    help="profiling aid: shorten a fixed-length workload to T tokens (not a bench line)")
    ap.add_argument("--shape", default=None,
                    help="profiling aid: T:H, a fixed-length problem of T tokens and H heads (B = 1) with workload 1's "
                         "value distributions, no initial state and an fp32 final state (not a bench line)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="profiling aid: time only the device launches (no e2e, CPU baseline or clock sampling)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode step (token-recurrent entry point, N=256 x T=1, H=96) and print "
                         "its measurement")
    ap.add_argument("--decode-N", type=int, default=DECODE_N, help="sequences of the --decode-only step")
    ap.add_argument("--decode-T", type=int, default=1, help="tokens per sequence of the --decode-only step")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, make_workload(args.workload), args.workload, rank)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.decode_only:
        if rank == 0:
            print(json.dumps(measure_decode(torch.cuda.current_stream(), steps=args.steps, warmup=args.warmup,
                                            n_seq=args.decode_N, T=args.decode_T)), flush=True)
        return
    p = make_workload(args.workload)
    if args.shape is not None:
        if not args.kernel_only:
            raise SystemExit("--shape is a profiling aid: use it with --kernel-only")
        from gated_delta_rule_23_gb300.inputs import make_problem
        T_, H_ = (int(x) for x in args.shape.split(":"))
        p = make_problem(B=1, T=T_, H=H_, seed=1, state_dtype=STATE_FP32, with_initial=False,
                         name=f"fixed-length T={T_} H={H_}")
    if args.T is not None:
        if p.cu_seqlens is not None:
            raise SystemExit("--T applies to fixed-length workloads only")
        p = dataclasses.replace(p, q=p.q[:, :args.T].copy(), k=p.k[:, :args.T].copy(), v=p.v[:, :args.T].copy(),
                                g=p.g[:, :args.T].copy(), beta=p.beta[:, :args.T].copy())
    run_ours(args, p, args.workload, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
