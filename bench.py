#!/usr/bin/env python3
"""Benchmark of the gated attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one gated_sdpa_fwd call on the headline prefill workload
(bf16, B=2, L=2048, d_model=2048, 16 heads of 128, causal, elementwise gate,
first-token share on): the gate GEMM sigma(X W_g) (its own kernel), then the
attention kernel -- head map and schedule, S = QK^T, online softmax, PV, the
gate-multiply epilogue -- and the first-token share.
The same run also times the decode workload (bf16, 64 single-query rows
against an 8192-token cache, GQA 32/8, elementwise gate) and reports it under
"decode" in GB/s, since the metric names both; the other configurations of
the metric (GQA headwise L4096, long-context GQA headwise L32768 with
sink-like keys, the float32 parity case) under "configs"; the layer as
unfused torch GPU ops under "unfused_context_ms" (context only); and, last in
the line, a compact "summary" of every configuration's time and fraction of
the measured peak.

Timing: W untimed warm-up steps, then exactly K back-to-back steps bracketed
by a barrier and a device synchronise and timed with one pair of CUDA events
on the stream the kernels run on. The prefill inputs (92 MB) fit in the
129 MB L2, so the steps rotate through enough copies of the inputs (>= 2x L2
in total) that no step finds its inputs in L2. value = FLOPs of all steps on
all ranks / the slowest rank's time. Under torchrun every rank runs its own
replica (no collective on the data path): scaling is weak.

--impl reference times the float64 CPU oracle (the reference arm of this
build) on the host cores, on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gated causal attention fwd TFLOP/s (bf16) and decode HBM GB/s, % of roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16_mha_elementwise_L2048")
    ap.add_argument("--decode-workload", default="bf16_decode_gqa_elementwise_Lk8192")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the GQA, long-context and float32 configurations")
    ap.add_argument("--no-unfused", action="store_true", help="skip the unfused torch context leg")
    ap.add_argument("--profile-backward", action="store_true",
                    help="with --profile-workload: the training forward once, then --profile-calls backward calls")
    ap.add_argument("--decode-steps", type=int, default=0, help="0: same as --steps, capped at 200")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: min(--steps, 50)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", default="", help="comma-separated workloads to time as extra lines on stderr")
    ap.add_argument("--profile-layer", action="store_true",
                    help="with --profile-workload: --profile-calls calls of the whole layer (projection, attention, W_O)")
    ap.add_argument("--profile-workload", default="",
                    help="for profilers: only run --profile-calls untimed calls of this workload and exit")
    ap.add_argument("--profile-calls", type=int, default=3)
    ap.add_argument("--profile-gate", default="", help="override the profiled workload's gate (none/headwise/elementwise)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self, backend):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.torch = torch
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64,
                              device="cuda" if self.pg.get_backend() == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ helpers

def row_flops(w, rows):
    """Algorithmic FLOPs of the listed (b, i) query rows (all heads)."""
    off = w.L_k - w.L_q
    n = 0
    for _, i in rows:
        keys = (off + i + 1) if w.causal else w.L_k
        n += 4 * w.H_q * w.d_k * keys + 2 * w.d_model * w.gate_cols
    return n


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def captured_traffic(profile_name, sources):
    """dram bytes per launch from a committed ncu summary in profiles/, or None
    when the kernel's sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, "gated_softmax_attention_gb300", "csrc", f), "rb").read())
    fields = dict(line.split(":", 1) for line in open(path) if line.startswith(("source_sha256:", "dram_bytes_per_launch:")))
    if fields.get("source_sha256", "").split()[0:1] != [h.hexdigest()[:16]]:
        return None
    return int(fields["dram_bytes_per_launch"].strip())


def oracle_cpu_baseline(w, inputs, seconds, seed=0):
    """Time the float64 oracle on a bounded, seeded row sample of workload w."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    all_rows = [(b, i) for b in range(w.B) for i in range(w.L_q)]
    cal = [all_rows[k] for k in rng.choice(len(all_rows), size=min(64, len(all_rows)), replace=False)]
    t0 = time.perf_counter()
    oracle.gated_sdpa(inputs["X"], inputs["Q"], inputs["K"], inputs["V"], inputs["W_g"], gate=w.gate,
                      causal=w.causal, rows=cal)
    dt = time.perf_counter() - t0
    rate = row_flops(w, cal) / max(dt, 1e-9)                     # FLOP/s
    per_row = row_flops(w, all_rows) / len(all_rows)
    n = int(min(len(all_rows), max(64, seconds * rate / per_row)))
    rows = [all_rows[k] for k in rng.choice(len(all_rows), size=n, replace=False)]
    t0 = time.perf_counter()
    oracle.gated_sdpa(inputs["X"], inputs["Q"], inputs["K"], inputs["V"], inputs["W_g"], gate=w.gate,
                      causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    return {"value": row_flops(w, rows) / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{n} of {len(all_rows)} query rows (all {w.H_q} heads each), uniform over (b, i), seed {seed}"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms, with timestamps
    so that only samples taken inside the timed region are summarised."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = ["-i", str(self.dev)]
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.4)  # nvidia-smi start-up
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, windows):
        """windows: list of (t0, t1) time.time() intervals, tried in order until one holds >= 3 samples."""
        import datetime
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.f.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for label, (t0, t1) in windows:
            sel = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
            if len(sel) >= 3 or label == windows[-1][0]:
                break
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0, "window": label}
        reasons = sorted({names[k] for *_, r in sel for k in range(4) if r[k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "window": label}


# ------------------------------------------------------------------ our arm

L2_BYTES = 129 * 1024 * 1024


def n_rotating_sets(bytes_per_set):
    """Input copies to cycle through so that the total is at least 2x L2."""
    return max(1, -(-2 * L2_BYTES // max(1, bytes_per_set)))


def time_calls(torch, call, K, W, stream):
    """Average milliseconds of call(k) over K back-to-back steps (one event pair)."""
    for k in range(W):
        call(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(K):
        call(k)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def capture_steps(torch, call, R):
    """CUDA graphs of the step (no host launch overhead between steps): `group`
    holds R consecutive steps, one per rotating input set, so that the kernels
    of consecutive steps follow each other inside one graph; `single[k]` holds
    step k alone, for step counts that are not a multiple of R."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for k in range(R):
            call(k)          # warm-up outside capture: first-call setup of the library
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    single = []
    for k in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(k)
        single.append(g)
    group = torch.cuda.CUDAGraph()
    with torch.cuda.graph(group):
        for k in range(R):
            call(k)
    torch.cuda.synchronize()
    return single, group


def replay_steps(graphs, K):
    """Run exactly K steps from the captured graphs."""
    single, group = graphs
    R = len(single)
    for _ in range(K // R):
        group.replay()
    for k in range(K % R):
        single[k].replay()


def time_steps(torch, graphs, K, W, stream):
    """Average milliseconds per step over K steps replayed back to back (one event pair)."""
    replay_steps(graphs, W)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay_steps(graphs, K)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def run_ours(args, d: Dist):
    import torch
    from gated_softmax_attention_gb300 import binding as gb
    from gated_softmax_attention_gb300 import build as gbuild
    from gated_softmax_attention_gb300.workloads import WORKLOADS, make_inputs

    if d.rank == 0 or not os.path.exists(gbuild.LIB):
        gbuild.build()
    d.barrier()
    gb.load()
    torch.cuda.set_device(d.local)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    K, W = args.steps, args.warmup

    # ---- CPU baseline first (before any long GPU work), rank 0 only
    w = WORKLOADS[args.workload]
    host = make_inputs(w)
    cpu_base = None
    if d.rank == 0 and not args.no_cpu_baseline:
        cpu_base = oracle_cpu_baseline(w, host, args.cpu_seconds)

    dev0 = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    in_bytes = sum(v.numel() * v.element_size() for v in dev0.values() if v is not None)
    R = n_rotating_sets(in_bytes)
    sets = [dev0] + [{k: (v.clone() if v is not None else None) for k, v in dev0.items()} for _ in range(R - 1)]
    outs = [torch.empty_like(dev0["Q"]) for _ in range(R)]
    sink = torch.empty((w.B, w.H_q), dtype=torch.float32, device="cuda")
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate, True, gb.BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def call(k, gate=w.gate, want_sink=True):
        dv = sets[k % R]
        gb.gated_sdpa_fwd(dv["X"], dv["Q"], dv["K"], dv["V"], dv["W_g"], gate=gate, causal=w.causal,
                          out=outs[k % R], sink=sink if want_sink else None, workspace=ws)

    g_main = capture_steps(torch, call, R)
    g_kern = capture_steps(torch, lambda k: call(k, want_sink=False), R)
    g_none = capture_steps(torch, lambda k: call(k, gate="none", want_sink=False), R)

    # ---- headline: K timed back-to-back steps
    replay_steps(g_main, W)
    torch.cuda.synchronize()
    d.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(d.local) as clk:
        t_start = time.time()
        wall0 = time.perf_counter()
        e0.record(stream)
        replay_steps(g_main, K)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        t_end = time.time()
        d.barrier()
        torch.cuda.synchronize()
        # the gated call without the first-token share (gate GEMM + attention kernel),
        # and the attention kernel alone (the same call without a gate), same clocks window
        kern_avg = time_steps(torch, g_kern, max(K, 200), W, stream)
        none_avg = time_steps(torch, g_none, max(K, 200), W, stream)
        t_end2 = time.time()
    clocks = clk.summary([("timed region", (t_start, t_end)),
                          ("timed region + kernel re-timing", (t_start, t_end2))])
    st = gb.check_device_error(stream)
    if st != gb.OK:
        raise RuntimeError(f"device error during the timed region: {gb.status_string(st)}")
    local_s = e0.elapsed_time(e1) / 1e3
    max_s = d.max(local_s)
    flops = w.flops()
    value = flops * K * d.world / max_s / 1e12

    # Dominant kernel: the attention kernel (the larger share of the step). In the
    # gated call it starts early under programmatic dependent launch and overlaps
    # the gate GEMM, so its own duration is taken from the call without a gate
    # (the same kernel minus the gate multiply), against the attention FLOPs.
    achieved = w.attn_flops() / (none_avg / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": peaks["source"] + " burst bf16 (cuBLAS)",
                "traffic": captured_traffic("prefill_kernel_bf16_mha_none_L2048.md",
                                            ["prefill_sm103.cu", "sm103_ptx.cuh", "gsdpa_internal.h", "gate_fn.cuh"]),
                "kernel": "prefill_kernel<128,0> (attention kernel; gate-free call)", "kernel_ms": round(none_avg, 4),
                "gated_call_ms": round(kern_avg, 4),
                "gated_call_tflops": round(flops / (kern_avg / 1e3) / 1e12, 2)}
    O = outs[0]
    dev = dev0

    # ---- end to end: pinned host inputs -> device -> call -> O back to the host,
    # every step, pipelined over two device buffer sets: step k's host-to-device
    # copies (their own stream) overlap step k-1's call (the launching stream) and
    # its device-to-host copies (a third stream)
    E = args.e2e_steps or min(K, 50)
    pinned = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
    d2h = O.numel() * O.element_size() + sink.numel() * sink.element_size()
    io = [dict(dev, O=O, sink=sink),
          dict({k: (torch.empty_like(v) if v is not None else None) for k, v in dev.items()},
               O=torch.empty_like(O), sink=torch.empty_like(sink))]
    for b in io:
        b["O_host"] = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
        b["sink_host"] = torch.empty(sink.shape, dtype=sink.dtype, pin_memory=True)
        b["ev"] = {n: torch.cuda.Event() for n in ("in", "done", "out")}
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step(k):
        b = io[k % 2]
        h2d_s.wait_event(b["ev"]["done"])          # the call two steps back has read these inputs
        with torch.cuda.stream(h2d_s):
            for n, v in pinned.items():
                if v is not None:
                    b[n].copy_(v, non_blocking=True)
        b["ev"]["in"].record(h2d_s)
        stream.wait_event(b["ev"]["in"])
        stream.wait_event(b["ev"]["out"])          # the copy two steps back has read this O
        gb.gated_sdpa_fwd(b["X"], b["Q"], b["K"], b["V"], b["W_g"], gate=w.gate, causal=w.causal,
                          out=b["O"], sink=b["sink"], workspace=ws, stream=stream)
        b["ev"]["done"].record(stream)
        d2h_s.wait_event(b["ev"]["done"])
        with torch.cuda.stream(d2h_s):
            b["O_host"].copy_(b["O"], non_blocking=True)
            b["sink_host"].copy_(b["sink"], non_blocking=True)
        b["ev"]["out"].record(d2h_s)

    for k in range(min(W, 3)):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    for k in range(E):
        e2e_step(k)
    stream.wait_stream(d2h_s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / E
    e2e_s = d.max(e2e_ms * E / 1e3)
    e2e = {"value": round(flops * E * d.world / e2e_s / 1e12, 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
           "pipelining": "two buffer sets; host-to-device, call and device-to-host copies on three streams"}

    launches_per_step = 2  # gate GEMM (also resets the per-call state) + attention kernel (also sums the share)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": d.world, "steps": K,
        "warmup": W, "ms_per_step": round(max_s * 1e3 / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) X/Q/K/V, W_g ~ N(0, 0.02^2), rounded once to bf16",
        "config": {"workload": w.name, "B": w.B, "L_q": w.L_q, "L_k": w.L_k, "d_model": w.d_model, "H_q": w.H_q,
                   "H_kv": w.H_kv, "d_k": w.d_k, "gate": w.gate, "causal": w.causal, "first_token_share": True,
                   "l2": f"inputs larger than L2: {R} rotating copies of the {in_bytes / 1e6:.0f} MB inputs",
                   "parallelism": f"replicas x{d.world}", "flops_per_step": flops,
                   "launch": f"CUDA graphs of {R} consecutive steps"},
        "clocks": clocks, "wall_s_timed_region": round(wall, 4),
        "e2e": e2e, "gpu_launches": launches_per_step * K,
        "roofline": roofline,
        "attention_only_tflops": round(w.attn_flops() / (none_avg / 1e3) / 1e12, 2),
        "gated_vs_ungated_time_ratio": round(kern_avg / none_avg, 4),
        "cpu_baseline": cpu_base,
    }

    # ---- decode leg
    if not args.no_decode:
        out["decode"] = run_decode(args, d, torch, gb, WORKLOADS[args.decode_workload], make_inputs, stream, peaks)
        out["gpu_launches"] += out["decode"]["gpu_launches"]

    # ---- backward leg (the layer's gradients for a training step), context beside the metric
    if not args.no_backward:
        out["backward"] = run_backward(args, d, torch, gb, w, host, stream, peaks)
        out["gpu_launches"] += out["backward"]["gpu_launches"]

    # ---- gate variants on the headline shape (context beside the metric)
    if not args.no_variants:
        out["variants"] = run_variants(args, d, torch, gb, w, host, stream, peaks)
        out["gpu_launches"] += out["variants"]["gpu_launches"]

    # ---- the whole layer (input projection, attention, output projection)
    if not args.no_layer:
        out["layer"] = run_layer(args, d, torch, gb, w, stream, peaks)
        out["gpu_launches"] += out["layer"]["gpu_launches"]
        # and on the two GQA configurations' shapes (headwise gate)
        out["layer_configs"] = {}
        for name in ("bf16_gqa_headwise_L4096", "bf16_gqa_headwise_sink_L32768"):
            out["layer_configs"][name] = run_layer(args, d, torch, gb, WORKLOADS[name], stream, peaks)
            out["gpu_launches"] += out["layer_configs"][name]["gpu_launches"]

    # ---- the other configurations of the metric: GQA headwise L4096 and the
    # long-context GQA headwise L32768 with sink-like keys (whole call with the
    # first-token share, and the attention kernel alone via the gate-free call),
    # and the float32 parity configuration (FFMA path)
    if not args.no_configs:
        out["configs"] = {}
        for name in ("bf16_gqa_headwise_L4096", "bf16_gqa_headwise_sink_L32768", "f32_mha_elementwise_L128"):
            out["configs"][name] = run_config(args, d, torch, gb, WORKLOADS[name], make_inputs, stream, peaks)
            out["gpu_launches"] += out["configs"][name]["gpu_launches"]

    # ---- unfused GPU context (not the target): torch SDPA + X W_g + sigmoid-multiply
    if not args.no_unfused:
        out["unfused_context_ms"] = {
            name: run_unfused(torch, WORKLOADS[name], make_inputs, stream)
            for name in ("bf16_mha_elementwise_L2048", "bf16_gqa_headwise_L4096", "bf16_gqa_headwise_sink_L32768",
                         "bf16_decode_gqa_elementwise_Lk8192")}

    # ---- compact summary of every configuration, last in the line (so that a
    # reader that keeps only the end of the line still sees every number)
    pk = peaks["bf16_tflops"]
    summ = {"bf16_mha_elementwise_L2048": {
        "call_ms": out["ms_per_step"], "tflops": out["value"], "frac": round(out["value"] / pk, 4),
        "attn_kernel_ms": roofline["kernel_ms"], "attn_frac": roofline["frac"]}}
    for name, c in out.get("configs", {}).items():
        summ[name] = {k: c[k] for k in ("call_ms", "tflops", "frac", "attn_kernel_ms", "attn_frac") if k in c}
    if "decode" in out:
        dec = out["decode"]
        summ[dec["workload"]] = {"call_ms": dec["ms_per_step"], "gbs": dec["value"],
                                 "frac": dec["roofline"]["frac"]}
    if "backward" in out:
        summ["backward_L2048"] = {"ms": out["backward"]["ms_per_step"], "frac": out["backward"]["roofline"]["frac"]}
    if "layer" in out:
        summ["layer_L2048"] = {"ms": out["layer"]["ms_per_step"], "frac": out["layer"]["roofline"]["frac"]}
        for name, c in out.get("layer_configs", {}).items():
            summ["layer_" + name.split("_")[-1]] = {"ms": c["ms_per_step"], "frac": c["roofline"]["frac"]}
    if "unfused_context_ms" in out:
        summ["unfused_torch_ms"] = out["unfused_context_ms"]
    out["summary"] = summ

    # ---- extra workloads (context only), one stderr line each
    for name in [x for x in args.extra.split(",") if x]:
        wx = WORKLOADS[name]
        hx = {k: (v.cuda() if v is not None else None) for k, v in make_inputs(wx).items()}
        Ox = torch.empty_like(hx["Q"])
        ms = time_calls(torch, lambda k: gb.gated_sdpa_fwd(hx["X"], hx["Q"], hx["K"], hx["V"], hx["W_g"],
                                                            gate=wx.gate, causal=wx.causal, out=Ox, stream=stream),
                        max(3, min(K, 20)), 2, stream)
        print(json.dumps({"extra": name, "ms": round(ms, 4), "TFLOP/s": round(wx.flops() / ms / 1e9, 2),
                          "frac_of_bf16_peak": round(wx.flops() / ms / 1e9 / peaks["bf16_tflops"], 4)}),
              file=sys.stderr)
        del hx, Ox
    return out


def run_config(args, d, torch, gb, w, make_inputs, stream, peaks):
    """One configuration of the metric, timed like the headline: CUDA graphs of
    consecutive calls (inputs rotated past L2 where they fit in it), the call
    with the first-token share and, for bf16, the same call without a gate
    (the attention kernel alone, against the attention FLOPs)."""
    host = make_inputs(w)
    dev0 = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    in_bytes = sum(v.numel() * v.element_size() for v in dev0.values() if v is not None)
    # (the float32 parity case's 1 MB inputs stay L2-resident: a few copies, not the 2x-L2 rotation)
    R = n_rotating_sets(in_bytes) if w.dtype == "bf16" else 4
    sets = [dev0] + [{k: (v.clone() if v is not None else None) for k, v in dev0.items()} for _ in range(R - 1)]
    outs = [torch.empty_like(dev0["Q"]) for _ in range(R)]
    sink = torch.empty((w.B, w.H_q), dtype=torch.float32, device="cuda")
    dtype = gb.BF16 if w.dtype == "bf16" else gb.F32
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate, True, dtype)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def call(k, gate=w.gate, want_sink=True):
        dv = sets[k % R]
        gb.gated_sdpa_fwd(dv["X"], dv["Q"], dv["K"], dv["V"], dv["W_g"] if gate != "none" else None, gate=gate,
                          causal=w.causal, out=outs[k % R], sink=sink if want_sink else None, workspace=ws)

    # about 50 ms of calls per timing (at least 5)
    K = max(5, min(args.steps, int(0.05 / max(w.flops() / 1.2e15, 1e-6))))
    d.barrier()
    ms = time_steps(torch, capture_steps(torch, call, R), K, args.warmup, stream)
    res = {"workload": w.name, "dtype": w.dtype, "call_ms": round(ms, 5), "steps": K,
           "tflops": round(w.flops() / ms / 1e9, 2), "flops_per_call": w.flops()}
    launches = K * (2 if w.dtype == "bf16" else 2)
    if w.dtype == "bf16":
        res["frac"] = round(w.flops() / ms / 1e9 / peaks["bf16_tflops"], 4)
        ms_none = time_steps(torch, capture_steps(torch, lambda k: call(k, gate="none", want_sink=False), R), K,
                             args.warmup, stream)
        res["attn_kernel_ms"] = round(ms_none, 5)
        res["attn_tflops"] = round(w.attn_flops() / ms_none / 1e9, 2)
        res["attn_frac"] = round(w.attn_flops() / ms_none / 1e9 / peaks["bf16_tflops"], 4)
        res["gated_vs_ungated_time_ratio"] = round(ms / ms_none, 4)
        launches += 2 * K
    else:
        res["note"] = "float32 parity configuration (FFMA path, latency-bound at this size); context only"
    res["gpu_launches"] = launches
    res["l2"] = (f"{R} rotating copies of the {in_bytes / 1e6:.0f} MB inputs" +
                 ("" if w.dtype == "bf16" else " (L2-resident)"))
    st = gb.check_device_error(stream)
    if st != gb.OK:
        raise RuntimeError(f"device error in {w.name}: {gb.status_string(st)}")
    del sets, outs, ws, dev0
    torch.cuda.empty_cache()
    return res


def run_unfused(torch, w, make_inputs, stream):
    """Context only (not the target): the gated layer as unfused torch GPU ops --
    scaled_dot_product_attention on [B, H, L, d] views, sigmoid(X W_g) as its
    own GEMM, and the gate multiply -- milliseconds per call (eager, events)."""
    import torch.nn.functional as F
    dev = {k: (v.cuda() if v is not None else None) for k, v in make_inputs(w).items()}
    q, k, v = (dev[n].transpose(1, 2) for n in ("Q", "K", "V"))
    # a single query row sees the whole cache (bottom-right alignment); torch's
    # causal mask is top-left, so the decode case runs unmasked
    causal = w.causal and w.L_q == w.L_k
    gqa = w.H_q != w.H_kv

    def call(_):
        o = F.scaled_dot_product_attention(q, k, v, is_causal=causal, enable_gqa=gqa).transpose(1, 2)
        g = torch.sigmoid(dev["X"] @ dev["W_g"])
        return o * g.view(w.B, w.L_q, w.H_q, -1)

    K = max(3, min(50, int(0.05 / max(w.flops() / 4e14, 1e-6))))
    ms = time_calls(torch, call, K, 3, stream)
    del dev, q, k, v
    torch.cuda.empty_cache()
    return round(ms, 4)


def backward_flops(w):
    """Algorithmic FLOPs of the backward: five attention products of the
    forward's size (S, dP, dV, dK, dQ; 2.5x the forward's attention FLOPs) and
    the gate's two (dW_g = X^T dGl, dX = dGl W_g^T). Recomputation is not counted."""
    return int(2.5 * w.attn_flops()) + 2 * (w.flops() - w.attn_flops())


def run_backward(args, d, torch, gb, w, host, stream, peaks):
    """The backward call on the headline workload: graph replays of R calls,
    each reading its own copy of the inputs (inputs larger than L2 in total).
    The elementwise gate's values come from the training forward
    (gated_sdpa_fwd_train_save_gate -> gated_sdpa_bwd_saved_gate); the call
    that recomputes them (gated_sdpa_bwd) is timed beside it."""
    dev = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    g = torch.Generator().manual_seed(4242)
    dO = torch.randn(dev["Q"].shape, generator=g).to(torch.bfloat16).cuda()
    saved = w.gate == "elementwise"
    if saved:
        O, _, lse, G = gb.gated_sdpa_fwd_train_save_gate(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"],
                                                         causal=w.causal)
    else:
        O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                            causal=w.causal)
        G = None
    per_set = sum(v.numel() * v.element_size() for v in list(dev.values()) + [O, dO, lse, G] if v is not None)
    R = n_rotating_sets(per_set)
    sets = [dict(dev, O=O, dO=dO, lse=lse, G=G)]
    for _ in range(R - 1):
        sets.append({k: (v.clone() if v is not None else None) for k, v in sets[0].items()})
    need = gb.bwd_workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    K = max(3, min(args.steps, 100))

    def timed(use_saved):
        def call(k):
            st = sets[k % R]
            gb.gated_sdpa_bwd(st["X"], st["Q"], st["K"], st["V"], st["W_g"], st["O"], st["dO"], st["lse"],
                              gate=w.gate, causal=w.causal, workspace=ws, gate_saved=st["G"] if use_saved else None)

        graphs = capture_steps(torch, call, R)
        ms = time_steps(torch, graphs, K, min(args.warmup, 5), stream)
        st = gb.check_device_error(stream)
        if st != gb.OK:
            raise RuntimeError(f"device error in the backward leg: {gb.status_string(st)}")
        return ms

    ms = timed(saved)
    ms_recompute = timed(False) if saved else ms
    flops = backward_flops(w)
    tf = flops / (ms / 1e3) / 1e12
    kernels = (5 if saved else 6) if w.gate != "none" else 3
    return {"workload": w.name, "metric": "gated attention bwd TFLOP/s (bf16; algorithmic: 5 attention products "
                                          "+ 2 gate GEMMs)", "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5), "flops_per_step": flops, "steps": K,
            "gate": "saved by the training forward" if saved else "recomputed",
            "with_gate_recompute": {"ms_per_step": round(ms_recompute, 5),
                                    "tflops": round(flops / (ms_recompute / 1e3) / 1e12, 2)},
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                         "scope": "whole call (prep, dQ, dK/dV, dX and dW_g GEMMs; the gate's values saved by "
                                  "the training forward)" if saved else "whole call (gate recompute, prep, dQ, "
                                  "dK/dV, dX and dW_g GEMMs)"},
            "gpu_launches": kernels * K + ((6 * K) if saved else 0)}


VARIANTS = [("elementwise", "sigmoid_mul"), ("elementwise", "ns_sigmoid_mul"), ("elementwise", "sigmoid_add"),
            ("elementwise", "silu_add"), ("elementwise", "identity_add"), ("elementwise_shared", "sigmoid_mul"),
            ("headwise", "sigmoid_mul"), ("headwise_shared", "sigmoid_mul"), ("static", "sigmoid_mul"),
            ("elementwise_averaged", "sigmoid_mul"), ("headwise_averaged", "sigmoid_mul"),
            ("none", "sigmoid_mul"), ("none", "silu_self"), ("none", "rmsnorm")]


def run_variants(args, d, torch, gb, w, host, stream, peaks):
    """Every gate variant (gated_sdpa_fwd_variant) on the headline shape: graph
    replays of R calls over rotating input copies, like the headline step;
    time per call and algorithmic TFLOP/s (the attention, plus the gate GEMM
    where the gate reads X), and the ratio to the default gate's call."""
    from gated_softmax_attention_gb300.workloads import variant_weight
    dev = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    per_set = sum(v.numel() * v.element_size() for v in dev.values() if v is not None)
    R = n_rotating_sets(per_set)
    sets = [dev] + [{k: (v.clone() if v is not None else None) for k, v in dev.items()} for _ in range(R - 1)]
    O = torch.empty_like(dev["Q"])
    gen = torch.Generator().manual_seed(97)
    rows = w.B * w.L_q
    cols = {"elementwise": w.H_q * w.d_k, "headwise": w.H_q, "elementwise_shared": w.d_k, "headwise_shared": 1,
            "elementwise_averaged": w.H_q * w.d_k, "headwise_averaged": w.H_q}
    K = max(3, min(args.steps, 100))
    res, launches, base_ms = [], 0, None
    for gate, fn in VARIANTS:
        if gate in ("elementwise", "headwise") and gate == w.gate:
            W = [st["W_g"] for st in sets]
        elif gate == "headwise":
            W = [(torch.randn((w.d_model, w.H_q), generator=gen) * 0.02).to(torch.bfloat16).cuda()] * R
        else:
            W = [variant_weight(w, gate, fn, device="cuda")] * R
        need = gb.workspace_bytes_variant(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, gate, fn, False,
                                          gb.BF16)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        reads_x = gate not in ("none", "static")

        def call(k, gate=gate, fn=fn, W=W, ws=ws, reads_x=reads_x):
            st = sets[k % R]
            gb.gated_sdpa_fwd_variant(st["X"] if reads_x else None, st["Q"], st["K"], st["V"], W[k % R], gate=gate,
                                      gate_fn=fn, causal=w.causal, out=O, workspace=ws)

        graphs = capture_steps(torch, call, R)
        ms = time_steps(torch, graphs, K, min(args.warmup, 5), stream)
        st = gb.check_device_error(stream)
        if st != gb.OK:
            raise RuntimeError(f"device error in the variants leg ({gate}/{fn}): {gb.status_string(st)}")
        flops = w.attn_flops() + 2 * rows * w.d_model * cols.get(gate, 0)
        if base_ms is None:
            base_ms = ms
        # (a gate pass or the state-zeroing kernel, the averaging pass of the averaged gates, the attention)
        launches += (3 if gate.endswith("_averaged") else 2) * K
        res.append({"gate": gate, "gate_fn": fn, "ms_per_call": round(ms, 5),
                    "tflops": round(flops / (ms / 1e3) / 1e12, 2), "vs_default_call": round(ms / base_ms, 4)})
        del graphs, ws
    # the default gate with its fused statistics (gated_sdpa_fwd_stats: 20 bins, threshold 0.1)
    import ctypes
    stats = torch.empty(3 + 20, dtype=torch.int64, device="cuda")
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate, False, gb.BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def call_stats(k):
        st = sets[k % R]
        p = lambda t: ctypes.c_void_p(t.data_ptr())
        rc = gb.load().gated_sdpa_fwd_stats(p(st["X"]), p(st["Q"]), p(st["K"]), p(st["V"]), p(st["W_g"]), p(O), None,
                                            p(stats), 20, 0.1, w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k,
                                            gb.GATE_CODES[w.gate], int(w.causal), gb.BF16, p(ws), need,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if rc != gb.OK:
            raise gb.GsdpaError(rc, "gated_sdpa_fwd_stats")

    graphs = capture_steps(torch, call_stats, R)
    ms = time_steps(torch, graphs, K, min(args.warmup, 5), stream)
    st = gb.check_device_error(stream)
    if st != gb.OK:
        raise RuntimeError(f"device error in the variants leg (statistics): {gb.status_string(st)}")
    flops = w.attn_flops() + 2 * rows * w.d_model * cols.get(w.gate, 0)
    launches += 3 * K   # counter zeroing, gate GEMM with the counting pass, attention kernel
    res.append({"gate": w.gate, "gate_fn": "sigmoid_mul + statistics (20 bins)", "ms_per_call": round(ms, 5),
                "tflops": round(flops / (ms / 1e3) / 1e12, 2), "vs_default_call": round(ms / base_ms, 4)})
    del graphs, ws
    return {"workload": w.name, "scope": "whole call (gate pass + attention kernel), graph replays, inputs larger "
                                         "than L2 in total", "steps": K, "results": res, "gpu_launches": launches}


def run_layer(args, d, torch, gb, w, stream, peaks):
    """gated_attention_layer on workload w's shape: X W_in (Q, K, V and, for the
    elementwise gate, the gate in one GEMM; the headwise gate's logits in a
    pre-pass), the attention, O W_O -- graph replays over rotating X copies;
    algorithmic FLOPs of the products."""
    from gated_softmax_attention_gb300.workloads import layer_weights, make_inputs
    X0 = make_inputs(w)["X"].cuda()
    W_in, W_O = layer_weights(w, device="cuda")
    R = n_rotating_sets(X0.numel() * X0.element_size() * 3)   # (X, Q/K/V/gate, O, Y move per call)
    Xs = [X0] + [X0.clone() for _ in range(R - 1)]
    Y = torch.empty_like(X0)
    need = gb.layer_workspace_bytes(w.B, w.L_q, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def call(k):
        gb.gated_attention_layer(Xs[k % R], W_in, W_O, H_q=w.H_q, H_kv=w.H_kv, d_k=w.d_k, gate=w.gate,
                                 causal=w.causal, out=Y, workspace=ws)

    graphs = capture_steps(torch, call, R)
    rows = w.B * w.L_q
    proj = 2 * rows * w.d_model * W_in.shape[1]
    outp = 2 * rows * w.H_q * w.d_k * w.d_model
    flops = proj + w.attn_flops() + outp
    K = max(3, min(args.steps, 100, int(0.05 / (flops / 1.2e15))))   # about 50 ms of calls
    d.barrier()
    ms = time_steps(torch, graphs, K, min(args.warmup, 5), stream)
    st = gb.check_device_error(stream)
    if st != gb.OK:
        raise RuntimeError(f"device error in the layer leg: {gb.status_string(st)}")
    del graphs, Xs, ws
    torch.cuda.empty_cache()
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": w.name, "metric": "gated attention layer TFLOP/s (bf16; X [W_Q|W_K|W_V|W_g], attention, "
                                          "O W_O)", "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5), "flops_per_step": flops, "steps": K,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                         "scope": "whole call (projection GEMM, attention, output GEMM)"},
            "gpu_launches": (4 if w.gate == "headwise" else 3) * K}


def run_decode(args, d, torch, gb, w, make_inputs, stream, peaks):
    host = make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    O = torch.empty_like(dev["Q"])
    sink = torch.empty((w.B, w.H_q), dtype=torch.float32, device="cuda")
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate, True, gb.BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def step():
        gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=w.causal, out=O,
                          sink=sink, workspace=ws, stream=stream)

    K = args.decode_steps or min(args.steps, 200)
    # Each step is timed alone (an event pair around the call) after a read of
    # 2x L2 of other data: the 2 GiB K/V sweep alone would evict W_g (32 MiB)
    # too, but the read makes sure no input is in L2 when a call starts. (A read,
    # not a write: dirty lines would be written back inside the next call.)
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for _ in range(args.warmup):
        flush.max()
        step()
    torch.cuda.synchronize()
    d.barrier()
    for e0, e1 in evs:
        flush.max()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / K
    del flush
    st = gb.check_device_error(stream)
    if st != gb.OK:
        raise RuntimeError(f"device error in decode: {gb.status_string(st)}")
    s = d.max(ms * K / 1e3)
    nbytes = w.algorithmic_bytes()
    gbs = nbytes * K * d.world / s / 1e9
    per_gpu = nbytes / (s / K) / 1e9
    # e2e with the 2 GiB cache copied from pinned host memory every step
    E = min(args.e2e_steps or 10, 10)
    pinned = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    O_host = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)

    def e2e_step():
        for k, v in pinned.items():
            if v is not None:
                dev[k].copy_(v, non_blocking=True)
        step()
        O_host.copy_(O, non_blocking=True)

    e2e_ms = time_calls(torch, lambda k: e2e_step(), E, 2, stream)
    e2e_s = d.max(e2e_ms * E / 1e3)
    return {"workload": w.name, "value": round(gbs, 2), "unit": "GB/s", "steps": K,
            "l2": "L2 flushed before every call (read of 2x L2); each call timed alone",
            "ms_per_step": round(s * 1e3 / K, 5), "bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(per_gpu, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                         "peak_source": peaks["source"] + " STREAM-style copy",
                         "scope": "whole call (gate-logit pre-pass + decode kernel)",
                         "traffic_decode_kernel": captured_traffic("decode_kernel_bf16_decode_gqa_elementwise_Lk8192.md",
                                                                  ["decode_sm103.cu", "sm103_ptx.cuh", "gsdpa_internal.h", "gate_fn.cuh"])},
            "e2e": {"value": round(nbytes * E * d.world / e2e_s / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": O.numel() * O.element_size(), "steps": E},
            "gpu_launches": 2 * K}


# ------------------------------------------------------------------ reference arm (the CPU oracle)

def run_reference(args, d: Dist):
    from gated_softmax_attention_gb300.workloads import WORKLOADS, make_inputs
    import numpy as np
    import oracle
    w = WORKLOADS[args.workload]
    host = make_inputs(w)
    oracle.build()
    K, W = args.steps, args.warmup
    # each step: a seeded row sample sized so that all W + K steps take about two minutes
    budget = 120.0 / max(1, K + W)
    rng = np.random.default_rng(0)
    all_rows = [(b, i) for b in range(w.B) for i in range(w.L_q)]
    cal = [all_rows[k] for k in rng.choice(len(all_rows), size=32, replace=False)]
    t0 = time.perf_counter()
    oracle.gated_sdpa(host["X"], host["Q"], host["K"], host["V"], host["W_g"], gate=w.gate, causal=w.causal, rows=cal)
    rate = row_flops(w, cal) / (time.perf_counter() - t0)
    per_row = row_flops(w, all_rows) / len(all_rows)
    n = int(min(len(all_rows), max(8, budget * rate / per_row)))
    samples = [[all_rows[k] for k in rng.choice(len(all_rows), size=n, replace=False)] for _ in range(K + W)]
    for r in samples[:W]:
        oracle.gated_sdpa(host["X"], host["Q"], host["K"], host["V"], host["W_g"], gate=w.gate, causal=w.causal,
                          rows=r)
    total_s, total_f = 0.0, 0
    for r in samples[W:]:
        t0 = time.perf_counter()
        oracle.gated_sdpa(host["X"], host["Q"], host["K"], host["V"], host["W_g"], gate=w.gate, causal=w.causal,
                          rows=r)
        total_s += time.perf_counter() - t0
        total_f += row_flops(w, r)
    value = total_f / total_s / 1e12
    sample = f"{n} of {len(all_rows)} query rows per step (all {w.H_q} heads), uniform over (b, i), seed 0"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": d.world,
        "steps": K, "warmup": W, "ms_per_step": round(total_s * 1e3 / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) X/Q/K/V, W_g ~ N(0, 0.02^2), rounded once to bf16, upcast to f64",
        "config": {"workload": w.name, "B": w.B, "L_q": w.L_q, "L_k": w.L_k, "d_model": w.d_model, "H_q": w.H_q,
                   "H_kv": w.H_kv, "d_k": w.d_k, "gate": w.gate, "causal": w.causal, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_profile(args):
    """Untimed calls of one workload (1 GPU), for ncu: nothing else runs on the device."""
    import torch
    from gated_softmax_attention_gb300 import binding as gb
    from gated_softmax_attention_gb300 import build as gbuild
    from gated_softmax_attention_gb300.workloads import WORKLOADS, make_inputs
    gbuild.build()
    w = WORKLOADS[args.profile_workload]
    dev = {k: (v.cuda() if v is not None else None) for k, v in make_inputs(w).items()}
    O = torch.empty_like(dev["Q"])
    gate = args.profile_gate or w.gate
    if args.profile_backward:
        O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=gate,
                                            causal=w.causal)
        dO = torch.randn(dev["Q"].shape, generator=torch.Generator().manual_seed(4242)).to(torch.bfloat16).cuda()
        for _ in range(args.profile_calls):
            gb.gated_sdpa_bwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], O, dO, lse, gate=gate,
                              causal=w.causal)
    if args.profile_layer:
        from gated_softmax_attention_gb300.workloads import layer_weights
        W_in, W_O = layer_weights(w)
        X, W_in, W_O = dev["X"], W_in.cuda(), W_O.cuda()
        for _ in range(args.profile_calls):
            gb.gated_attention_layer(X, W_in, W_O, H_q=w.H_q, H_kv=w.H_kv, d_k=w.d_k, gate=w.gate, causal=w.causal)
    for _ in range(0 if (args.profile_backward or args.profile_layer) else args.profile_calls):
        gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=gate, causal=w.causal, out=O)
    st = gb.check_device_error()
    print(json.dumps({"profile_workload": w.name, "gate": gate, "calls": args.profile_calls,
                      "status": gb.status_string(st)}))
    if st != gb.OK:
        sys.exit(1)


def main():
    args = parse()
    if args.profile_workload:
        run_profile(args)
        return
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work or rendezvous
        if int(os.environ.get("RANK", "0")) != 0:
            return
        d = Dist.__new__(Dist)
        d.world = int(os.environ.get("WORLD_SIZE", "1"))
        print(json.dumps(run_reference(args, d)))
        return
    d = Dist("nccl")
    out = run_ours(args, d)
    if d.rank == 0:
        print(json.dumps(out))
    d.close()


if __name__ == "__main__":
    main()
