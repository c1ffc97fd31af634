"""Benchmark of the chunked gated-delta-rule prefill on GB300.

Default: N=1, the B=4, T=8192, nk=16, nv=32, dk=dv=128 workload with a carried
fp32 state (seeded synthetic inputs, resident in HBM before timing). One step
is one prefill call over the whole batch: every stage of the method (gates,
WY solve, state spine, output) for all 32,768 tokens x 32 heads.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_synth  # noqa: E402

METRIC = "GDN prefill tokens/s (nv=32,dk=dv=128,T=8192) and % of roofline, 1×GB300"
FLOP_PER_TOKEN_HEAD = 139_136  # W.S, Kd^T u, Q.S_c, KK^T, solve, QK^T, A.u (dk=dv=128, C=64)
# the spine kernel's own sources: its recorded DRAM traffic holds while these are unchanged
KERNEL_SOURCES = ["gated_delta_rule_17_gb300/csrc/gdn_prefill_kernel.cuh",
                  "gated_delta_rule_17_gb300/csrc/gdn_common.cuh", "gated_delta_rule_17_gb300/csrc/tc.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gdn_prefill_kernel_B4_T8192_nv32_full.md")
# Half the sequences of the B=4 workload: ~415 MB of I/O (above the 129 MB L2), 64
# spine CTAs, short enough for ncu's ~40-pass captures.
PROFILE_CASE = "B=2 T=8192 nk=16 nv=32 dk=dv=128 h0~N(0,0.02), seed 4242"



def algorithmic_bytes(p) -> int:
    """Each input read once, each output written once, state read and written."""
    tokens = p.tokens
    per_token = 2 * p.nk * p.dk * 2 + p.nv * p.dv * 2 * 2 + p.nv * 8
    return tokens * per_token + 2 * p.B * p.nv * p.dk * p.dv * 4


def spine_algorithmic_bytes(p) -> int:
    """The spine kernel's own I/O floor: q, k, v, g read once, out written once, the
    state read and written (beta is read only by the WY solve)."""
    return algorithmic_bytes(p) - p.tokens * p.nv * 4


def algorithmic_flops(p) -> int:
    return p.tokens * p.nv * FLOP_PER_TOKEN_HEAD


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was captured on
    the current kernel source and this workload (else None)."""
    try:
        with open(TRAFFIC_FILE) as fh:
            fields = dict(line.split(": ", 1) for line in fh.read().splitlines() if ": " in line
                          and line.split(": ", 1)[0] in ("traffic_bytes_per_launch", "kernel_sha", "workload"))
    except OSError:
        return None
    if fields.get("kernel_sha") != kernel_sha() or fields.get("workload") != workload:
        return None
    return int(fields["traffic_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile

        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class OracleSample:
    """A bounded sample of the workload for the fp64 CPU oracle, calibrated once
    so that one timed call takes about ``seconds`` on this host."""

    def __init__(self, p, seconds: float):
        import oracle

        self.oracle = oracle
        self.nv = p.nv
        self.cores = oracle.max_threads()
        probe = gdn_synth.make_problem(seed=1002, B=1, T=256, nk=p.nk, nv=p.nv, h0_std=0.02)
        t0 = time.perf_counter()
        oracle.token_loop(probe, heads=list(range(min(p.nv, max(2, self.cores)))))
        per_token_head = max(time.perf_counter() - t0, 1e-4) / (256 * min(p.nv, max(2, self.cores)))
        self.heads = list(range(p.nv))
        self.tokens = int(max(64, min(8192, seconds / (per_token_head * p.nv))))
        self.sub = gdn_synth.make_problem(seed=1002, B=1, T=self.tokens, nk=p.nk, nv=p.nv, h0_std=0.02)
        self.sample = (f"1 sequence x {self.tokens} tokens x all {p.nv} v-heads with the B=4 T=8192 "
                       f"workload's shapes and distributions; fp64 token loop on {self.cores} threads")

    def run(self):
        """Returns (tokens/s of the full nv-head workload, seconds)."""
        t0 = time.perf_counter()
        self.oracle.token_loop(self.sub, heads=self.heads)
        dt = time.perf_counter() - t0
        return self.tokens * len(self.heads) / dt / self.nv, dt


def run_reference(args, world, rank):
    if rank != 0:
        return
    p_shape = gdn_synth.config_problem(2, T=64)  # shapes and distributions only
    per_step = max(1.0, min(args.ref_seconds, 150.0 / (args.warmup + args.steps)))
    sample = OracleSample(p_shape, per_step)
    times, rates = [], []
    for i in range(args.warmup + args.steps):
        rate, dt = sample.run()
        if i >= args.warmup:
            times.append(dt)
            rates.append(rate)
    value = statistics.median(rates)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": gdn_synth.CONFIG_NAMES[2] + " (bounded oracle sample per step)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": sample.cores, "kind": "oracle",
                             "sample": sample.sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, world, rank, local):
    import torch

    import gated_delta_rule_17_gb300 as gdn
    from gated_delta_rule_17_gb300 import build as gbuild

    gbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.profile_case:
        p = gdn_synth.make_problem(seed=4242, B=2, T=8192, nk=16, nv=32, h0_std=0.02, qk_raw=args.qk_l2norm)
        workload = PROFILE_CASE
    else:
        p = gdn_synth.config_problem(args.config, qk_raw=args.qk_l2norm)
        workload = gdn_synth.CONFIG_NAMES[args.config]
    if args.qk_l2norm:
        workload += ", raw q/k rows normalised in the kernels (fused prologue)"
    from gdn_synth.device import DeviceProblem

    dp = DeviceProblem(p, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws = None
    ws_bytes = gdn.workspace_bytes(p.B, p.T, p.nv, p.varlen)
    # the profiling case mirrors the B=4 workload's single spine launch at half the
    # sequences, so it keeps the serial schedule
    if (args.no_segments or args.profile_case) and not p.varlen:
        ws = torch.empty(0, dtype=torch.uint8, device=dev)  # declines the segment schedule
        workload += ", serial spine (no segment workspace)"
    elif ws_bytes:  # varlen schedule, or the segment schedule of a long dense batch
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step():
        dp.run(workspace=ws)

    for _ in range(args.warmup):
        step()
    launches_per_step = gdn.last_launch_count()
    torch.cuda.synchronize()
    gdn.check()

    # ---- device-resident timing: K steps between two events on the launching stream
    # (nothing recorded between the steps or between the kernels of a step) ----
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for _ in range(args.steps):
            step()
        t_all1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(t_all0.elapsed_time(t_all1), world)
    gdn.check()
    clocks = clk.summary()

    # ---- per-kernel times: a second pass of K steps with events that the library
    # records before the WY solve, between the kernels and after the spine. The event
    # between them serialises the spine behind the WY kernel (no dependent launch), so
    # these are each kernel's own times; the headline pass above runs without them.
    k_wy, k_sp, k_end = ([torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] for _ in range(3))
    for ev in k_wy + k_sp + k_end:  # torch creates an event on its first record
        ev.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        gdn.set_timing_events(k_wy[i], k_sp[i], k_end[i])
        step()
    gdn.set_timing_events()
    torch.cuda.synchronize()
    wy_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(k_wy, k_sp))
    spine_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(k_sp, k_end))
    gdn.check()

    tokens = p.tokens
    ms_per_step = total_ms / args.steps
    value = world * tokens / (ms_per_step / 1e3)
    hbm_peak, tf_peak, peak_src = measured_peaks()
    op_ms = ms_per_step
    abytes = algorithmic_bytes(p)
    sbytes = spine_algorithmic_bytes(p)
    aflops = algorithmic_flops(p)
    achieved_gbs = sbytes / (spine_ms / 1e3) / 1e9  # the dominant kernel: the spine
    op_gbs = abytes / (op_ms / 1e3) / 1e9
    roofline_ms = max(aflops / (tf_peak * 1e12), abytes / (hbm_peak * 1e9)) * 1e3

    # ---- end to end through the C ABI's host-buffer entry point (gdn_prefill_host):
    # page-locked host inputs and state, copied in, the op, the output rows and the
    # state copied back, every step; the state is carried on the host in place ------------
    host = {}
    for name in ("q", "k", "v", "g", "beta"):
        t = getattr(dp, name)
        host[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    h_state = torch.from_numpy(p.h0.copy()).pin_memory()  # contiguous [B, nv, dk, dv]
    h_out = torch.empty(dp.out.shape, dtype=dp.out.dtype, pin_memory=True)
    h_cu = None if dp.cu is None else dp.cu.cpu().pin_memory()
    h2d = sum(host[n].numel() * host[n].element_size() for n in host) + h_state.numel() * 4
    d2h = h_out.numel() * h_out.element_size() + h_state.numel() * 4
    e2e_steps = max(3, min(args.steps, 10))
    h_scratch = torch.empty(gdn.host_scratch_bytes(p.B, p.T, p.nk, p.nv, p.varlen), dtype=torch.uint8, device=dev)

    def e2e_step():
        gdn.prefill_host(host["q"], host["k"], host["v"], host["g"], host["beta"], h_state, h_out, nk=p.nk,
                         nv=p.nv, B=p.B, T=p.T, cu_seqlens=h_cu, scratch=h_scratch, qk_l2norm=dp.qk_l2norm)

    e2e_step()
    e2e_launches = gdn.last_launch_count()
    torch.cuda.synchronize()
    gdn.check()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    barrier(world)

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(p, args.ref_seconds)
        rate, _ = sample.run()
        cpu = {"value": rate, "unit": "tokens/s", "cores": sample.cores, "kind": "oracle", "sample": sample.sample}
    traffic = recorded_traffic(workload)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 I/O, fp16/bf16 tensor-core operands, fp32 accumulate and state",
        "data": "synthetic",
        "config": {"workload": workload, "tokens_per_step": tokens, "l2": "no flush: inputs+outputs "
                   f"{abytes / 1e6:.0f} MB per step > 129 MB L2", "parallelism": "replicas" if world > 1 else "1 GPU",
                   "state": "carried from step to step (in place)"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                     "kernel": "gdn_prefill_kernel", "kernel_ms": spine_ms, "algorithmic_bytes": sbytes,
                     "kernels_ms": {"gdn_wy_kernel": wy_ms, "gdn_prefill_kernel": spine_ms},
                     "op": {"ms": op_ms, "algorithmic_bytes": abytes, "achieved": op_gbs, "frac": op_gbs / hbm_peak,
                            "algorithmic_flops": aflops, "tflops": aflops / (op_ms / 1e3) / 1e12,
                            "roofline_ms": roofline_ms, "frac_of_roofline_time": roofline_ms / op_ms},
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "entry_point": "gdn_prefill_host",
                "kernels_per_step": e2e_launches},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_decode(args, world, rank, local):
    """The single-token decode step at a serving batch (B sequences x 32 v-heads), one
    token per sequence per step, state carried in place; HBM-bound on the state."""
    import torch

    import gated_delta_rule_17_gb300 as gdn
    from gated_delta_rule_17_gb300 import build as gbuild

    gbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B = args.decode_batch
    p = gdn_synth.make_problem(seed=6100, B=B, T=args.steps + args.warmup, nk=16, nv=32, h0_std=0.02)
    from gdn_synth.device import DeviceProblem

    dp = DeviceProblem(p, device=dev)
    stream = torch.cuda.current_stream(dev)
    views = [x.view(p.B, p.T, *x.shape[1:]) for x in (dp.q, dp.k, dp.v, dp.g, dp.beta, dp.out)]

    def step(t):
        q, k, v, g, beta, out = (x[:, t] for x in views)
        gdn.decode(q, k, v, g, beta, dp.state, out, nk=p.nk, nv=p.nv)

    for t in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    gdn.check()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for t in range(args.warmup, args.warmup + args.steps):
            step(t)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    gdn.check()
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    hbm_peak, _, peak_src = measured_peaks()
    state_bytes = 2 * B * p.nv * p.dk * p.dv * 4
    io_bytes = B * (2 * p.nk * p.dk * 2 + 2 * p.nv * p.dv * 2 + p.nv * 8)
    achieved = (state_bytes + io_bytes) / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "GDN decode tokens/s (one token per sequence, nv=32, dk=dv=128), 1xGB300",
            "value": world * B / (ms / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 I/O, fp32 state and arithmetic", "data": "synthetic",
            "config": {"workload": f"decode B={B} nk=16 nv=32 dk=dv=128 h0~N(0,0.02)",
                       "l2": f"no flush: {state_bytes / 1e6:.0f} MB of state per step", "parallelism": "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None, "kernel": "gdn_decode_kernel",
                         "algorithmic_bytes": state_bytes + io_bytes, "peak_source": peak_src},
            "gpu_launches": args.steps, "clocks": clk.summary()}), flush=True)


def run_backward(args, world, rank, local):
    """The backward of the prefill (dL/dq, dk, dv, dg, dbeta, dS_0 from dL/do and
    dL/dS_T) on a workload of --config, inputs resident in HBM."""
    import torch

    import gated_delta_rule_17_gb300 as gdn
    from gated_delta_rule_17_gb300 import build as gbuild

    gbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    p = gdn_synth.config_problem(args.config)
    from gdn_synth.device import DeviceProblem

    dp = DeviceProblem(p, device=dev)
    rng = torch.Generator(device=dev).manual_seed(7)
    rows = p.rows
    f32 = dict(dtype=torch.float32, device=dev)
    dout = torch.randn((rows, p.nv * p.dv), generator=rng, **f32)
    dst = torch.randn((p.B, p.nv, p.dk, p.dv), generator=rng, **f32)
    dq = torch.empty((rows, p.nk * p.dk), **f32)
    dk = torch.empty_like(dq)
    dv = torch.empty((rows, p.nv * p.dv), **f32)
    dg = torch.empty((rows, p.nv), **f32)
    dbeta = torch.empty_like(dg)
    dh0 = torch.empty((p.B, p.nv, p.dk, p.dv), **f32)
    ws = torch.empty(gdn.backward_workspace_bytes(p.B, p.T, p.nv, p.varlen), dtype=torch.uint8, device=dev)
    h0 = dp.state  # the initial state (no forward runs here)
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.backward(dp.q, dp.k, dp.v, dp.g, dp.beta, h0, dout, dq, dk, dv, dg, dbeta, nk=p.nk, nv=p.nv,
                     B=p.B, T=p.T, cu_seqlens=dp.cu, dST=dst, dh0=dh0, state_is_table=dp.table, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    gdn.check()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    gdn.check()
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    launches = gdn.last_launch_count()
    hbm_peak, _, peak_src = measured_peaks()
    tokens = p.tokens
    # each input read once and each gradient written once, the states in and out
    io = tokens * (2 * p.nk * p.dk * 2 + p.nv * p.dv * 2 + p.nv * 8 + p.nv * p.dv * 4
                   + 2 * p.nk * p.dk * 4 + p.nv * p.dv * 4 + p.nv * 8) + 3 * p.B * p.nv * p.dk * p.dv * 4
    achieved = io / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "GDN prefill backward tokens/s (dq, dk, dv, dg, dbeta, dS_0), 1xGB300",
            "value": world * tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 inputs, fp16 tensor-core operands, fp32 accumulate, states and gradients",
            "data": "synthetic",
            "config": {"workload": gdn_synth.CONFIG_NAMES[args.config], "parallelism": "1 GPU",
                       "l2": "no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None,
                         "kernel": "whole backward (WY, two chains, per-chunk gradients)",
                         "algorithmic_bytes": io, "peak_source": peak_src},
            "gpu_launches": launches * args.steps, "clocks": clk.summary()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--config", type=int, default=2, help="workload index (2 = B=4 T=8192 nv=32)")
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="prefill", choices=["prefill", "decode", "backward"],
                    help="prefill (the headline) or the single-token decode step")
    ap.add_argument("--no-segments", action="store_true",
                    help="dense batches: run the serial spine even where the segment schedule applies")
    ap.add_argument("--qk-l2norm", action="store_true",
                    help="un-normalised q/k inputs, normalised by the fused prologue")
    ap.add_argument("--decode-batch", type=int, default=256, help="sequences per decode step")
    ap.add_argument("--profile-case", action="store_true",
                    help="the smaller case ncu's multi-pass captures use: " + PROFILE_CASE)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.op == "decode":
        run_decode(args, world, rank, local)
    elif args.op == "backward":
        run_backward(args, world, rank, local)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
