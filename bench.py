#!/usr/bin/env python
"""Benchmark of the sparse MLA training backward on one GB300 (or N replicas).

One step = one full backward (delta, CSR build, S/dP/P/dS, dKV intermediate,
dq, atomic-free dKV gather, d_sink) through the C ABI on the headline
workload of the aiter page's Performance table: T=4096, H=128, D=512,
topk=512, num_kv=5120 (128-row causal window + 384 uniform pool picks),
synthetic seeded inputs (no dataset exists for it). O and lse come from the
library's forward, which is also timed on its own and reported under
"forward" (not part of the step).

Prints ONE JSON line (rank 0). The metric is TFLOPS over the valid
(token, head, rank) triples at 5 GEMMs x 2 x 512 FLOPs each; ms/call is
reported next to it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the correctness reference) on a
bounded token slice of the same workload, on the host's cores.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-MLA bwd TFLOPS & ms/call (T=4096,H=128,topk=512,D=512) vs BF16 peak"
WORKLOAD = "headline"
PAGES_CONTEXT = {"hardware": "AMD MI355X", "bwd_end_to_end_ms": 3.238, "bwd_tflops_nominal": 424}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() in ("active", "0x1", "1", "yes")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _busy(step, dev, seconds: float) -> None:
    """Runs `step` untimed for about `seconds` (synchronising every few steps)."""
    import torch
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(4):
            step()
        torch.cuda.synchronize(dev)


def _max_over_ranks(x: float, world: int, device) -> float:
    """The largest `x` over all ranks of the process group (x itself on one rank).
    Replicas are timed on their own; the job takes as long as the slowest one."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _whole_job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Throughput of the whole job: every rank's work over the (max-over-ranks) time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def _percentiles(ms_list) -> dict:
    """Median, p10, p90, mean, min and max of a list of per-call times (ms)."""
    s = sorted(float(x) for x in ms_list)
    if not s:
        return {}

    def pct(p):
        # linear interpolation between order statistics
        k = (len(s) - 1) * p
        lo = int(k)
        hi = min(lo + 1, len(s) - 1)
        return s[lo] + (s[hi] - s[lo]) * (k - lo)
    return {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9), "mean": sum(s) / len(s),
            "min": s[0], "max": s[-1], "n": len(s)}


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_sample(spec, inp, seconds: float = 12.0):
    """Times the fp64 oracle backward on a token slice sized to about `seconds`."""
    import numpy as np
    import oracle
    from sparse_mla_attention_gb300 import workloads as W

    kv64 = oracle.bf16_to_f64(inp["kv"])
    t0 = spec.T // 2

    def run(n):
        sl = slice(t0, t0 + n)
        q64 = oracle.bf16_to_f64(inp["q"][sl])
        do64 = oracle.bf16_to_f64(inp["do"][sl])
        topk = np.ascontiguousarray(inp["topk"][sl])
        sink = None if inp["sink"] is None else inp["sink"].astype(np.float64)
        o64, lse = oracle.fwd(q64, kv64, topk, sink, inp["scale"])
        o_in = oracle.bf16_to_f64(oracle.f64_to_bf16(o64))
        lse_in = lse.astype(np.float32).astype(np.float64)
        t = time.perf_counter()
        oracle.bwd(q64, kv64, do64, o_in, lse_in, topk, sink, inp["scale"])
        dt = time.perf_counter() - t
        return dt, W.flops_valid(topk, spec.H)

    dt, fl = run(4)
    n = int(max(4, min(spec.T - t0, 4 * seconds / max(dt, 1e-3))))
    dt, fl = run(n)
    return {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": oracle.threads(),
            "cpu_model": _cpu_model(), "kind": "oracle",
            "sample": f"full fp64 backward (dq, dkv scatter, d_sink) of tokens "
                      f"{t0}..{t0 + n - 1} of the {spec.name} workload ({dt:.1f} s); TFLOPS over "
                      f"that slice's valid triples, extrapolated to the whole workload at the "
                      f"same rate",
            "extrapolated": True, "ms_per_token": dt * 1e3 / n}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from sparse_mla_attention_gb300 import workloads as W
    import oracle
    oracle.build()
    spec = W.WORKLOADS[args.workload]
    inp = W.make_inputs(spec)
    per_step = max(2.0, 60.0 / max(args.steps + args.warmup, 1))
    res = None
    vals = []
    for i in range(args.warmup + args.steps):
        res = cpu_oracle_sample(spec, inp, seconds=per_step)
        if i >= args.warmup:
            vals.append(res["value"])
    value = statistics.median(vals) if vals else res["value"]
    total_flops = W.flops_valid(inp["topk"], spec.H)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_flops / (value * 1e12) * 1e3 if value > 0 else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": spec.name, "shape": spec.describe(),
                   "note": "each step times the fp64 oracle on a bounded token slice; "
                           "ms_per_step is extrapolated to the whole workload from that "
                           "slice's rate (not measured over the whole workload)",
                   "ms_per_step_extrapolated": True},
        "cpu_baseline": {"kind": res["kind"], "cores": res["cores"], "cpu_model": res["cpu_model"],
                         "sample": res["sample"], "extrapolated": True,
                         "value": value, "unit": "TFLOPS"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sparse_mla_attention_gb300 import build as smla_build
    smla_build.build()
    import sparse_mla_attention_gb300 as smla
    from sparse_mla_attention_gb300 import _lib, workloads as W

    spec = W.WORKLOADS[args.workload]
    inp = W.make_inputs(spec)
    if args.tokens and args.tokens < spec.T:
        # a token prefix of the workload (profiling runs on small cases)
        import dataclasses
        spec = dataclasses.replace(spec, T=args.tokens)
        for k in ("q", "do", "topk"):
            inp[k] = np.ascontiguousarray(inp[k][: args.tokens])
    T, H, K, N = spec.T, spec.H, spec.topk, spec.num_kv

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, kv, do = (dev_bf16(inp[k]) for k in ("q", "kv", "do"))
    topk = torch.from_numpy(inp["topk"]).to(dev)
    sink = None if inp["sink"] is None else torch.from_numpy(inp["sink"]).to(dev)
    o, lse = smla.sparse_mla_fwd(q, kv, topk, sink, scale=inp["scale"])
    r_chunk = spec.r_chunk or None
    ws = smla.Workspace(dev)
    dq = torch.empty_like(q)
    dkv = torch.empty_like(kv)
    dsink = None if sink is None else torch.empty(H, dtype=torch.float32, device=dev)
    out = (dq, dkv, dsink)

    def step():
        smla.sparse_mla_bwd(q, kv, do, o, lse, topk, sink, scale=inp["scale"], r_chunk=r_chunk,
                            workspace=ws, out=out, check_status=False)

    step()
    st = smla.device_status(ws.buf)
    if st != 0:
        raise RuntimeError(f"device status {st} after the first step")
    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    # the clock samples (every 100 ms) should see the GPU under this load: the
    # same step runs untimed for about 0.4 s before and 0.3 s after the K timed
    # steps (the timed region itself lasts only K steps)
    _busy(step, dev, 0.4)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # K + 1 events on the launching stream: the region e[0] -> e[K] is the timed
    # total (its mean is ms_per_step); e[i] -> e[i+1] is call i (median, p10, p90)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    elapsed_ms = evs[0].elapsed_time(evs[-1])
    per_call = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    # the phase split comes from a second, untimed pass of the same K steps with
    # the library's phase events on (no profiler event inside the timed region)
    _lib.profiling(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    phases = _lib.profile_read()
    _lib.profiling(False)
    _busy(step, dev, 0.3)
    clk = clocks.stop()
    ms = _max_over_ranks(elapsed_ms / args.steps, world, dev)
    call_stats = _percentiles(per_call)

    flops = W.flops_valid(inp["topk"], H)
    flops_nom = W.flops_nominal(T, H, K)
    value = _whole_job_tflops(flops, world, ms)
    launches = int(sum(p["launches"] for p in phases.values()))

    # ---- end to end: host (pinned) inputs -> device -> backward -> host results
    e2e = None
    if not args.no_e2e:
        host_in = {"q": q.cpu().pin_memory(), "kv": kv.cpu().pin_memory(),
                   "do": do.cpu().pin_memory(), "o": o.cpu().pin_memory(),
                   "lse": lse.cpu().pin_memory(), "topk": topk.cpu().pin_memory()}
        if sink is not None:
            host_in["sink"] = sink.cpu().pin_memory()
        host_out = {"dq": torch.empty(dq.shape, dtype=dq.dtype).pin_memory(),
                    "dkv": torch.empty(dkv.shape, dtype=dkv.dtype).pin_memory()}
        if dsink is not None:
            host_out["dsink"] = torch.empty(dsink.shape, dtype=dsink.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())
        ws_host = smla.Workspace(dev)

        def e2e_step():
            # the public host-buffer entry point: copies in, backward, copies out,
            # pipelined by token chunks inside the library
            smla.sparse_mla_bwd_host(host_in["q"], host_in["kv"], host_in["do"], host_in["o"],
                                     host_in["lse"], host_in["topk"], host_in.get("sink"),
                                     scale=inp["scale"], r_chunk=r_chunk, workspace=ws_host,
                                     out=(host_out["dq"], host_out["dkv"], host_out.get("dsink")),
                                     device=dev, synchronize=False)

        # the first calls of a fresh process pay for first touches of the host and
        # device buffers: warm up like the device leg (at least 3 calls)
        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 10))
        if world > 1:
            dist.barrier()
        # each call timed on its own (host-device copies share the machine's
        # host links, whose speed varies): the median call is reported
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_e2e)]
        for a_, b_ in evs:
            a_.record(stream)
            e2e_step()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        per_call = sorted(a_.elapsed_time(b_) for a_, b_ in evs)
        ms_e2e = _max_over_ranks(per_call[len(per_call) // 2], world, dev)
        e2e = {"value": _whole_job_tflops(flops, world, ms_e2e), "unit": "TFLOPS",
               "ms_per_step": ms_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "calls": n_e2e, "ms_per_step_median_of": "calls",
               "ms_per_step_mean": sum(per_call) / len(per_call),
               "ms_per_step_min": per_call[0], "ms_per_step_max": per_call[-1],
               "per_call_ms": _percentiles(per_call),
               "api": "smla_bwd_host (host buffers, copies pipelined by token chunks)"}

    # ---- roofline of the dominant kernel (live CUDA-event phase times)
    peaks = _peaks()
    # A phase overlapped with others has an event span that is not its own run
    # time, so it is not a candidate for the dominant kernel.
    dom_name, dom = max(((k, v) for k, v in phases.items() if k not in OVERLAPPED_PHASES),
                        key=lambda kv_: kv_[1]["ms"])
    per_launch_ms = dom["ms"] / max(dom["calls"], 1)
    roofline = {"kernel": dom_name, "share_of_step": dom["ms"] / max(elapsed_ms, 1e-9)}
    algo = _algorithmic(dom_name, spec, inp["topk"])
    if algo["bound"] == "tensor":
        achieved = algo["flops"] / (per_launch_ms * 1e-3) / 1e12
        roofline.update({"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                         "peak_source": peaks["source"] + " bf16 burst"})
    elif algo["bound"] == "alu":
        achieved = algo["flops"] / (per_launch_ms * 1e-3) / 1e12
        alu_peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        roofline.update({"bound": "alu", "achieved": achieved, "peak": alu_peak,
                         "unit": "TFLOP/s", "frac": achieved / alu_peak,
                         "peak_source": "derived: 152 SMs x 128 fp32 FMA/clk x 2 x max SM clock"})
    else:
        achieved = algo["bytes"] / (per_launch_ms * 1e-3) / 1e9
        roofline.update({"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "peak_source": peaks["source"] + " copy"})
    traffic, tnote = _traffic(dom_name, T)
    roofline["traffic"] = traffic
    roofline["traffic_note"] = tnote
    roofline["per_launch_ms"] = per_launch_ms

    # ---- the forward (O, lse) on the same inputs, timed on its own; not part of the step
    fwd = None
    if not args.no_fwd:
        f_o = torch.empty_like(q)
        f_lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        ws_f = smla.Workspace(dev)

        def fwd_step():
            smla.sparse_mla_fwd(q, kv, topk, sink, scale=inp["scale"], workspace=ws_f,
                                check_status=False, out=(f_o, f_lse))

        for _ in range(max(3, args.warmup)):
            fwd_step()
        if smla.device_status(ws_f.buf) != 0:
            raise RuntimeError("device status set by the forward")
        torch.cuda.synchronize(dev)
        fev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        fev[0].record(stream)
        for i in range(args.steps):
            fwd_step()
            fev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        ms_f = _max_over_ranks(fev[0].elapsed_time(fev[-1]) / args.steps, world, dev)
        f_calls = _percentiles(fev[i].elapsed_time(fev[i + 1]) for i in range(args.steps))
        f_flops = 2 * 2 * 512 * H * W.valid_ranks(inp["topk"])   # S and O GEMMs
        f_tf = _whole_job_tflops(f_flops, world, ms_f)
        tc = H % 32 == 0 and 1 <= K <= 512
        f_traffic, f_note = _traffic("fwd_tc", T) if tc else (None, None)
        fwd = {"ms_per_call": ms_f, "tflops_valid": f_tf, "calls": args.steps, "per_call_ms": f_calls,
               "kernel": "fwd_tc_kernel" if tc else "fwd_kernel",
               "roofline": {"bound": "tensor", "achieved": f_tf, "peak": peaks["bf16_tflops"],
                            "unit": "TFLOP/s", "frac": f_tf / peaks["bf16_tflops"],
                            "peak_source": peaks["source"] + " bf16 burst",
                            "traffic": f_traffic, "traffic_note": f_note},
               "flops_valid_per_call": f_flops}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(spec, inp, seconds=args.cpu_seconds)

    # ---- the other configurations of the workload table, timed the same way
    # (after the headline's timed region; one GPU only)
    others = None
    if world == 1 and not args.no_configs and not args.tokens and args.workload == WORKLOAD:
        others = _other_configs(dev, peaks, steps=max(10, args.steps // 5), warmup=3)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": spec.name, "shape": spec.describe(),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (q, dO, O: 1.5 GB)",
                   "flops_valid_per_step": flops, "flops_nominal_per_step": flops_nom,
                   "tflops_nominal": _whole_job_tflops(flops_nom, world, ms),
                   "frac_of_bf16_peak": value / world / peaks["bf16_tflops"]},
        "per_call_ms": call_stats,
        "phases_ms_per_step": {k: v["ms"] / args.steps for k, v in phases.items()},
        "phases_note": "CUDA-event phase times from a separate untimed pass of the same steps",
        "phases_overlapped": list(OVERLAPPED_PHASES),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "forward": fwd,
        "other_configs": others,
        "gpu_launches": launches,
        "clocks": clk,
        "pages_context": PAGES_CONTEXT,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _other_configs(dev, peaks, steps: int, warmup: int) -> dict:
    """ms per backward call (median, p10, p90 of `steps` calls) and valid TFLOP/s
    of the workload table's other large configurations: H=64 with four rank
    chunks of 128, and T=8192 with Zipf pool picks and 30 % masked ranks."""
    import numpy as np
    import torch
    import sparse_mla_attention_gb300 as smla
    from sparse_mla_attention_gb300 import workloads as W
    res = {}
    stream = torch.cuda.current_stream(dev)
    for name in ("headline_h64_chunked", "t8192_zipf"):
        spec = W.WORKLOADS[name]
        inp = W.make_inputs(spec)

        def up(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

        q, kv, do = (up(inp[k]) for k in ("q", "kv", "do"))
        topk = torch.from_numpy(inp["topk"]).to(dev)
        sink = None if inp["sink"] is None else torch.from_numpy(inp["sink"]).to(dev)
        o, lse = smla.sparse_mla_fwd(q, kv, topk, sink, scale=inp["scale"])
        ws = smla.Workspace(dev)
        out = (torch.empty_like(q), torch.empty_like(kv),
               None if sink is None else torch.empty(spec.H, dtype=torch.float32, device=dev))

        def step():
            smla.sparse_mla_bwd(q, kv, do, o, lse, topk, sink, scale=inp["scale"],
                                r_chunk=spec.r_chunk or None, workspace=ws, out=out, check_status=False)

        step()
        if smla.device_status(ws.buf) != 0:
            raise RuntimeError(f"device status set by the {name} backward")
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        calls = _percentiles(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
        flops = W.flops_valid(inp["topk"], spec.H)
        tf = flops / (calls["median"] * 1e-3) / 1e12
        res[name] = {"shape": spec.describe(), "per_call_ms": calls, "flops_valid_per_call": flops,
                     "tflops_valid": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 burst"}
        del q, kv, do, topk, sink, o, lse, ws, out
        torch.cuda.empty_cache()
    return res


# Phases that run concurrently with others (the CSR build and dq on the
# library's side stream, the dKV gather beside dq): their event spans are not
# their own run times.
OVERLAPPED_PHASES = ("csr", "attn_dq", "gather")

# DRAM traffic per launch of the dominant kernels, from one ncu capture (see
# profiles/), valid only while the kernel source is the one captured.
_NCU_TRAFFIC = {
    "attn_sdi": {"sources": ("sparse_mla_attention_gb300/csrc/k_attn_tc.cu", "c0d38424e2c5da67"),
                 "bytes_per_token": (140.994816e6 + 275.318272e6) / 512,
                 "note": "ncu capture of the first 512 tokens, scaled by tokens"},
    "attn_dq": {"sources": ("sparse_mla_attention_gb300/csrc/k_attn_tc.cu", "c0d38424e2c5da67"),
                "bytes_per_token": (68.702208e6 + 23.128832e6) / 512,
                "note": "ncu capture of the first 512 tokens, scaled by tokens"},
    "fwd_tc": {"sources": ("sparse_mla_attention_gb300/csrc/k_fwd_tc.cu", "1debdf8c27880f41"),
               "bytes_per_token": (73.644544e6 + 18.696448e6) / 512,
               "note": "ncu capture of the first 512 tokens, scaled by tokens"},
}


def _traffic(phase: str, T: int):
    import hashlib
    ent = _NCU_TRAFFIC.get(phase)
    if not ent:
        return None, None
    path, want = ent["sources"]
    try:
        got = hashlib.sha256(open(os.path.join(ROOT, path), "rb").read()).hexdigest()[:16]
    except OSError:
        return None, None
    if got != want:
        return None, "kernel changed since the ncu capture"
    return ent["bytes_per_token"] * T, ent["note"]


def _algorithmic(phase: str, spec, topk):
    """Algorithmic work per launch of one phase (FLOPs or bytes)."""
    from sparse_mla_attention_gb300 import workloads as W
    T, H, K, N = spec.T, spec.H, spec.topk, spec.num_kv
    valid = W.valid_ranks(topk)
    nchunks = K // (spec.r_chunk or K)
    if phase == "attn_sdi":       # S, dP, interm: 4 of the 5 GEMMs
        return {"bound": "tensor", "flops": 4 * 2 * 512 * H * valid / nchunks}
    if phase == "attn_dq":
        return {"bound": "tensor", "flops": 1 * 2 * 512 * H * valid / nchunks}
    if phase == "delta":
        return {"bound": "hbm", "bytes": 2 * T * H * 512 * 2 + T * H * 4}
    if phase == "gather":
        per = valid / nchunks
        return {"bound": "hbm", "bytes": per * 512 * 2 + per * 4 + N * 512 * 2}
    if phase == "csr":
        per = T * (K // nchunks)
        return {"bound": "hbm", "bytes": per * 4 * 6}
    return {"bound": "hbm", "bytes": T * H * 8}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fwd", action="store_true", help="skip the separate forward timing")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other configurations (H=64 chunked, T=8192 Zipf)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--tokens", type=int, default=0,
                    help="time only the first N tokens of the workload (small profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
