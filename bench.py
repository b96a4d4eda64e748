#!/usr/bin/env python3
"""GMA forward benchmark on one GB300 (or N independent replicas under torchrun).

Metric: tokens*heads per second of the Gaussian Mixture Attention forward.
One step = one bidirectional forward plus one causal forward over the
N = 8192 workload (B=8, H=12, N=8192, d=64, K=64, dv=64, bf16 inputs and
outputs), so every step of the path runs: parameter prologue,
responsibilities, latent write, read, and the causal chunked scan.
A step processes 2 * B * H * N tokens*heads.

Inputs are synthetic (seeded, see gaussian_mixture_latent_gb300/inputs.py).
Two input sets of 302 MB each (more than the 129 MB L2) alternate between
steps, so every step streams its inputs from HBM.

Output: one JSON line (rank 0).  --impl reference times the CPU fp64 oracle
on the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from gaussian_mixture_latent_gb300 import accounting, inputs  # noqa: E402

WORKLOAD = "causal_bf16_n8192"
METRIC = "GMA fwd tokens·heads/s (bidir & causal, N=8192); % of HBM/tensor roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 3 s, 20..5000)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--direction", choices=["both", "bidir", "causal", "diagnostics", "cross", "decode", "backward",
                                            "backward_causal", "project"],
                    default="both",
                    help="which forward(s) one step runs (default: both, the headline step); "
                         "diagnostics: one step is gma_diagnostics over the workload's query vectors; "
                         "cross: one step is gma_forward_cross, the workload's queries reading a context; "
                         "decode: one step is gma_decode of one new token for every head; "
                         "project: one step is gma_project, the Q/K/V projections of the workload's rows "
                         "from a model width of H d")
    ap.add_argument("--schedule", choices=["multi", "sequential"], default="multi",
                    help="both directions: one gma_forward_multi request with the causal scan on a second "
                         "stream beside the bidirectional forward (default), or two gma_forward calls one "
                         "after the other on one stream")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's sequence length N (a reduced case for profiling)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size B")
    ap.add_argument("--context", type=int, default=0,
                    help="context length of --direction cross (default: 4 x the workload's N)")
    return ap.parse_args()


def workload(args):
    """The named workload, with its sequence length replaced when --seq-len is given."""
    w = inputs.WORKLOADS[args.workload]
    if args.seq_len:
        w = w.replace(N=args.seq_len)
    return w.replace(B=args.batch) if args.batch else w


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device="cpu"):
    """The largest per-rank value of `x` over the process group (the slowest rank's step
    time); `x` itself outside a multi-rank run."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def device_status(gma, ws=None, offsets=()):
    """The device status of the library's default workspace, or of every call region of a
    gma_forward_multi workspace (the first error found)."""
    import torch
    if ws is None:
        return gma.gma_get_status()
    stream = int(torch.cuda.current_stream().cuda_stream)
    for off in offsets:
        st = gma._load().gma_get_status(int(ws.data_ptr()) + int(off), stream)
        if st:
            return st
    return 0


def whole_job_rate(units_per_rank, world, ms_per_step):
    """Units per second of the whole job: every rank processes `units_per_rank` per step
    (heads are independent: weak scaling, no data-path collective), timed by the slowest."""
    return world * units_per_rank / (ms_per_step / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "sm_max_mhz": p.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def fp32_simt_peak_tflops(sm_mhz):
    # 152 SMs x 128 FP32 lanes x 2 flops per FMA x clock
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


# The sources that define each measured kernel: its translation unit and the device headers
# it includes.  A recorded traffic figure holds while these files are unchanged.
KERNEL_SOURCES = {
    "tc_causal": ("gma_tc_causal.cu", "gma_tc_common.cuh", "gma_sm100.cuh"),
    "tc_causal_seg": ("gma_tc_causal.cu", "gma_tc_common.cuh", "gma_sm100.cuh"),
    "tc_prefix": ("gma_tc.cu", "gma_tc_common.cuh", "gma_sm100.cuh"),
    "tc_write": ("gma_tc.cu", "gma_tc_common.cuh", "gma_sm100.cuh"),
    "tc_read": ("gma_tc.cu", "gma_tc_common.cuh", "gma_sm100.cuh"),
}


def csrc_hash(kernel=None):
    """Hash of the CUDA sources of `kernel` (every file of csrc when it is not listed)."""
    csrc = os.path.join(ROOT, "gaussian_mixture_latent_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel)
    paths = [os.path.join(csrc, n) for n in names] if names else sorted(glob.glob(os.path.join(csrc, "*")))
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


DOM_EVERY = 8   # the dominant kernel is bracketed by CUDA events on every 8th timed step
PRE_ROLL = 2    # untimed warm-up steps queued right before the headline's start event


def known_traffic(kernel):
    """DRAM bytes (read + write) per launch of `kernel` on this workload, from an ncu
    capture recorded in profiles/kernel_traffic.txt, or None when the recorded capture
    was taken on different sources of that kernel (csrc_hash(kernel))."""
    path = os.path.join(ROOT, "profiles", "kernel_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == WORKLOAD \
                    and parts[2] == csrc_hash(kernel):
                return int(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_id_for(dev_index):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if dev_index < len(ids):
            return ids[dev_index]
    return str(dev_index)


def cpu_baseline(w, dirs=(False, True), seconds=12.0):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload:
    the first `heads` heads, full sequence, both directions, one thread per head,
    repeated until about `seconds` of wall time have passed."""
    import oracle
    cores = max(1, len(os.sched_getaffinity(0)))
    heads = min(w.G, cores)
    p = inputs.gen_params(w)
    data = []
    for g in range(heads):
        data.append({n: inputs.widen(inputs.gen_head(w, n, g, p), w.dtype) for n in ("Qx", "Kx", "V")})
    Q = np.stack([x["Qx"] for x in data])[None]
    Kx = np.stack([x["Kx"] for x in data])[None]
    V = np.stack([x["V"] for x in data])[None]
    hs = [g % w.H for g in range(heads)]
    mu, rho, al = p["mu"][hs], p["rho"][hs], p["alpha"][hs]
    reps, t0 = 0, time.perf_counter()
    while True:
        for causal in dirs:
            oracle.forward(Q, Kx, V, mu, rho, al, w.var_floor, w.eps, causal, threads=heads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    units = len(dirs) * heads * w.N * reps
    what = " + ".join("causal" if c else "bidirectional" for c in dirs)
    return {"value": units / dt, "unit": "tokens·heads/s", "cores": heads, "kind": "oracle",
            "sample": f"{heads} heads x N={w.N} of the {w.name} workload, {what}, "
                      f"{reps} passes (fp64 C oracle, one thread per head), {dt:.1f} s wall"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = workload(args)
    import oracle
    oracle.build()
    cores = max(1, len(os.sched_getaffinity(0)))
    heads = min(w.G, cores)
    p = inputs.gen_params(w)
    data = [{n: inputs.widen(inputs.gen_head(w, n, g, p), w.dtype) for n in ("Qx", "Kx", "V")}
            for g in range(heads)]
    Q = np.stack([x["Qx"] for x in data])[None]
    Kx = np.stack([x["Kx"] for x in data])[None]
    V = np.stack([x["V"] for x in data])[None]
    hs = [g % w.H for g in range(heads)]
    mu, rho, al = p["mu"][hs], p["rho"][hs], p["alpha"][hs]

    dirs = {"both": (False, True), "bidir": (False,), "causal": (True,)}[args.direction]
    what = " + ".join("causal" if c else "bidirectional" for c in dirs)

    def step():
        for causal in dirs:
            oracle.forward(Q, Kx, V, mu, rho, al, w.var_floor, w.eps, causal, threads=heads)

    steps = args.steps if args.steps is not None else 3
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t0) / steps
    value = len(dirs) * heads * w.N / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens·heads/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                                        "K": w.K, "dv": w.dv, "step": what + " forward",
                                        "sample_heads": heads},
        "cpu_baseline": {"value": value, "unit": "tokens·heads/s", "cores": heads, "kind": "oracle",
                         "sample": f"each step: {heads} heads x N={w.N}, {what}"},
        "e2e": {"value": value, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, rank, world, local):
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    w = workload(args)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    # two resident input sets (each larger than L2), generated on the host
    def make_set(seed):
        ws = w.replace(seed=seed)
        x = inputs.gen_all(ws)
        def t(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)
        return {k: t(v) for k, v in x.items()}, x

    sets = [make_set(0), make_set(1)]
    dsets = [s[0] for s in sets]
    dirs = {"both": (False, True), "bidir": (False,), "causal": (True,)}[args.direction]
    outs = {c: torch.empty((w.B, w.H, w.N, w.dv), dtype=tdt, device=dev) for c in dirs}
    plan = {c: gma.gma_forward_plan(w.B, w.H, w.N, w.d, w.K, w.dv, tdt, causal=c) for c in dirs}
    stream = torch.cuda.current_stream()

    def new_event():
        # torch creates the CUDA event lazily at its first record(); the library
        # re-records it at the launch it brackets.
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    def forward(x, causal, events=None):
        return gma.gma_forward(x["Qx"], x["Kx"], x["V"], x["mu"], x["rho"], x["alpha"], eps=w.eps,
                               causal=causal, out=outs[causal], var_floor=w.var_floor,
                               events=events)

    # The step's forwards: with two directions, one gma_forward_multi request whose causal
    # scan (one CTA per head) runs on `aux` beside the bidirectional forward on `stream`.
    multi = len(dirs) > 1 and args.schedule == "multi"
    aux = torch.cuda.Stream(device=dev)
    mws, moffs = torch.zeros(1, dtype=torch.uint8, device=dev), []

    def step_forwards(x, evs=None, out=None, st=None):
        evs = evs or {}
        out = out or outs
        if not multi:
            for c in dirs:
                gma.gma_forward(x["Qx"], x["Kx"], x["V"], x["mu"], x["rho"], x["alpha"], eps=w.eps, causal=c,
                                out=out[c], var_floor=w.var_floor, events=evs.get(c), stream=st)
            return
        calls = [dict(Qx=x["Qx"], Kx=x["Kx"], V=x["V"], mu=x["mu"], rho=x["rho"], pi_logits=x["alpha"], eps=w.eps,
                      causal=c, out=out[c], var_floor=w.var_floor, events=evs.get(c)) for c in dirs]
        gma.gma_forward_multi(calls, workspace=mws, stream=st, aux_stream=aux)

    if multi:
        import ctypes
        nb, offs = ctypes.c_size_t(0), (ctypes.c_size_t * len(dirs))()
        calls = (gma.gma_forward_call * len(dirs))()
        for k, c in enumerate(dirs):
            calls[k].desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, tdt, tdt, w.var_floor, 0)
            calls[k].causal = int(c)
        assert gma._load().gma_forward_multi_workspace_size(calls, len(dirs), ctypes.byref(nb), offs) == 0
        mws, moffs = torch.zeros(nb.value, dtype=torch.uint8, device=dev), list(offs)

    # warm-up with every launch bracketed by events: finds the dominant kernel
    per = {}
    torch.cuda.nvtx.range_push("gma:warmup")          # coarse NVTX ranges, for ncu / nsys filters
    for it in range(max(3, args.warmup)):
        evs = {c: [new_event() for _ in range(2 * len(plan[c]))] for c in dirs}
        # keep the GPU busy while the host enqueues, so the events bracket GPU time only
        torch.cuda._sleep(2_000_000)
        step_forwards(dsets[it % 2], evs)
        torch.cuda.synchronize()
        if it >= 1:
            for c in dirs:
                for i, name in enumerate(plan[c]):
                    per.setdefault((c, name), []).append(evs[c][2 * i].elapsed_time(evs[c][2 * i + 1]))
    status = device_status(gma, mws if multi else None, moffs)
    if status:
        raise RuntimeError("device status after warm-up: " + gma.gma_status_string(status))
    share = {k: statistics.median(v) for k, v in per.items()}
    dom_c, dom_name = max(share, key=share.get)
    dom_idx = plan[dom_c].index(dom_name)

    # step count
    step_ms_est = sum(share.values())
    steps = args.steps if args.steps is not None else int(min(5000, max(20, 3000.0 / max(step_ms_est, 1e-3))))

    # timed region: events around the dominant kernel on every DOM_EVERY-th step.  An event
    # recorded between two kernels keeps the second from starting while the first drains
    # (programmatic dependent launch), so bracketing every step would slow the step itself
    # (by about 5 us even around the causal scan alone on its own stream, measured)
    dom_steps = list(range(0, steps, DOM_EVERY))
    dom_events = {it: [new_event(), new_event()] for it in dom_steps}
    sampler = ClockSampler(gpu_id_for(local))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_pop()
    torch.cuda.nvtx.range_push("gma:timed")
    # a GPU spin ahead of the start event lets the host enqueue the first steps before the GPU
    # reaches them, so the timed region starts with work queued (device time, not the host's
    # first launches); about the steps' estimated time, at most 20 ms.  PRE_ROLL untimed
    # warm-up steps run between the spin and the start event.
    torch.cuda._sleep(int(2.0e6 * min(20.0, (steps + PRE_ROLL) * max(step_ms_est, 0.1))))
    for it in range(PRE_ROLL):
        step_forwards(dsets[it % 2])
    t_start.record(stream)
    # a kernel between the timing event and the first request's fork: with the fork recorded
    # right after a timing event, that step's causal scan measured about 160 us slower (once);
    # a ~0.5 us spin in between removes it
    torch.cuda._sleep(1000)
    for it in range(steps):
        evs = None
        if it in dom_events:
            evs = {dom_c: [None] * (2 * len(plan[dom_c]))}
            evs[dom_c][2 * dom_idx], evs[dom_c][2 * dom_idx + 1] = dom_events[it]
        step_forwards(dsets[it % 2], evs)
    t_end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    clocks = sampler.stop()
    ms_per_step = max_over_ranks(t_start.elapsed_time(t_end) / steps, device=dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    status = device_status(gma, mws if multi else None, moffs)
    if status:
        raise RuntimeError("device status after timed region: " + gma.gma_status_string(status))
    dom_ms = statistics.mean(a.elapsed_time(b) for a, b in dom_events.values())
    units_per_step = len(dirs) * w.G * w.N
    value = whole_job_rate(units_per_step, world, ms_per_step)

    # roofline of the dominant kernel
    pk = peaks()
    bound, amount, unit = accounting.kernel_work(dom_name, w.G, w.N, w.d, w.K, w.dv, w.dtype,
                                                 w.dtype, H=w.H)
    if bound == "hbm":
        achieved = amount / (dom_ms / 1e3) / 1e9
        peak, runit = pk["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        achieved = amount / (dom_ms / 1e3) / 1e12
        peak, runit = pk["bf16_tflops"], "TFLOP/s"
    else:
        achieved = amount / (dom_ms / 1e3) / 1e12
        peak, runit = fp32_simt_peak_tflops(pk["sm_max_mhz"]), "TFLOP/s"
        bound = "alu"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": runit,
                "frac": achieved / peak, "traffic": known_traffic(dom_name), "kernel": dom_name,
                "kernel_ms": dom_ms, "kernel_timed_launches": len(dom_events), "peak_source": pk["source"] if bound != "alu" else
                "derived: 152 SMs x 128 FP32 lanes x 2 flop x max SM clock"}

    # whole-path roofline of one step (both directions)
    alg_bytes = len(dirs) * accounting.algorithmic_bytes(w.G, w.N, w.d, w.K, w.dv, w.dtype, w.dtype, H=w.H)
    alg_flops = len(dirs) * accounting.algorithmic_flops(w.G, w.N, w.d, w.K, w.dv)
    t_roof = max(alg_bytes / (pk["hbm_gbs"] * 1e9), alg_flops / (pk["bf16_tflops"] * 1e12))
    path = {"algorithmic_bytes_per_step": alg_bytes, "algorithmic_flops_per_step": alg_flops,
            "roofline_ms_per_step": t_roof * 1e3, "frac": t_roof * 1e3 / ms_per_step,
            "per_kernel_ms": {f"{'causal' if c else 'bidir'}:{n}": round(v, 5) for (c, n), v in share.items()}}

    # end to end through the public API from pinned host memory
    e2e = None
    if args.e2e_steps > 0:
        torch.cuda.nvtx.range_push("gma:e2e")
        # Pipelined like a serving loop: host->device copies, the forwards and device->host
        # copies run on three streams over two device buffer sets, so step i's uploads and
        # step i-1's downloads overlap step i-1 / i's kernels.  Every step still copies its
        # own inputs in and its own results out inside the timed region.
        host = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in dsets]
        hout = [{c: torch.empty(outs[c].shape, dtype=tdt, pin_memory=True) for c in dirs} for _ in range(2)]
        staging = [{k: torch.empty_like(v) for k, v in dsets[0].items()} for _ in range(2)]
        douts = [{c: torch.empty_like(outs[c]) for c in dirs} for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host[0].values())
        d2h = sum(v.numel() * v.element_size() for v in hout[0].values())
        s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        up_done = [ev(), ev()]          # inputs of the buffer set are on the device
        comp_done = [ev(), ev()]        # the forwards of the set are done (inputs free, outputs ready)
        down_done = [ev(), ev()]        # the outputs of the set have reached the host
        for e_ in comp_done + down_done:
            e_.record(stream)

        def e2e_step(i):
            b_ = i % 2
            with torch.cuda.stream(s_up):
                s_up.wait_event(comp_done[b_])                   # the set's previous forwards are done
                for k, v in host[i % 2].items():
                    staging[b_][k].copy_(v, non_blocking=True)
                up_done[b_].record(s_up)
            stream.wait_event(up_done[b_])
            stream.wait_event(down_done[b_])                     # the set's previous results were read
            step_forwards(staging[b_], out=douts[b_])
            comp_done[b_].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[b_])
                for c in dirs:
                    hout[b_][c].copy_(douts[b_][c], non_blocking=True)
                down_done[b_].record(s_down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_up)
        for i in range(args.e2e_steps):
            e2e_step(i)
        s_down.wait_stream(stream)
        s_down.wait_stream(s_up)
        b.record(s_down)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.e2e_steps, device=dev)
        e2e = {"value": whole_job_rate(units_per_step, world, e2e_ms), "unit": "tokens·heads/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        torch.cuda.nvtx.range_pop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        torch.cuda.nvtx.range_push("gma:cpu_baseline")
        cpu = cpu_baseline(w, dirs)
        torch.cuda.nvtx.range_pop()

    if rank == 0:
        launches = steps * sum(len(plan[c]) for c in dirs)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens·heads/s", "n_gpus": world,
            "steps": steps, "warmup": max(3, args.warmup) + PRE_ROLL, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K,
                       "dv": w.dv, "step": {"both": "bidirectional + causal forward", "bidir": "bidirectional forward",
                                "causal": "causal forward"}[args.direction],
                       "schedule": ("one gma_forward_multi request: the causal scan on a second stream beside "
                                    "the bidirectional forward" if multi else "gma_forward calls in order, one stream"),
                       "l2": "two alternating input sets of %d MB each (> 129 MB L2)" %
                             (sum(v.numel() * v.element_size() for v in dsets[0].values()) // 2**20),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "path_roofline": path, "clocks": clocks,
            "gpu_launches": launches, "kernels": {("causal" if c else "bidir"): plan[c] for c in dirs},
            "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


DIAG_METRIC = "GMA responsibility diagnostics tokens·heads/s (Eqs. 24-29); % of HBM roofline"


def diag_units(w):
    return w.B * w.H * w.N          # token-head responsibility vectors per step


def diag_oracle_sample(w, seconds):
    """The oracle's diagnostics on a bounded sample: sequence 0, all heads, the first n rows
    (n doubled until one call takes about `seconds` / 4); returns (token-heads per second, n)."""
    import oracle
    oracle.build()
    x = inputs.gen_all(w.replace(B=1))
    Q = inputs.widen(x["Qx"], w.dtype)
    n, dt = 256, 0.0
    while True:
        n = min(n, w.N)
        t0 = time.perf_counter()
        oracle.diagnostics(Q[:, :, :n], x["mu"], x["rho"], x["alpha"], w.var_floor)
        dt = time.perf_counter() - t0
        if dt >= seconds / 4 or n == w.N:
            break
        n *= 2
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.diagnostics(Q[:, :, :n], x["mu"], x["rho"], x["alpha"], w.var_floor)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return w.H * n / dt, n, reps, dt


def run_diagnostics(args, rank, world, local):
    """Responsibility diagnostics (section 5.4, Eqs. 24-29): one step is one gma_diagnostics
    call over the query routing vectors of the whole workload (every head of every sequence)."""
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build
    w = workload(args)
    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, n, reps, dt = diag_oracle_sample(w, 12.0)
        sample = f"sequence 0, {w.H} heads x the first {n} rows of {w.name}, {reps} calls, one thread"
        line = {"impl": "reference", "metric": DIAG_METRIC, "value": rate, "unit": "tokens·heads/s",
                "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": dt * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "step": "diagnostics (sampled)"},
                "cpu_baseline": {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": rate, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    host = [inputs.gen_all(w.replace(seed=s)) for s in (0, 1)]
    dsets = [{k: to_dev(x[k]) for k in ("Qx", "mu", "rho", "alpha")} for x in host]
    stream = torch.cuda.current_stream()

    def step(x):
        return gma.gma_diagnostics(x["Qx"], x["mu"], x["rho"], x["alpha"], var_floor=w.var_floor)

    for it in range(max(3, args.warmup)):
        step(dsets[it % 2])
    torch.cuda.synchronize()
    if gma.gma_get_status():
        raise RuntimeError("device status after warm-up")
    steps = args.steps if args.steps is not None else 200
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(gpu_id_for(local))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    # a GPU spin ahead of the loop lets the host enqueue every step before the GPU reaches them,
    # so each step's events bracket GPU time (one step's kernels take less than its host call)
    torch.cuda._sleep(int(2.0e6 * steps * 0.25))
    for it in range(steps):
        evs[it][0].record(stream)
        step(dsets[it % 2])
        evs[it][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if gma.gma_get_status():
        raise RuntimeError("device status after the timed region")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), device=dev)
    value = whole_job_rate(diag_units(w), world, ms)

    # end to end: Qx uploaded from pinned host memory, p, the statistics and z read back, every step
    hq = [torch.from_numpy(x["Qx"].view(np.int16)).view(torch.bfloat16).pin_memory() for x in host]
    dq = [torch.empty_like(d["Qx"]) for d in dsets]
    hp = torch.empty((w.K,), dtype=torch.float32).pin_memory()
    hs = torch.empty((3,), dtype=torch.float32).pin_memory()
    hz = torch.empty((w.B, w.N), dtype=torch.int32).pin_memory()
    e_steps = 10
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for it in range(e_steps):
        dq[it % 2].copy_(hq[it % 2], non_blocking=True)
        x = dict(dsets[it % 2], Qx=dq[it % 2])
        p, st, z = step(x)
        hp.copy_(p, non_blocking=True)
        hs.copy_(st, non_blocking=True)
        hz.copy_(z, non_blocking=True)
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1) / e_steps, device=dev)
    h2d = hq[0].numel() * 2
    d2h = (w.K + 3 + w.B * w.N) * 4

    pk = peaks()
    rows = w.B * w.H * w.N
    bytes_alg = rows * w.d * 2 + w.B * w.N * 4 + 4 * w.H * (2 * w.K * w.d + w.K)
    flops_alg = rows * 2 * w.K * (2 * w.d + 16)
    t_hbm = bytes_alg / (pk["hbm_gbs"] * 1e9)
    t_tc = flops_alg / (pk["bf16_tflops"] * 1e12)
    achieved = bytes_alg / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
                "kernel": "tc_params + tc_diag + tc_diag_finalize (whole call)", "kernel_ms": ms,
                "peak_source": pk["source"],
                "tensor_frac": flops_alg / (ms / 1e3) / 1e12 / pk["bf16_tflops"]}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, reps, dt = diag_oracle_sample(w, 12.0)
        cpu = {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
               "sample": f"sequence 0, {w.H} heads x the first {n} rows of {w.name}, {reps} calls, one thread"}
    if rank == 0:
        line = {"metric": DIAG_METRIC, "value": value, "unit": "tokens·heads/s", "n_gpus": world,
                "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K,
                           "step": "responsibility diagnostics of the query vectors",
                           "l2": "two alternating input sets of %d MB each" %
                                 (dsets[0]["Qx"].numel() * 2 // 2**20),
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "roofline": roofline, "clocks": clocks, "gpu_launches": 3 * steps,
                "e2e": {"value": whole_job_rate(diag_units(w), world, e2e_ms), "unit": "tokens·heads/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


CROSS_METRIC = "GMA cross-attention query tokens·heads/s (Eq. 5-8, context memory); % of HBM roofline"


def cross_oracle_sample(w, Nkv, seconds):
    """The oracle's cross head on a bounded sample: head 0, the whole context, the first n
    query rows (n doubled until one call takes about `seconds` / 4)."""
    import oracle
    oracle.build()
    q = inputs.gen_all(w.replace(B=1, H=1))
    c = inputs.gen_all(w.replace(B=1, H=1, N=Nkv, seed=w.seed + 1000))
    Q, Ky, Vy = (inputs.widen(a[0, 0], w.dtype) for a in (q["Qx"], c["Kx"], c["V"]))
    n = 256
    while True:
        n = min(n, w.N)
        t0 = time.perf_counter()
        oracle.cross_head(Q[:n], Ky, Vy, q["mu"][0], q["rho"][0], q["alpha"][0], w.var_floor, w.eps)
        if time.perf_counter() - t0 >= seconds / 4 or n == w.N:
            break
        n *= 2
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.cross_head(Q[:n], Ky, Vy, q["mu"][0], q["rho"][0], q["alpha"][0], w.var_floor, w.eps)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return n / dt, n, reps, dt


def run_cross(args, rank, world, local):
    """Cross-attention (sections 3.1, 6): one step is one gma_forward_cross call, the workload's
    queries [B, H, N, d] reading the memory of a context of --context rows (the write over the
    context, the read over the queries)."""
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build
    w = workload(args)
    Nkv = args.context or 4 * w.N
    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, n, reps, dt = cross_oracle_sample(w, Nkv, 12.0)
        sample = f"head 0: the first {n} queries of {w.name} reading a {Nkv}-row context, {reps} calls, one thread"
        print(json.dumps({"impl": "reference", "metric": CROSS_METRIC, "value": rate, "unit": "tokens·heads/s",
                          "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": dt * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": w.name, "context": Nkv,
                                                          "step": "cross-attention (sampled)"},
                          "cpu_baseline": {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": rate, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    sets = []
    for seed in (0, 1):
        q = inputs.gen_all(w.replace(seed=seed))
        c = inputs.gen_all(w.replace(N=Nkv, seed=seed + 1000))
        sets.append({"Qx": to_dev(q["Qx"]), "Ky": to_dev(c["Kx"]), "Vy": to_dev(c["V"]),
                     **{k: to_dev(q[k]) for k in ("mu", "rho", "alpha")}})
    out = torch.empty((w.B, w.H, w.N, w.dv), dtype=sets[0]["Qx"].dtype, device=dev)
    stream = torch.cuda.current_stream()

    def step(x):
        gma.gma_forward_cross(x["Qx"], x["Ky"], x["Vy"], x["mu"], x["rho"], x["alpha"], eps=w.eps,
                              var_floor=w.var_floor, out=out)

    for it in range(max(3, args.warmup)):
        step(sets[it % 2])
    torch.cuda.synchronize()
    if gma.gma_get_status():
        raise RuntimeError("device status after warm-up")
    steps = args.steps if args.steps is not None else 100
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(gpu_id_for(local))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    torch.cuda._sleep(int(2.0e6 * 20))                     # let the host enqueue ahead of the GPU
    for it in range(steps):
        evs[it][0].record(stream)
        step(sets[it % 2])
        evs[it][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if gma.gma_get_status():
        raise RuntimeError("device status after the timed region")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), device=dev)
    units = w.B * w.H * w.N
    value = whole_job_rate(units, world, ms)
    pk = peaks()
    e = 2
    bytes_alg = w.B * w.H * (w.N * e * (w.d + w.dv) + Nkv * e * (w.d + w.dv))
    achieved = bytes_alg / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": None,
                "kernel": "tc_params + tc_write + tc_reduce + tc_read (whole call)", "kernel_ms": ms,
                "peak_source": pk["source"]}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, reps, dt = cross_oracle_sample(w, Nkv, 12.0)
        cpu = {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
               "sample": f"head 0: the first {n} queries of {w.name} reading a {Nkv}-row context, {reps} calls"}
    if rank == 0:
        print(json.dumps({"metric": CROSS_METRIC, "value": value, "unit": "tokens·heads/s", "n_gpus": world,
                          "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic",
                          "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "context": Nkv, "d": w.d,
                                     "K": w.K, "dv": w.dv, "step": "cross-attention forward",
                                     "l2": "two alternating input sets",
                                     "parallelism": "replicas" if world > 1 else "single GPU"},
                          "roofline": roofline, "clocks": clocks, "gpu_launches": 4 * steps,
                          "cpu_baseline": cpu}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


DECODE_METRIC = "GMA causal decode token·heads/s (one new token per head, carried state, Eq. 6b/8b)"


def decode_oracle_sample(w, seconds):
    """The oracle's causal recurrence, one token per head (sampled: 16 heads), timed as the
    cost of extending a sequence by one position from its memory."""
    import oracle
    oracle.build()
    x = inputs.gen_all(w.replace(B=1, H=min(w.H, 16), N=1))
    H = x["Qx"].shape[1]
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for h in range(H):
            oracle.forward_head(*(inputs.widen(x[n][0, h], w.dtype) for n in ("Qx", "Kx", "V")), x["mu"][h],
                                x["rho"][h], x["alpha"][h], w.var_floor, w.eps, True)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return H / dt, H, reps, dt


def run_decode(args, rank, world, local):
    """Causal decode (section 3.5): one step is one gma_decode call appending one token to every
    head of the workload (B x H heads) from a carried state."""
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build
    w = workload(args)
    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, H, reps, dt = decode_oracle_sample(w, 5.0)
        print(json.dumps({"impl": "reference", "metric": DECODE_METRIC, "value": rate, "unit": "tokens·heads/s",
                          "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": dt * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": w.name, "step": "decode (sampled)"},
                          "cpu_baseline": {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
                                           "sample": f"{H} heads, one token each, {reps} passes"},
                          "e2e": {"value": rate, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    steps = args.steps if args.steps is not None else 500
    x = inputs.gen_all(w.replace(N=steps + 8))

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    d = {n: to_dev(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")}
    toks = [{n: d[n][:, :, t:t + 1].contiguous() for n in ("Qx", "Kx", "V")} for t in range(steps + 8)]
    state = torch.zeros((w.B, w.H, w.K, w.dv + 1), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.H, 1, w.dv), dtype=d["Qx"].dtype, device=dev)
    stream = torch.cuda.current_stream()

    def step(t):
        gma.gma_decode(toks[t]["Qx"], toks[t]["Kx"], toks[t]["V"], d["mu"], d["rho"], d["alpha"], state,
                       eps=w.eps, var_floor=w.var_floor, out=out)

    for t in range(8):                                     # warm-up: the first 8 tokens
        step(t)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(gpu_id_for(local))
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    torch.cuda._sleep(int(2.0e6 * 40))                     # let the host enqueue ahead of the GPU
    for t in range(steps):
        evs[t][0].record(stream)
        step(8 + t)
        evs[t][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if gma.gma_get_status():
        raise RuntimeError("device status after the timed region")
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    pk = peaks()
    e = 2 if w.dtype == "bf16" else 4
    bytes_alg = w.B * w.H * (2 * 4 * w.K * (w.dv + 1) + e * (2 * w.d + 2 * w.dv)) + 4 * w.H * w.K * (2 * w.d + 1)
    achieved = bytes_alg / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        rate, H, reps, dt = decode_oracle_sample(w, 5.0)
        cpu = {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
               "sample": f"{H} heads, one token each, {reps} passes"}
    print(json.dumps({"metric": DECODE_METRIC, "value": w.B * w.H / (ms / 1e3), "unit": "tokens·heads/s",
                      "n_gpus": 1, "steps": steps, "warmup": 8, "ms_per_step": ms, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                      "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "K": w.K, "dv": w.dv,
                                 "step": "decode one token per head (median call time)"},
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                   "frac": achieved / pk["hbm_gbs"], "traffic": None,
                                   "kernel": "decode (one launch)", "kernel_ms": ms,
                                   "peak_source": pk["source"]},
                      "clocks": clocks, "gpu_launches": steps, "cpu_baseline": cpu}), flush=True)
    return 0


BWD_METRIC = "GMA {} backward token·heads/s (gradients of Qx, Kx, V, mu, rho, alpha; section 4.1)"


def bwd_flops_per_row(w):
    """fp32 flops the backward kernels compute per row of one head (2 per multiply-add; the
    masked 64 x 64 tile products of the causal passes counted in full)."""
    sc = 2 * 2 * w.d * w.K                                   # scores [x, x^2] . W
    mem = sc + 2 * w.K * (w.dv + 1)                          # memory pass
    rows = 4 * w.K * w.d + 4 * w.K * w.d                     # dX (two products) + parameter sums
    if not w.causal:                                         # the key pass reuses the memory pass's gamma^K
        qry = sc + 4 * w.K * w.dv + 2 * w.K * (w.dv + 1) + rows
        key = 4 * w.K * w.dv + rows
        return mem + qry + key
    t = 2 * 64                                               # one 64-row tile product per row, per K/dv column
    qry = sc + t * w.K + 2 * w.K * w.dv + t * w.dv + t * w.dv + 2 * w.dv * w.K + t * w.K \
        + 2 * w.K * w.dv + 2 * w.K * w.dv                    # gamma^Q, A, num, Bm, g^Q, [R | r] totals, state update
    key = t * w.dv + t * w.K + 2 * w.dv * w.K + t * w.K + t * w.dv + 2 * w.K * w.dv \
        + 2 * w.K * w.dv                                     # Ct, g^K, Dt, dV, state update (stored gammas)
    return mem + qry + key + 2 * rows


def bwd_general_flops_per_row(w, C=16):
    """fp32 flops the general backward path computes per row of one head (2 per multiply-add),
    for shapes other than d = dv = K = 64: the responsibilities of both sides (3 flops per
    component and coordinate), the memory, [num | den], g^Q, [R | r], g^K and dV products, dx
    and the parameter sums; the causal walks add their chunk products (C rows, counted in
    full) and the running-state updates in place of the bidirectional row-times-matrix tiles."""
    K, d, dv, W = w.K, w.d, w.dv, w.dv + 1
    common = 2 * 3 * K * d + 2 * K * W + 2 * (2 * K * 2 * d) + 2 * (2 * K * (2 * d + 1)) + 2 * K * W
    if not w.causal:
        return common + 2 * K * W + 2 * W * K + 2 * W * K + 2 * K * dv
    qry = 2 * C * K + 2 * K * W + 2 * C * W + 2 * C * W + 2 * W * K + 2 * C * K + 2 * K * W
    key = 2 * C * K + 2 * C * W + 2 * W * K + 2 * C * K + 2 * K * dv + 2 * C * dv + 2 * K * W
    return common + qry + key


def bwd_simt64_path(w):
    """Whether gma_backward takes the CUDA-core kernels specialised to d = dv = K = 64."""
    return w.d == 64 and w.dv == 64 and w.K == 64 and not bwd_tc_path(w)


def bwd_tc_path(w):
    """Whether gma_backward takes the tensor-core passes for this workload (bidirectional,
    bf16, d = dv = K = 64, more than one 128-row tile per head)."""
    return (not w.causal and w.dtype == "bf16" and w.d == 64 and w.dv == 64 and w.K == 64 and w.N > 128)


def bwd_bytes_per_row(w):
    """Bytes one row of one head must move at the least: the bf16 inputs Qx, Kx, V and dO read
    once, the fp32 gradients dQx, dKx, dV written once."""
    return 2 * (2 * w.d + 2 * w.dv) + 4 * (2 * w.d + w.dv)


def bwd_tc_flops_per_row(w):
    """Tensor-core flops of the tensor-core passes per row of one head (2 per multiply-add):
    the write pass (log-density and [V | 1]^T Gamma), and per query and key row the
    log-density, the two-term memory products, [a | b]^T Gamma (queries), dx and [x | x^2]^T ds."""
    ld = 2 * (2 * w.d + 16) * w.K                     # [x, x^2/256] . W plus the constant k-step
    write = ld + 2 * 128 * w.K
    qry = ld + 2 * 2 * w.K * 80 + 2 * 2 * 80 * w.K + 2 * 128 * w.K + 2 * w.K * 2 * w.d + 2 * 128 * w.K
    key = ld + 2 * 2 * 80 * w.K + 2 * 2 * w.K * w.dv + 2 * w.K * 2 * w.d + 2 * 128 * w.K
    return write + qry + key


def bwd_oracle_sample(w, seconds):
    """The oracle's backward of whole heads of the workload (one thread), repeated for about
    ``seconds``."""
    import oracle
    oracle.build()
    x = inputs.gen_all(w.replace(B=1, H=1))
    z = inputs.normal(inputs.stream_key(w.seed, "dO"), 0, w.N * w.dv).reshape(w.N, w.dv)
    dO = inputs.widen(inputs.f32_to_bf16_bits(z.astype(np.float32)), "bf16") if w.dtype == "bf16" else z
    reps, t0 = 0, time.perf_counter()
    while reps == 0 or time.perf_counter() - t0 < seconds:
        oracle.backward_head(*(inputs.widen(x[n][0, 0], w.dtype) for n in ("Qx", "Kx", "V")), x["mu"][0],
                             x["rho"][0], x["alpha"][0], w.var_floor, w.eps, w.causal, dO)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return w.N / dt, reps, dt


def run_backward(args, rank, world, local):
    """Backward pass (section 4.1): one step is one gma_backward call over the workload's
    B x H heads (bidirectional), from the inputs and dL/dO to every gradient."""
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build
    w = workload(args).replace(causal=args.direction == "backward_causal")
    metric = BWD_METRIC.format("causal" if w.causal else "bidirectional")
    if args.impl == "reference":
        if rank != 0:
            return 0
        rate, reps, dt = bwd_oracle_sample(w, 12.0)
        print(json.dumps({"impl": "reference", "metric": metric, "value": rate, "unit": "tokens·heads/s",
                          "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": dt * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": w.name, "step": "backward (sampled)"},
                          "cpu_baseline": {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
                                           "sample": f"one head of {w.name} (N = {w.N}), {reps} passes"},
                          "e2e": {"value": rate, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    sets = []
    for seed in (0, 1):
        x = inputs.gen_all(w.replace(seed=seed))
        z = inputs.normal(inputs.stream_key(seed, "dO"), 0, w.B * w.H * w.N * w.dv).astype(np.float32)
        x["dO"] = (inputs.f32_to_bf16_bits(z) if w.dtype == "bf16" else z).reshape(w.B, w.H, w.N, w.dv)
        sets.append({k: to_dev(x[k]) for k in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")})
    f32 = dict(dtype=torch.float32, device=dev)
    grads = (torch.empty((w.B, w.H, w.N, w.d), **f32), torch.empty((w.B, w.H, w.N, w.d), **f32),
             torch.empty((w.B, w.H, w.N, w.dv), **f32), torch.empty((w.H, w.K, w.d), **f32),
             torch.empty((w.H, w.K, w.d), **f32), torch.empty((w.H, w.K), **f32))
    stream = torch.cuda.current_stream()

    def step(x):
        gma.gma_backward(x["Qx"], x["Kx"], x["V"], x["mu"], x["rho"], x["alpha"], x["dO"], eps=w.eps,
                         var_floor=w.var_floor, causal=w.causal, grads=grads)

    warm = max(3, args.warmup)
    for it in range(warm):
        step(sets[it % 2])
    torch.cuda.synchronize()
    if gma.gma_get_status():
        raise RuntimeError("device status after warm-up")
    steps = args.steps if args.steps is not None else 20
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(gpu_id_for(local))
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for it in range(steps):
        evs[it][0].record(stream)
        step(sets[it % 2])
        evs[it][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if gma.gma_get_status():
        raise RuntimeError("device status after the timed region")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    units = w.B * w.H * w.N
    tc = bwd_tc_path(w)
    launches = 9
    if tc:
        # tensor-core passes: bound by the bytes the call must move (HBM); the tensor-pipe
        # fraction beside it
        pk = peaks()
        achieved = units * bwd_bytes_per_row(w) / (ms / 1e3) / 1e9
        tflops = units * bwd_tc_flops_per_row(w) / (ms / 1e3) / 1e12
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": None,
                "kernel": f"gma_backward (whole call: {launches} launches)", "kernel_ms": ms,
                "bytes_per_row": bwd_bytes_per_row(w), "peak_source": pk["source"],
                "tensor": {"achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": tflops / pk["bf16_tflops"], "flops_per_row": bwd_tc_flops_per_row(w)}}
    else:
        per_row = bwd_flops_per_row(w) if bwd_simt64_path(w) else bwd_general_flops_per_row(w)
        flops = units * per_row
        alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12        # fp32 lanes x 2 flops x max SM clock, TFLOP/s
        achieved = flops / (ms / 1e3) / 1e12
        launches = (9 if w.causal else 7) if bwd_simt64_path(w) else (17 if w.causal else 22)
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": None,
                "kernel": f"gma_backward (whole call: {launches} launches)", "kernel_ms": ms,
                "flops_per_row": per_row, "peak_source": "fp32 lanes x 2 x 2070 MHz"}
    cpu = None
    if not args.no_cpu_baseline:
        rate, reps, dt = bwd_oracle_sample(w, 12.0)
        cpu = {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
               "sample": f"one head of {w.name} (N = {w.N}), {reps} passes"}
    print(json.dumps({"metric": metric, "value": units / (ms / 1e3), "unit": "tokens·heads/s", "n_gpus": 1,
                      "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if tc else "f32",
                      "data": "synthetic",
                      "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K, "dv": w.dv,
                                 "inputs": w.dtype,
                                 "step": f"{'causal' if w.causal else 'bidirectional'} backward, all gradients",
                                 "path": "tensor-core passes" if tc else ("CUDA-core passes (fp32)" if bwd_simt64_path(w)
                                                                          else "general CUDA-core path (fp32)"),
                                 "l2": "two alternating input sets (> 129 MB L2)", "parallelism": "single GPU"},
                      "roofline": roof,
                      "clocks": clocks, "gpu_launches": launches * steps, "cpu_baseline": cpu}),
          flush=True)
    return 0


PROJ_METRIC = "GMA Q/K/V projection token·heads/s (Eq. 4, bf16, model width H d)"


def run_project(args, rank, world, local):
    """Input projections (Eq. 4): one step is one gma_project call producing Qx, Kx and V of
    every head of the workload from X [B, N, D], D = H d (the model width of a layer whose
    heads split it evenly: a reading, the configurations give no D)."""
    import torch
    import gaussian_mixture_latent_gb300 as gma
    from gaussian_mixture_latent_gb300 import _build
    w = workload(args)
    D = w.H * w.d
    flops_per_row = 2 * D * w.H * (2 * w.d + w.dv)            # one token, every head
    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        rows = 64
        x = inputs.normal(inputs.stream_key(0, "X"), 0, rows * D).reshape(1, rows, D)
        ws = [inputs.normal(inputs.stream_key(0, n), 0, w.H * D * c).reshape(w.H, D, c) / D ** 0.5
              for n, c in (("Wq", w.d), ("Wk", w.d), ("Wv", w.dv))]
        reps, t0 = 0, time.perf_counter()
        while reps == 0 or time.perf_counter() - t0 < 10.0:
            oracle.project(x, *ws)
            reps += 1
        dt = (time.perf_counter() - t0) / reps
        rate = rows * w.H / dt
        print(json.dumps({"impl": "reference", "metric": PROJ_METRIC, "value": rate, "unit": "tokens·heads/s",
                          "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": dt * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": w.name, "D": D, "step": "projection (sampled)"},
                          "cpu_baseline": {"value": rate, "unit": "tokens·heads/s", "cores": 1, "kind": "oracle",
                                           "sample": f"{rows} rows of X, {reps} passes"},
                          "e2e": {"value": rate, "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()

    def gen(seed, name, shape, std):
        z = inputs.normal(inputs.stream_key(seed, name), 0, int(np.prod(shape))).reshape(shape) * std
        return torch.from_numpy(inputs.f32_to_bf16_bits(z.astype(np.float32)).view(np.int16)).view(
            torch.bfloat16).to(dev)

    sets = [(gen(seed, "X", (w.B, w.N, D), 1.0), gen(seed, "Wq", (w.H, D, w.d), D ** -0.5),
             gen(seed, "Wk", (w.H, D, w.d), D ** -0.5), gen(seed, "Wv", (w.H, D, w.dv), D ** -0.5))
            for seed in (0, 1)]
    bf = dict(dtype=torch.bfloat16, device=dev)
    outs = (torch.empty((w.B, w.H, w.N, w.d), **bf), torch.empty((w.B, w.H, w.N, w.d), **bf),
            torch.empty((w.B, w.H, w.N, w.dv), **bf))
    stream = torch.cuda.current_stream()
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)

    def step(x):
        gma.gma_project(*x, out=outs, workspace=ws)

    warm = max(3, args.warmup)
    for it in range(warm):
        step(sets[it % 2])
    torch.cuda.synchronize()
    if gma.gma_get_status(ws):
        raise RuntimeError("device status after warm-up")
    steps = args.steps if args.steps is not None else 20
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(gpu_id_for(local))
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for it in range(steps):
        evs[it][0].record(stream)
        step(sets[it % 2])
        evs[it][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if gma.gma_get_status(ws):
        raise RuntimeError("device status after the timed region")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    rows = w.B * w.N
    pk = peaks()
    tflops = rows * flops_per_row / (ms / 1e3) / 1e12
    hbm = rows * 2 * (D + w.H * (2 * w.d + w.dv)) / (ms / 1e3) / 1e9      # X read once, outputs written once
    print(json.dumps({"metric": PROJ_METRIC, "value": rows * w.H / (ms / 1e3), "unit": "tokens·heads/s",
                      "n_gpus": 1, "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": w.name, "B": w.B, "N": w.N, "D": D, "H": w.H, "d": w.d, "dv": w.dv,
                                 "step": "gma_project (one launch)",
                                 "l2": "two alternating input sets (> 129 MB L2)", "parallelism": "single GPU"},
                      "roofline": {"bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops"],
                                   "unit": "TFLOP/s", "frac": tflops / pk["bf16_tflops"], "traffic": None,
                                   "kernel": "proj_kernel", "kernel_ms": ms, "flops_per_row": flops_per_row,
                                   "peak_source": pk["source"],
                                   "hbm": {"achieved": hbm, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                           "frac": hbm / pk["hbm_gbs"]}},
                      "clocks": clocks, "gpu_launches": steps, "cpu_baseline": None}), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.direction == "decode":
        return run_decode(args, rank, world, local)
    if args.direction == "diagnostics":
        return run_diagnostics(args, rank, world, local)
    if args.direction == "cross":
        return run_cross(args, rank, world, local)
    if args.direction in ("backward", "backward_causal"):
        return run_backward(args, rank, world, local)
    if args.direction == "project":
        return run_project(args, rank, world, local)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gpu(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
