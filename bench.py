"""Benchmark of the fused CFG sampler step on one B300 (or N replicas under torchrun).

A "step" is one call of the fused step kernel: rel-MAE + schedule update +
guidance + DDIM/Euler update over the whole latent of one batch.  The
default workload is the largest: the video latent 2x16x13x90x160 (bf16
storage, 50-step DDIM, eta = 0, w = 6).  Inputs are synthetic and resident in
HBM; the steps rotate over enough buffer sets that every step's inputs come
from HBM (not the 126 MB L2).  K steps form one CUDA graph with programmatic
dependent launch (K = --steps rounded up to a multiple of itself of at least
100: a graph boundary costs about one step); --replays (>= 10) such graphs run
back to back, each timed by CUDA events, and the line reports the median
per-step time.

Prints ONE JSON line (rank 0):
  value / unit       latent elements per second per step, whole job
  roofline           algorithmic HBM bytes / measured step time vs the measured copy peak
  e2e                the same metric through the public Python API with pinned host
                     buffers, host->device and device->host copies inside the timed region
  cpu_baseline       the CPU oracle timed on a bounded sample, the host's core count and CPU
                     model, and one whole oracle run on a slice of the latent (rank 0, N = 1)
  sweep              the same device measurement on every other workload, the eta = 1
                     workload at eta = 0 (its noise-free floor), and the default workload as a
                     batched call with a schedule per sample (rank 0, N = 1)
  sampler_run        whole runs of every workload through the public API with a synthetic
                     denoiser, as a captured CUDA graph, with the denoiser alone timed the same
                     way; the default workload also as the eager host loop and with two branch
                     streams (rank 0, N = 1)

``--impl reference`` times the CPU oracle instead (the slow reference program)
and prints the same kind of line with ``"impl": "reference"``.

Multi-GPU: the step needs no exchange on one latent per GPU, so N ranks run N
independent replicas (weak scaling): barrier, time, max over ranks.
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
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "video_b2_bf16"
FALLBACK_HBM_GBS = 6400.0
PROFILE_DIR = ROOT / "profiles"
KERNEL_SRC = (ROOT / "cfg_guided_sampler_step_b300" / "csrc" / "cfgstep.cu",
              ROOT / "cfg_guided_sampler_step_b300" / "csrc" / "cfg_noise.cuh")


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only; no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# Peaks, profiles, clocks
# ---------------------------------------------------------------------------
def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001 - absent or unreadable: the documented fallback
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C++/CUDA source with comments, trailing blanks and blank lines removed (the kernel
    sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """sha256[:16] of the step kernel's code (the kernel file, then the noise header; comments
    and blank lines excluded, so a change of wording does not void a profile)."""
    h = hashlib.sha256()
    for f in KERNEL_SRC:
        h.update(code_only(f.read_text()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    f = PROFILE_DIR / f"cfg_step_kernel_{workload}.md"
    if not f.exists():
        return None
    text = f.read_text()
    m_src = re.search(r"kernel source sha256\[:16\][^|\n]*\|\s*`?([0-9a-f]{16})", text)
    m_b = re.search(r"dram bytes per launch \(read \+ write\)\s*\|\s*([0-9][0-9,]*)", text)
    if not m_src or not m_b or m_src.group(1) != kernel_source_hash():
        return None
    return int(m_b.group(1).replace(",", ""))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 11:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
            except (ValueError, IndexError):
                continue
            if self.t0 is not None and not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                continue
            n += 1
            try:
                sm.append(float(f[3]))
                smax.append(float(f[4]))
            except ValueError:
                pass
            for name, val in zip(names, f[7:11]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------
# The device measurement
# ---------------------------------------------------------------------------
def step_plan(wl: W.Workload, cs):
    """Per-step (step index, coefficients) of one sampler run of the workload."""
    N = wl.n_steps
    if wl.mode == "ddim":
        abar = cs.abar_linear(wl.T, wl.beta_start, wl.beta_end)
        ts = cs.ddim_timesteps(N, wl.T)
        return [dict(step=s, abar_t=float(abar[ts[s]]),
                     abar_prev=float(abar[ts[s + 1]]) if s + 1 < N else 1.0) for s in range(N)]
    return [dict(step=s, t_cur=1.0 - s / N, t_next=1.0 - (s + 1) / N) for s in range(N)]


def enqueue_step(cs, wl, bufs, plan_s, ws, st, sp, M=None, batch=1, stream=None, exact=False):
    x, pc, pu = bufs[:3]
    xo = bufs[3] if len(bufs) > 3 else x
    if wl.mode == "ddim":
        cs.ddim_step(xo, x, pc, pu, w=wl.w, abar_t=plan_s["abar_t"], abar_prev=plan_s["abar_prev"],
                     eta=wl.eta, seed=wl.seed, step=plan_s["step"], M_out=M, state=st, sched=sp,
                     workspace=ws, batch=batch, stream=stream, exact_rounding=exact)
    else:
        cs.flow_step(xo, x, pc, pu, w=wl.w, t_cur=plan_s["t_cur"], t_next=plan_s["t_next"],
                     step=plan_s["step"], M_out=M, state=st, sched=sp, workspace=ws, batch=batch,
                     stream=stream, exact_rounding=exact)


def make_sets(wl, n_sets, device, torch):
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    sets = []
    for _ in range(n_sets):
        x = torch.randn(wl.n, generator=g, device=device, dtype=torch.float32).to(dt)
        pu = torch.randn(wl.n, generator=g, device=device, dtype=torch.float32).to(dt)
        pc = (pu.float() + 0.1 * torch.randn(wl.n, generator=g, device=device)).to(dt)
        sets.append((x, pc, pu, torch.empty_like(x)))
    return sets


MIN_GRAPH_STEPS = 100


def graph_length(steps: int) -> int:
    """Steps in one timed graph: `steps` rounded up to a multiple of itself of at least
    MIN_GRAPH_STEPS (a graph boundary costs about one step)."""
    k = max(1, int(steps))
    return k * math.ceil(MIN_GRAPH_STEPS / k)


def replay_plan(K: int, n_sets: int, n_steps: int, max_graphs: int = 400):
    """Distinct K-step graphs needed so that back-to-back replays continue one sequence.

    Step p of the sequence uses buffer set p % n_sets and sampler step p % n_steps, so a
    set is reused only after every other set has passed; graph g covers steps
    [gK, (g+1)K) modulo the period lcm(K, n_sets, n_steps).  Returns (graphs, period).
    """
    period = math.lcm(K, n_sets, n_steps)
    D = period // K
    if D > max_graphs:
        raise SystemExit(f"--steps {K} needs {D} distinct graphs over {n_sets} buffer sets; "
                         f"choose a divisor or multiple of {n_sets}")
    return D, period


def time_device(wl: W.Workload, steps: int, warmup: int, device, world: int, clocks=None,
                sets=None, batch=1, replays: int = 15, eta=None, min_seconds: float = 0.0,
                exact: bool = False):
    """Median per-step time of `replays` timed replays of K fused steps (K = `steps` rounded
    up to a multiple of itself of at least MIN_GRAPH_STEPS).

    The steps rotate over HBM-resident buffer sets (default: >= 4x the L2 in whole sampler
    runs), so every step reads its inputs from HBM.  Each replay is one CUDA graph of K steps
    with programmatic dependent launch; the replays run back to back on one stream and each
    is timed by its own pair of CUDA events, after >= `warmup` untimed steps that also
    replay (and so upload) every graph once.  Consecutive replays continue one sequence of
    sampler steps, so each step's deferred reduction is completed by the next launch as in a
    sampler run.  `sets` overrides the number of buffer sets (fewer only to keep a profiler
    capture small); `batch` > 1 times the batched step; `eta` overrides the workload's eta;
    `min_seconds` raises the replay count until the timed region lasts that long (so the clock
    sampler sees it several times; the line still reports the median replay); `exact` times the
    correctly rounded bf16 steps (CFG_BF16_EXACT).
    """
    import torch
    import cfg_guided_sampler_step_b300 as cs
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    set_bytes = 4 * wl.n * wl.elem_bytes          # x_in, pred_c, pred_u, x_out
    # enough sets for 4x the L2, rounded up to whole sampler runs
    n_sets = max(2, math.ceil(4 * l2 / set_bytes))
    n_sets = wl.n_steps * math.ceil(n_sets / wl.n_steps)
    if sets:
        n_sets = int(sets)
    # A graph boundary costs about one step (programmatic dependent launch does not overlap
    # steps across graph launches: 8.81 / 8.54 / 8.46 / 8.43 us per video step in graphs of
    # 20 / 50 / 100 / 200 steps, measured), so each timed replay is a graph of at least
    # MIN_GRAPH_STEPS steps: `steps` rounded up to a multiple of itself.
    K = graph_length(steps)
    D, period = replay_plan(K, n_sets, wl.n_steps)
    bufs = make_sets(wl, n_sets, device, torch)
    code = cs.CFG_F32 if wl.dtype == "f32" else cs.CFG_BF16
    ws = cs.new_workspace(wl.n, code, device, batch=batch)
    st = cs.new_sched_state(device, batch=batch)
    # as in a sampler run: each step's reduction is completed by the next step's launch
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, tau_cap=wl.tau_cap,
                        defer=True)
    plan = step_plan(wl, cs)
    wl_eta = wl if eta is None else dataclasses.replace(wl, eta=eta)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))

    def enqueue(p):
        enqueue_step(cs, wl_eta, bufs[p % n_sets], plan[p % wl.n_steps], ws, st, sp, batch=batch,
                     stream=s, exact=exact)

    with torch.cuda.stream(s):                      # eager warm-up of the launch path
        for p in range(wl.n_steps):
            enqueue(p)
    torch.cuda.synchronize(device)
    graphs = []
    for g in range(D):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for j in range(K):
                enqueue(g * K + j)
        graphs.append(gr)
    torch.cuda.synchronize(device)
    # warm-up: whole cycles over every graph (each replayed, hence uploaded, once or more)
    cycles = max(1, math.ceil(max(warmup, 3) / (D * K)))
    with torch.cuda.stream(s):
        for _ in range(cycles):
            for gr in graphs:
                gr.replay()
    torch.cuda.synchronize(device)
    cycles_extra = 0
    if min_seconds > 0:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            for gr in graphs:
                gr.replay()
            b.record(s)
        b.synchronize()
        per_replay_s = a.elapsed_time(b) * 1e-3 / len(graphs)
        cycles_extra = D * K
        replays = max(replays, min(20000, math.ceil(min_seconds / max(per_replay_s, 1e-9))))
    # every rank times the same number of replays
    replays = int(max_over_ranks(float(replays), world, device))
    torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    if clocks:
        clocks.mark_begin()
    with torch.cuda.stream(s):
        for r in range(replays):
            ev[r][0].record(s)
            graphs[r % D].replay()
            ev[r][1].record(s)
    ev[-1][1].synchronize()
    torch.cuda.synchronize(device)
    if clocks:
        clocks.mark_end()
    barrier(world)
    with torch.cuda.stream(s):
        cs.workspace_flush(ws, batch=batch)
    torch.cuda.synchronize(device)
    per_step_ms = sorted(a.elapsed_time(b) / K for a, b in ev)
    state = cs.read_sched_state(st)
    return {"ms": statistics.median(per_step_ms) * K, "step_ms_median": statistics.median(per_step_ms),
            "step_ms_min": per_step_ms[0], "step_ms_max": per_step_ms[-1],
            "replays": replays, "graph_steps": K, "distinct_graphs": D,
            "warmup_steps": cycles * D * K + cycles_extra, "n_sets": n_sets, "set_bytes": set_bytes,
            "l2_bytes": l2, "launches": replays * K, "state_flags": state["flags"]}


def time_e2e(wl: W.Workload, steps: int, device, depth: int = 3):
    """Same metric through the public API with pinned host inputs and a host read of each result.

    Every step copies its three inputs host->device, runs the step and copies its result and
    M device->host, all inside the timed region.  As a serving loop would, consecutive steps
    are pipelined over `depth` buffer slots on three streams (uploads, steps, downloads)
    ordered by events, so one step's uploads overlap the previous step's download.  Timed by
    the host's wall clock from an idle device to the last result being on the host.
    """
    import torch
    import cfg_guided_sampler_step_b300 as cs
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    inp = W.draw_prediction_pair(wl.n, wl.dtype, wl.seed)

    def host(a):
        # page-locked buffers from the library's host allocator (cfg_host_alloc)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        t = t.view(dt) if a.dtype == np.uint16 else t
        h = cs.pinned_empty(t.numel(), dt)
        h.copy_(t)
        return h

    hx, hc, hu = host(inp["x"]), host(inp["c"]), host(inp["u"])
    slots = []
    for _ in range(depth):
        dx = torch.empty(wl.n, dtype=dt, device=device)
        slots.append(dict(x=dx, c=torch.empty_like(dx), u=torch.empty_like(dx),
                          M=torch.zeros(1, dtype=torch.float64, device=device),
                          hout=cs.pinned_empty(wl.n, dt),
                          hM=cs.pinned_empty(1, torch.float64),
                          ev_in=torch.cuda.Event(), ev_run=torch.cuda.Event(),
                          ev_out=torch.cuda.Event(), used=False))
    ws = cs.new_workspace(wl.n, cs.CFG_F32 if wl.dtype == "f32" else cs.CFG_BF16, device)
    st = cs.new_sched_state(device)
    # every step finishes its own reduction, so each step's M is complete when read back
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, tau_cap=wl.tau_cap,
                        defer=False)
    plan = step_plan(wl, cs)
    s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
    h_in, h_run, h_out = s_in.cuda_stream, s_run.cuda_stream, s_out.cuda_stream

    def one(i):
        sl = slots[i % depth]
        if sl["used"]:
            s_in.wait_event(sl["ev_out"])             # the slot's last result is on the host
        cs.copy_async(sl["x"], hx, stream=h_in)
        cs.copy_async(sl["c"], hc, stream=h_in)
        cs.copy_async(sl["u"], hu, stream=h_in)
        sl["ev_in"].record(s_in)
        s_run.wait_event(sl["ev_in"])
        enqueue_step(cs, wl, (sl["x"], sl["c"], sl["u"]), plan[i % wl.n_steps], ws, st, sp,
                     M=sl["M"], stream=h_run)
        sl["ev_run"].record(s_run)
        s_out.wait_event(sl["ev_run"])
        cs.copy_async(sl["hout"], sl["x"], stream=h_out)
        cs.copy_async(sl["hM"], sl["M"], stream=h_out)
        sl["ev_out"].record(s_out)
        sl["used"] = True

    for i in range(max(20, 3 * depth)):
        one(i)
    torch.cuda.synchronize(device)
    # wall clock from an idle device to the last result on the host: the host's own work
    # (enqueueing every copy and step) is part of the end-to-end time
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize(device)
    ms = (time.perf_counter() - t0) * 1e3
    eb = wl.elem_bytes
    return {"value": wl.n * steps / (ms * 1e-3), "unit": "latent elements/s",
            "h2d_bytes_per_step": 3 * wl.n * eb, "d2h_bytes_per_step": wl.n * eb + 8,
            "steps": steps, "ms_per_step": ms / steps, "pipeline_depth": depth,
            "host_enqueue_us_per_step": host_s * 1e6 / steps,
            "host_buffers": "page-locked (cfg_host_alloc), copies by cfg_copy_async"}


def time_sampler_runs(wl: W.Workload, device, runs: int = 10, forms: bool = False):
    """Whole sampler runs of the workload through the public API, per denoising step.

    Each step runs a synthetic denoiser (the workload's Gaussian posterior mean, or the flow
    point mass; fp32 torch ops, the model stand-in) for both branches, then the fused step.
    The run is recorded into one CUDA graph (``sampler_run`` under stream capture) and
    replayed; the same denoiser calls without the steps are recorded and replayed too, so
    the step's share is the difference.  With ``forms``, the eager host loop and
    ``sampler_run_branches`` (two branch streams joined by events) are timed as well.
    Microseconds per step, host wall clock around whole runs with the device synchronised.
    """
    import torch
    import cfg_guided_sampler_step_b300 as cs
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    inp = W.draw_inputs(wl)
    reps = wl.n // int(np.prod(wl.mean_shape))
    mc = torch.from_numpy(np.tile(inp["mean_c"].reshape(-1), reps)).to(device)
    mu = torch.from_numpy(np.tile(inp["mean_u"].reshape(-1), reps)).to(device)
    x_T = torch.randn(wl.n, device=device).to(dt)
    x = torch.empty_like(x_T)
    pc, pu = torch.empty_like(x), torch.empty_like(x)
    std2 = wl.data_std * wl.data_std

    def branch(b, step, timestep, t):
        mean, out = (mc, pc) if b == 0 else (mu, pu)
        if wl.mode == "ddim":
            A = math.sqrt(1.0 - t) / (t * std2 + 1.0 - t)
            out.copy_((x.float() - math.sqrt(t) * mean) * A)
        else:
            out.copy_((x.float() - mean) * (1.0 / t))

    def both(step, timestep, t):
        branch(0, step, timestep, t)
        branch(1, step, timestep, t)

    code = cs.CFG_F32 if wl.dtype == "f32" else cs.CFG_BF16
    ws, st = cs.new_workspace(wl.n, code, device), cs.new_sched_state(device)
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, tau_cap=wl.tau_cap)
    kw = dict(mode=cs.CFG_MODE_DDIM if wl.mode == "ddim" else cs.CFG_MODE_FLOW,
              n_steps=wl.n_steps, w=wl.w, pred_c=pc, pred_u=pu, sched=sp, state=st, workspace=ws,
              eta=wl.eta, seed=wl.seed)
    if wl.mode == "ddim":
        abar = cs.abar_linear(wl.T, wl.beta_start, wl.beta_end)
        ts = cs.ddim_timesteps(wl.n_steps, wl.T)
        kw["abar_table"], kw["timesteps"] = abar, ts
        ts_args = [(s_, int(ts[s_]), float(abar[ts[s_]])) for s_ in range(wl.n_steps)]
    else:
        ts_args = [(s_, s_, 1.0 - s_ / wl.n_steps) for s_ in range(wl.n_steps)]
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    sc, su = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def full():
        x.copy_(x_T)
        cs.sampler_run(x, denoise=both, **kw)

    def denoiser_only():
        x.copy_(x_T)
        for a in ts_args:
            both(*a)

    def branches():
        x.copy_(x_T)
        cs.sampler_run_branches(x, denoise_branch=branch, stream_c=sc, stream_u=su, **kw)

    def wall(fn):
        with torch.cuda.stream(s):
            fn()
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            for _ in range(runs):
                fn()
            torch.cuda.synchronize(device)
        return (time.perf_counter() - t0) / runs / wl.n_steps * 1e6

    def graph(fn):
        with torch.cuda.stream(s):
            fn()                                    # warm-up outside capture
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        return wall(g.replay)

    res = {"graph_us_per_step": graph(full), "denoiser_graph_us_per_step": graph(denoiser_only)}
    res["step_us_per_step"] = res["graph_us_per_step"] - res["denoiser_graph_us_per_step"]
    if forms:
        res["eager_us_per_step"] = wall(full)
        res["branch_streams_us_per_step"] = wall(branches)
    return res


# ---------------------------------------------------------------------------
# The oracle (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step_fn(wl: W.Workload, n_sample: int):
    """One oracle step of the workload on the first n_sample elements (stored inputs)."""
    from oracle import cfg_oracle as O
    inp = W.draw_prediction_pair(n_sample, wl.dtype, wl.seed)
    x = W.stored_to_f64(inp["x"], wl.dtype)
    c = W.stored_to_f64(inp["c"], wl.dtype)
    u = W.stored_to_f64(inp["u"], wl.dtype)
    if wl.mode == "ddim":
        abar = O.abar_linear(wl.T, wl.beta_start, wl.beta_end)
        ts = O.ddim_timesteps(wl.n_steps, wl.T)
        sched = [(float(abar[ts[s]]), float(abar[ts[s + 1]]) if s + 1 < wl.n_steps else 1.0)
                 for s in range(wl.n_steps)]

        def fn(i):
            s = i % wl.n_steps
            ab, abp = sched[s]
            return O.ddim_step(x, c, u, wl.dtype, wl.w, ab, abp, wl.eta, wl.seed, s,
                               last=(s == wl.n_steps - 1))
    else:
        t = O.flow_times(wl.n_steps)

        def fn(i):
            s = i % wl.n_steps
            return O.flow_step(x, c, u, wl.dtype, wl.w, float(t[s]), float(t[s + 1]))
    return fn


def time_oracle(wl: W.Workload, steps: int, warmup: int, budget_s: float):
    """Time `steps` oracle steps, each on a sample sized so the run fits in about budget_s."""
    probe_n = min(wl.n, 1 << 16)
    fn = oracle_step_fn(wl, probe_n)
    t0 = time.perf_counter()
    fn(0)
    t_probe = time.perf_counter() - t0
    fn_small = oracle_step_fn(wl, 64)
    t0 = time.perf_counter()
    for i in range(5):
        fn_small(i)
    t_fixed = (time.perf_counter() - t0) / 5
    per_elem = max((t_probe - t_fixed) / probe_n, 1e-10)
    per_step_budget = budget_s / max(steps + warmup, 1)
    n_sample = int((per_step_budget - t_fixed) / per_elem)
    n_sample = max(64, min(wl.n, n_sample))
    fn = oracle_step_fn(wl, n_sample)
    for i in range(warmup):
        fn(i)
    t0 = time.perf_counter()
    for i in range(steps):
        fn(i)
    dt = time.perf_counter() - t0
    return {"value": n_sample * steps / dt, "n_sample": n_sample, "seconds": dt, "steps": steps}


def oracle_threads() -> int:
    # numpy elementwise ufuncs and np.sum run on one thread; no BLAS call is on this path
    return 1


def time_randn(n: int, launches: int, warmup: int, device):
    """The eta noise alone: `launches` cfg_randn calls of n normals, replayed from CUDA graphs.

    The step kernel draws the same Philox4x32-10 + Box-Muller stream in registers; this
    isolates its ALU cost (the output is 4n bytes, written once per launch).
    """
    import torch
    import cfg_guided_sampler_step_b300 as cs
    out = torch.empty(max(n, 1), dtype=torch.float32, device=device)
    G = max(1, min(100, launches))
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for j in range(warmup):
            cs.randn(out[:n], seed=7, step=j, stream=s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for j in range(G):
            cs.randn(out[:n], seed=7, step=j, stream=s)
    reps = max(1, launches // G)
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):              # a graph replays on the current stream
        ev0.record(s)
        for _ in range(reps):
            g.replay()
        ev1.record(s)
    ev1.synchronize()
    us = ev0.elapsed_time(ev1) * 1e3 / (reps * G)
    return {"kernel": "randn_kernel", "normals": n, "launches": reps * G, "us_per_launch": us,
            "g_normals_per_s": n / us * 1e-3}


# ---------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100,
                    help="steps per timed replay (one CUDA graph), rounded up to a multiple of "
                         f"itself of at least {MIN_GRAPH_STEPS}; the line reports the median "
                         "per-step time over --replays replays")
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--replays", type=int, default=15)
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="more replays until the timed region lasts this long (clock samples)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="cfgstep", choices=["cfgstep", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--sweep-steps", type=int, default=100)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sets", type=int, default=None,
                    help="buffer sets to rotate over (default: >= 4x L2); fewer only for profiling")
    ap.add_argument("--eta", type=float, default=None,
                    help="override the workload's DDIM eta (e.g. 0 for the noise-free floor)")
    ap.add_argument("--randn", type=int, default=None, metavar="N",
                    help="time only the eta-noise stream (cfg_randn, N normals per launch) and exit")
    args = ap.parse_args(argv)
    if args.replays < 10:
        ap.error("--replays must be >= 10 (the line reports a median over replays)")
    world, rank, local = dist_env()
    wl = W.WORKLOADS[args.workload]
    if args.eta is not None:
        wl = dataclasses.replace(wl, eta=args.eta)
    warmup = max(args.warmup, 3)
    metric = "latent elements/s per CFG sampler step"
    unit = "latent elements/s"

    if args.impl == "reference":
        if rank != 0:
            return 0
        budget = min(150.0, 20.0 + 1e-4 * (args.steps + warmup))
        r = time_oracle(wl, args.steps, warmup, budget)
        sample = (f"oracle step (fp64 NumPy: rel-MAE, guidance, {wl.mode} update, {wl.dtype} "
                  f"rounding) on {r['n_sample']} of the {wl.n} latent elements per step")
        line = {"impl": "reference", "metric": metric, "value": r["value"], "unit": unit,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
                "ms_per_step": 1e3 * r["seconds"] / max(args.steps, 1), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_config(wl),
                "cpu_baseline": {"value": r["value"], "unit": unit, "cores": oracle_threads(),
                                 "kind": "oracle", "sample": sample, "host": host_info()},
                "e2e": {"value": r["value"], "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    import cfg_guided_sampler_step_b300 as cs  # noqa: F401  (fails loudly if not built)
    if args.randn is not None:
        if rank == 0:
            print(json.dumps(time_randn(args.randn, args.steps, warmup, device)), flush=True)
        return 0

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:  # noqa: BLE001
        uuid = None
    clocks = ClockSampler(uuid) if rank == 0 else None
    if clocks:
        clocks.start()
    dev = time_device(wl, args.steps, warmup, device, world, clocks, sets=args.sets,
                      replays=args.replays, min_seconds=args.min_seconds)
    clk = clocks.stop() if clocks else None
    # the job's per-step time is its slowest rank's; every rank processes one latent per step
    step_s = max_over_ranks(dev["step_ms_median"], world, device) * 1e-3
    total_elems = sum_over_ranks(float(wl.n), world, device)
    value = total_elems / step_s
    peak, peak_kind = hbm_peak()
    achieved = wl.bytes_per_step / (dev["step_ms_median"] * 1e-3) / 1e9
    e2e = time_e2e(wl, args.e2e_steps, device)
    e2e_v = sum_over_ranks(e2e["value"], world, device)
    if rank != 0:
        return 0
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": dev["warmup_steps"], "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(wl), parallelism=f"replicas{world}",
                       l2=f"rotating {dev['n_sets']} buffer sets of {dev['set_bytes']} B "
                          f"({dev['n_sets'] * dev['set_bytes'] / 2**20:.0f} MiB; the L2 holds "
                          f"{dev['l2_bytes'] / 2**20:.0f} MiB), inputs larger than L2",
                       launch=f"CUDA graphs of {dev['graph_steps']} steps, programmatic dependent "
                              f"launch",
                       timing=f"median over {dev['replays']} back-to-back replays of a "
                              f"{dev['graph_steps']}-step graph (--steps {args.steps} rounded up "
                              f"to a multiple of at least {MIN_GRAPH_STEPS}: a graph boundary "
                              f"costs about one step), each timed by CUDA events; "
                              f"per-step min {dev['step_ms_min'] * 1e3:.3f} us, max "
                              f"{dev['step_ms_max'] * 1e3:.3f} us"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(wl.name),
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.4 TB/s",
                     "algorithmic_bytes_per_launch": wl.bytes_per_step,
                     "frac_of_8tbs_spec": achieved / 8000.0},
        "e2e": {"value": e2e_v, "unit": e2e["unit"], "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "us_per_step": e2e["ms_per_step"] * 1e3,
                "pipeline": f"{e2e['pipeline_depth']} buffer slots; upload, step and download "
                            "streams ordered by events",
                "timer": "host wall clock, device synchronised at both ends",
                "host_buffers": e2e["host_buffers"],
                "host_enqueue_us_per_step": e2e["host_enqueue_us_per_step"]},
        "gpu_launches": dev["launches"],
        "clocks": clk,
    }
    if world == 1 and not args.no_sweep:
        line["sampler_run"] = {name: time_sampler_runs(W.WORKLOADS[name], device,
                                                       forms=(name == wl.name))
                               for name in W.WORKLOAD_ORDER}
        line["sampler_run"]["denoiser"] = ("synthetic posterior-mean / flow point-mass denoiser, "
                                           "fp32 torch ops, both branches")
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if world == 1 and not args.no_sweep:
        line["sweep"] = sweep(wl, args.sweep_steps, args.replays, device, peak)
    print(json.dumps(line), flush=True)
    return 0


def sweep(wl: W.Workload, steps: int, replays: int, device, peak: float):
    """The same device measurement on every other workload, the 3840px workload without noise
    (eta = 0, its floor), the default workload as a batched call with a rel-MAE and schedule
    per sample, and every bf16 workload with correctly rounded steps (CFG_BF16_EXACT)."""
    out = {}

    def row(w2, **kw):
        d2 = time_device(w2, steps, 100, device, 1, replays=replays, **kw)
        s = d2["step_ms_median"] * 1e-3
        return {"value": w2.n / s, "us_per_step": s * 1e6,
                "us_per_step_min": d2["step_ms_min"] * 1e3,
                "achieved_gbs": w2.bytes_per_step / s / 1e9,
                "frac": w2.bytes_per_step / s / 1e9 / peak}

    for name in W.WORKLOAD_ORDER:
        w2 = W.WORKLOADS[name]
        if name != wl.name:
            out[name] = dict(row(w2), traffic=profiled_traffic(name))
        if w2.eta > 0:
            out[f"{name}/eta0"] = row(w2, eta=0.0)
    if wl.shape[0] > 1:
        out[f"{wl.name}/per_sample"] = dict(row(wl, batch=wl.shape[0]), batch=wl.shape[0])
    for name in W.WORKLOAD_ORDER:
        if W.WORKLOADS[name].dtype == "bf16":
            out[f"{name}/exact"] = row(W.WORKLOADS[name], exact=True)
    return out


def slice_shape(shape, n_target: int):
    """The leading slice of `shape` (fewer samples, channels, frames ...) with at most
    n_target elements, keeping at least the last axis."""
    shape = list(shape)
    for i in range(len(shape) - 1):
        if int(np.prod(shape)) <= n_target:
            break
        rest = int(np.prod(shape[i + 1:]))
        shape[i] = max(1, min(shape[i], n_target // rest))
    return tuple(shape)


def host_info():
    model = None
    try:
        for line in Path("/proc/cpuinfo").read_text().splitlines():
            if line.startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def cpu_baseline(wl: W.Workload, seconds: float):
    """The oracle's step on the full latent, repeated for about `seconds` on one host core,
    and one whole oracle run (denoiser and steps) on a slice of the latent."""
    from oracle import cfg_oracle as O
    fn = oracle_step_fn(wl, wl.n)
    fn(0)
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn(reps)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    # a whole run on a leading slice of the latent sized for about `seconds`, from the rate
    # of a probe run on a small slice
    def run(shape):
        sl = wl.scaled(shape)
        inp = W.draw_inputs(sl)
        pert = (lambda s_, b: W.draw_perturbation(sl, s_, b)) if sl.perturb_std else None
        t0 = time.perf_counter()
        O.run_sampler(sl, inp, perturb=pert)
        return sl, time.perf_counter() - t0

    probe, t_probe = run(slice_shape(wl.shape, 1 << 16))
    n_target = int(seconds * probe.n / max(t_probe, 1e-6))
    sl, run_s = run(slice_shape(wl.shape, max(probe.n, n_target)))
    shape = sl.shape
    return {"value": wl.n * reps / dt, "unit": "latent elements/s", "cores": oracle_threads(),
            "kind": "oracle",
            "sample": f"{reps} oracle steps (fp64 NumPy) on the full {wl.n}-element latent, {dt:.1f} s",
            "host": host_info(),
            "full_run": {"shape": list(shape), "n": sl.n, "steps": sl.n_steps,
                         "seconds": run_s, "latent_elements_per_s": sl.n * sl.n_steps / run_s,
                         "what": "oracle run_sampler: synthetic denoiser and step, every step"}}


def workload_config(wl: W.Workload):
    return {"workload": wl.name, "shape": list(wl.shape), "n": wl.n, "storage": wl.dtype,
            "sampler": (f"DDIM eta={wl.eta} {wl.n_steps} steps" if wl.mode == "ddim"
                        else f"Euler flow {wl.n_steps} steps"),
            "w": wl.w, "global_batch": wl.shape[0]}


if __name__ == "__main__":
    sys.exit(main())
