"""GPU-side harness for the parity tests: the synthetic denoisers on the device.

The denoisers stand in for the model; they are not part of the sampler step.
They follow the same definition as the oracle's (``oracle.cfg_oracle.gaussian_eps``
/ ``flow_velocity``): evaluate in float64 one operation at a time
(``(x - sa*mean) * A (+ perturbation)``, or ``(x - mean) * (1/t)``), round to
fp32, then to the storage type -- so, given the same stored ``x``, both sides
store the same prediction bits.  Implemented here independently with torch
float64 device ops (each op a separate IEEE-rounded kernel, no fusion).
The sampler step itself always runs in the library (``cfg_sampler_run``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np
import torch

import cfg_guided_sampler_step_b300 as cs
import workloads as W

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_device_stored(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Upload a stored array (float32, or bf16 bits as uint16) as a tensor of the storage dtype."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    bits = np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(bits).to(device).view(torch.bfloat16)


def to_host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64).reshape(-1)


class Denoiser:
    """Synthetic CFG denoiser of a workload on the device (fills pred_c / pred_u)."""

    def __init__(self, wl: W.Workload, inputs: Dict[str, np.ndarray], x: torch.Tensor,
                 pred_c: torch.Tensor, pred_u: torch.Tensor, preload: bool = False):
        self.wl = wl
        dev = x.device
        reps = wl.n // int(np.prod(wl.mean_shape))
        self.mc = torch.from_numpy(np.tile(inputs["mean_c"].reshape(-1), reps).astype(np.float64)).to(dev)
        self.mu = torch.from_numpy(np.tile(inputs["mean_u"].reshape(-1), reps).astype(np.float64)).to(dev)
        self.x, self.pc, self.pu = x, pred_c, pred_u
        self.calls = 0
        # preload: every step's perturbations on the device up front (a run recorded into a
        # CUDA graph may not copy from pageable host memory while it is being captured)
        self.pert = None
        if preload and wl.perturb_std:
            self.pert = {(s, b): self._upload(s, b) for s in range(wl.n_steps) for b in "cu"}

    def _store(self, t64: torch.Tensor, out: torch.Tensor) -> None:
        out.view(-1).copy_(t64.to(torch.float32).to(out.dtype))

    def _upload(self, step: int, branch: str) -> Optional[torch.Tensor]:
        p = W.draw_perturbation(self.wl, step, branch)
        if p is None:
            return None
        return torch.from_numpy(p.astype(np.float64)).to(self.x.device)

    def _perturb(self, step: int, branch: str) -> Optional[torch.Tensor]:
        if self.pert is not None:
            return self.pert[(step, branch)]
        return self._upload(step, branch)

    def branch(self, b: int, step: int, timestep: int, t: float) -> None:
        """One branch only (0: conditional into pred_c, 1: unconditional into pred_u), with the
        same arithmetic as __call__, on the current stream."""
        self.calls += 1
        wl = self.wl
        mean, out, br = (self.mc, self.pc, "c") if b == 0 else (self.mu, self.pu, "u")
        x64 = self.x.view(-1).to(torch.float64)
        if wl.mode == "ddim":
            abar = t
            sa = math.sqrt(abar)
            A = math.sqrt(1.0 - abar) / (abar * wl.data_std * wl.data_std + (1.0 - abar))
            v = mean * sa
            v = x64 - v
            v = v * A
            p = self._perturb(step, br)
            if p is not None:
                v = v + p
        else:
            v = x64 - mean
            v = v * (1.0 / t)
        self._store(v, out)

    def __call__(self, step: int, timestep: int, t: float) -> None:
        self.calls += 1
        wl = self.wl
        x64 = self.x.view(-1).to(torch.float64)
        if wl.mode == "ddim":
            abar = t
            sa = math.sqrt(abar)
            A = math.sqrt(1.0 - abar) / (abar * wl.data_std * wl.data_std + (1.0 - abar))
            for mean, out, br in ((self.mc, self.pc, "c"), (self.mu, self.pu, "u")):
                v = mean * sa
                v = x64 - v
                v = v * A
                p = self._perturb(step, br)
                if p is not None:
                    v = v + p
                self._store(v, out)
        else:
            inv_t = 1.0 / t
            for mean, out in ((self.mc, self.pc), (self.mu, self.pu)):
                v = x64 - mean
                v = v * inv_t
                self._store(v, out)


@dataclass
class GpuRun:
    x0: np.ndarray
    state: Dict[str, object]


def run_workload(wl: W.Workload, inputs: Dict[str, np.ndarray], device="cuda",
                 start_from: Optional[tuple] = None, stop_after: Optional[int] = None,
                 exact_rounding: bool = False) -> GpuRun:
    """The whole sampler of a workload through cfg_sampler_run, with the device denoiser
    (``exact_rounding``: bf16 steps correctly rounded, CFG_BF16_EXACT)."""
    x = to_device_stored(inputs["x_T"], wl.dtype, device)
    pc = torch.empty_like(x)
    pu = torch.empty_like(x)
    ws = cs.new_workspace(wl.n, cs.CFG_F32 if wl.dtype == "f32" else cs.CFG_BF16, device)
    st = cs.new_sched_state(device)
    start = 0
    if start_from is not None:
        x0_saved, st_saved, start = start_from
        x.copy_(x0_saved)
        st.copy_(st_saved)
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, tau_cap=wl.tau_cap)
    den = Denoiser(wl, inputs, x, pc, pu)
    kw = dict(mode=cs.CFG_MODE_DDIM if wl.mode == "ddim" else cs.CFG_MODE_FLOW,
              n_steps=wl.n_steps, w=wl.w, denoise=den, pred_c=pc, pred_u=pu, sched=sp, state=st,
              workspace=ws, eta=wl.eta, seed=wl.seed, start_step=start,
              exact_rounding=exact_rounding)
    if wl.mode == "ddim":
        kw["abar_table"] = (cs.abar_cosine(wl.T) if wl.schedule == "cosine"
                            else cs.abar_linear(wl.T, wl.beta_start, wl.beta_end))
        kw["timesteps"] = cs.timesteps(wl.n_steps, wl.T, wl.spacing)
    if stop_after is not None:
        # run only steps [start, stop_after): emulate an interrupted run
        n_total = wl.n_steps

        def den_stop(step, timestep, t):
            if step >= stop_after:
                raise StopIteration(step)
            den(step, timestep, t)
        kw["denoise"] = den_stop
        try:
            cs.sampler_run(x, **kw)
        except StopIteration:
            pass
        torch.cuda.synchronize()
        assert n_total == wl.n_steps
        return GpuRun(to_host_f64(x), {"x": x.clone(), "st": st.clone()})
    cs.sampler_run(x, **kw)
    torch.cuda.synchronize()
    return GpuRun(to_host_f64(x), cs.read_sched_state(st))


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max_i |got - ref| / max(|ref|, 1)."""
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)))


def ulp_distance_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def ulp_distance_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return ulp_distance_f32(a, b) >> 16


# ---------------------------------------------------------------------------
# Exact rounding checks
# ---------------------------------------------------------------------------
def _dist_to_midpoint(q, lo_val: float, hi_val: float):
    """|q - (lo + hi)/2| for a Fraction q and two adjacent bf16 values."""
    from fractions import Fraction as F
    return abs(q - (F(lo_val) + F(hi_val)) / 2)


def certify_bf16_mismatches(got: np.ndarray, ref: np.ndarray, exact_value, rel: float = 2.0**-40,
                            abs_floor: float = 2.0**-17, limit: int = 20000) -> np.ndarray:
    """Elements where a correctly rounded bf16 step and the oracle's may differ.

    ``got`` and ``ref`` are bf16 values (as float64).  Each element that differs must be one
    bf16 ulp away from the oracle's, with the exact value of the step (``exact_value(i)``:
    ``(Fraction value, scale)`` with ``scale`` the sum of the magnitudes of its terms)
    within ``rel * scale`` of the midpoint between the two -- where either neighbour is a
    correct rounding within the evaluation error of either side -- or be within
    ``abs_floor`` of it (a result cancelled to below the evaluation's absolute error).
    Returns the indices that fail (empty when all differences are certified)."""
    bad = np.flatnonzero(got != ref)
    assert bad.size <= limit, bad.size
    failed = []
    for i in bad:
        if abs(got[i] - ref[i]) <= abs_floor:
            continue
        if ulp_distance_bf16(got[i:i + 1], ref[i:i + 1])[0] != 1:
            failed.append(i)
            continue
        q, scale = exact_value(int(i))
        lo_v, hi_v = sorted((float(got[i]), float(ref[i])))
        if float(_dist_to_midpoint(q, lo_v, hi_v)) > rel * scale:
            failed.append(i)
    return np.array(failed, dtype=np.int64)


def flow_exact(x, c, u, w: float, t_cur: float, t_next: float):
    """Exact value (Fraction) and term scale of the Euler step x + (t_next - t_cur) v,
    v = u + w (c - u), on exact inputs and the fp64 time step the library is given."""
    from fractions import Fraction as F

    def fn(i):
        dt = F(t_next - t_cur)
        v = F(float(u[i])) + F(w) * (F(float(c[i])) - F(float(u[i])))
        q = F(float(x[i])) + dt * v
        return q, abs(float(x[i])) + abs(float(dt * v)) + 1e-300
    return fn


def ddim_exact(x, c, u, w: float, abar_t: float, abar_prev: float):
    """Exact value and term scale of the noise-free DDIM step on exact inputs, with the
    square roots the oracle uses (fp64): sqrt(abar_prev) (x - sqrt(1 - abar_t) e) /
    sqrt(abar_t) + sqrt(1 - abar_prev) e, or the x0 prediction when abar_prev = 1."""
    from fractions import Fraction as F
    sa, sb = F(math.sqrt(abar_t)), F(math.sqrt(1.0 - abar_t))
    sap, sd = F(math.sqrt(abar_prev)), F(math.sqrt(max(0.0, 1.0 - abar_prev)))

    def fn(i):
        e = F(float(u[i])) + F(w) * (F(float(c[i])) - F(float(u[i])))
        x0 = (F(float(x[i])) - sb * e) / sa
        q = x0 if abar_prev == 1.0 else sap * x0 + sd * e
        scale = (abs(float(sap * F(float(x[i])) / sa)) + abs(float(sap * sb * e / sa))
                 + abs(float(sd * e)) + 1e-300)
        return q, scale
    return fn
