"""Batched steps with per-sample rel-MAE and schedules (needs a GPU).

One launch over `batch` samples: every element's update is the unbatched step's (the noise
counter is the element's index in the whole batch), while each sample b gets its own
M_b (the oracle's rel_mae_per_sample) and its own tau1/tau2 state (the oracle's schedule
rule on that sample's trace).  Tolerances are those of the single-step and whole-run
parity tests.
"""
import numpy as np
import pytest
import torch

import cfg_guided_sampler_step_b300 as cs
import workloads as W
from gpu_harness import Denoiser, to_device_stored, to_host_f64, ulp_distance_bf16
from oracle import cfg_oracle as O

pytestmark = pytest.mark.gpu


def _code(dtype):
    return cs.CFG_F32 if dtype == "f32" else cs.CFG_BF16


def _pair(n, dtype, seed, cuda):
    d = W.draw_prediction_pair(n, dtype, seed)
    dev = {k: to_device_stored(d[k], dtype, cuda) for k in ("x", "c", "u")}
    f64 = {k: W.stored_to_f64(d[k], dtype) for k in ("x", "c", "u")}
    return dev, f64


# storage under test: fp32, bf16 with the default rounding, bf16 correctly rounded
STORAGES = [("f32", False), ("bf16", False), ("bf16", True)]
STORAGE_IDS = ["f32", "bf16", "bf16_exact"]


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("batch,n_ps", [(1, 4096), (3, 4096), (8, 65536), (5, 1003), (2, 3 * 2**18 + 8)])
@pytest.mark.parametrize("eta", [0.0, 1.0])
def test_batched_ddim_step(cuda, dtype, exact, batch, n_ps, eta):
    n = batch * n_ps
    d, f = _pair(n, dtype, 600 + batch + n_ps % 97, cuda)
    abar = O.abar_linear()
    ab, abp = float(abar[400]), float(abar[380])
    ref_out, out = torch.empty_like(d["x"]), torch.empty_like(d["x"])
    M1 = torch.zeros(1, dtype=torch.float64, device=cuda)
    MB = torch.full((batch,), -1.0, dtype=torch.float64, device=cuda)
    cs.ddim_step(ref_out, d["x"], d["c"], d["u"], w=6.0, abar_t=ab, abar_prev=abp, eta=eta, seed=5,
                 step=7, M_out=M1, workspace=cs.new_workspace(n, _code(dtype), cuda),
                 exact_rounding=exact)
    cs.ddim_step(out, d["x"], d["c"], d["u"], w=6.0, abar_t=ab, abar_prev=abp, eta=eta, seed=5,
                 step=7, M_out=MB, workspace=cs.new_workspace(n, _code(dtype), cuda, batch=batch),
                 batch=batch, exact_rounding=exact)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)                 # the update is the unbatched step's
    if exact and eta == 0.0:                         # correctly rounded: the oracle's, element by element
        want, _ = O.ddim_step(f["x"], f["c"], f["u"], "bf16", 6.0, ab, abp, 0.0, 5, 7)
        bad = np.flatnonzero(to_host_f64(out) != want)
        assert bad.size == 0, bad[:10]
    ref = O.rel_mae_per_sample(f["c"], f["u"], batch)
    got = MB.cpu().numpy()
    assert np.all(np.abs(got / ref - 1) <= 1e-6), (got, ref)


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("batch,n_ps", [(4, 4096), (3, 777)])
def test_batched_flow_step_and_reduce(cuda, dtype, exact, batch, n_ps):
    n = batch * n_ps
    d, f = _pair(n, dtype, 700 + batch, cuda)
    ref_out, out = torch.empty_like(d["x"]), torch.empty_like(d["x"])
    MB = torch.full((batch,), -1.0, dtype=torch.float64, device=cuda)
    MR = torch.full((batch,), -1.0, dtype=torch.float64, device=cuda)
    ws = cs.new_workspace(n, _code(dtype), cuda, batch=batch)
    cs.flow_step(ref_out, d["x"], d["c"], d["u"], w=3.5, t_cur=0.5, t_next=0.45,
                 workspace=cs.new_workspace(n, _code(dtype), cuda), exact_rounding=exact)
    cs.flow_step(out, d["x"], d["c"], d["u"], w=3.5, t_cur=0.5, t_next=0.45, M_out=MB,
                 workspace=ws, batch=batch, exact_rounding=exact)
    cs.relmae_reduce(d["c"], d["u"], M_out=MR, workspace=ws, batch=batch)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    if exact:                                        # correctly rounded: the oracle's, element by element
        want, _ = O.flow_step(f["x"], f["c"], f["u"], "bf16", 3.5, 0.5, 0.45)
        bad = np.flatnonzero(to_host_f64(out) != want)
        assert bad.size == 0, bad[:10]
    ref = O.rel_mae_per_sample(f["c"], f["u"], batch)
    for M in (MB, MR):
        assert np.all(np.abs(M.cpu().numpy() / ref - 1) <= 1e-6)


@pytest.mark.parametrize("defer", [False, True])
def test_batched_schedules_follow_each_sample(cuda, defer):
    """A 12-step sequence with different predictions per sample and step: every sample's
    state is the oracle's rule on that sample's own trace; deferral changes nothing."""
    batch, n_ps, N = 6, 20_000, 12
    n = batch * n_ps
    g = np.random.default_rng(44)
    abar = O.abar_linear()
    ts = O.ddim_timesteps(N)
    st = cs.new_sched_state(cuda, batch=batch)
    sp = cs.SchedParams(n_steps=N, L=2, g_slope=0.02, k=3, defer=defer)
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda, batch=batch)
    MB = torch.full((N, batch), -1.0, dtype=torch.float64, device=cuda)
    x = torch.from_numpy(W.f32_to_bf16_bits(g.standard_normal(n)).view(np.int16)).to(cuda).view(torch.bfloat16)
    traces = np.empty((N, batch))
    for s in range(N):
        u = g.standard_normal(n)
        # per-sample discrepancy scales that move over the run, so the traces differ
        scale = np.repeat(0.05 + 0.1 * np.abs(np.sin(0.4 * s + np.arange(batch))), n_ps)
        c = u + g.standard_normal(n) * scale
        cb, ub = W.store(c, "bf16"), W.store(u, "bf16")
        traces[s] = O.rel_mae_per_sample(W.stored_to_f64(cb, "bf16"), W.stored_to_f64(ub, "bf16"), batch)
        dc, du = (to_device_stored(a, "bf16", cuda) for a in (cb, ub))
        abp = 1.0 if s == N - 1 else float(abar[ts[s + 1]])
        cs.ddim_step(x, x, dc, du, w=4.0, abar_t=float(abar[ts[s]]), abar_prev=abp, step=s,
                     M_out=MB[s], state=st, sched=sp, workspace=ws, batch=batch)
    torch.cuda.synchronize()
    got_M = MB.cpu().numpy()
    assert np.all(np.abs(got_M / traces - 1) <= 1e-6)
    for b in range(batch):
        got = cs.read_sched_state(st, b)
        ref = O.schedule(got["M"], sp.c.L, sp.c.g_slope, sp.c.k, -1)
        assert np.array_equal(got["M"], got_M[:, b])
        assert np.allclose(got["M"], traces[:, b], rtol=1e-6, atol=0)
        assert {k: got[k] for k in ref.as_dict()} == ref.as_dict(), b
        assert np.array_equal(got["G"], ref.G, equal_nan=True)
        assert np.array_equal(got["phase"], ref.phase)
        assert got["flags"] == 0 and got["n_seen"] == N


def test_batched_full_sdxl_run_per_sample_schedules(cuda):
    """The SDXL 1024px workload, batch 8, 50 DDIM steps, one batched step per denoising step:
    x_0 within the whole-run tolerance of the oracle, each sample's M trace within 1e-3 and
    its tau1', tau_cap, tau1, tau2 exactly the oracle's per-sample schedule."""
    wl = W.WORKLOADS["sdxl_1024_b8_bf16"]
    batch = wl.shape[0]
    inputs = W.draw_inputs(wl)
    ref = O.run_sampler(wl, inputs, batch=batch)
    x = to_device_stored(inputs["x_T"], wl.dtype, cuda)
    pc, pu = torch.empty_like(x), torch.empty_like(x)
    den = Denoiser(wl, inputs, x, pc, pu)
    st = cs.new_sched_state(cuda, batch=batch)
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, defer=True)
    ws = cs.new_workspace(wl.n, cs.CFG_BF16, cuda, batch=batch)
    abar = cs.abar_linear(wl.T, wl.beta_start, wl.beta_end)
    ts = cs.ddim_timesteps(wl.n_steps, wl.T)
    for s in range(wl.n_steps):
        ab = float(abar[ts[s]])
        abp = 1.0 if s == wl.n_steps - 1 else float(abar[ts[s + 1]])
        den(s, int(ts[s]), ab)
        cs.ddim_step(x, x, pc, pu, w=wl.w, abar_t=ab, abar_prev=abp, eta=wl.eta, seed=wl.seed,
                     step=s, state=st, sched=sp, workspace=ws, batch=batch)
    torch.cuda.synchronize()
    g = to_host_f64(x)
    dx = g - ref.x0
    assert np.linalg.norm(dx) <= 2e-2 * np.linalg.norm(ref.x0)
    assert float(np.mean(ulp_distance_bf16(g, ref.x0) > 1)) <= 0.01
    for b in range(batch):
        got = cs.read_sched_state(st, b)
        assert np.max(np.abs(got["M"] / ref.M_samples[:, b] - 1)) <= 1e-3
        assert {k: got[k] for k in ref.sched_samples[b].as_dict()} == ref.sched_samples[b].as_dict(), b
        assert got["n_seen"] == wl.n_steps and got["flags"] == 0


def _batched_run(wl, inputs, cuda, batch):
    """The workload's whole run as a Python loop of batched steps (per-sample schedules,
    deferred reductions) with the device denoiser; returns (x_0, [state of each sample])."""
    x = to_device_stored(inputs["x_T"], wl.dtype, cuda)
    pc, pu = torch.empty_like(x), torch.empty_like(x)
    den = Denoiser(wl, inputs, x, pc, pu)
    st = cs.new_sched_state(cuda, batch=batch)
    sp = cs.SchedParams(n_steps=wl.n_steps, L=wl.L, g_slope=wl.g_slope, k=wl.k, defer=True)
    ws = cs.new_workspace(wl.n, _code(wl.dtype), cuda, batch=batch)
    N = wl.n_steps
    if wl.mode == "ddim":
        abar = cs.abar_linear(wl.T, wl.beta_start, wl.beta_end)
        ts = cs.ddim_timesteps(N, wl.T)
    for s in range(N):
        if wl.mode == "ddim":
            ab = float(abar[ts[s]])
            abp = 1.0 if s == N - 1 else float(abar[ts[s + 1]])
            den(s, int(ts[s]), ab)
            cs.ddim_step(x, x, pc, pu, w=wl.w, abar_t=ab, abar_prev=abp, eta=wl.eta, seed=wl.seed,
                         step=s, state=st, sched=sp, workspace=ws, batch=batch)
        else:
            t, tn = 1.0 - s / N, 1.0 - (s + 1) / N
            den(s, s, t)
            cs.flow_step(x, x, pc, pu, w=wl.w, t_cur=t, t_next=tn, step=s, state=st, sched=sp,
                         workspace=ws, batch=batch)
    torch.cuda.synchronize()
    return to_host_f64(x), [cs.read_sched_state(st, b) for b in range(batch)]


@pytest.mark.parametrize("name,shape", [("dit_flow_b4_bf16", None), ("video_b2_bf16", None),
                                        ("sd_3840px_eta1_bf16", (3, 4, 64, 64)),
                                        ("sd_point_mass_f32", (4, 4, 32, 32))])
def test_batched_whole_runs_per_sample(cuda, name, shape):
    """Whole runs of the flow, video, eta = 1 and fp32 workloads as batched steps: x_0 within
    the whole-run tolerance of the oracle, and each sample's M trace and tau values against
    the oracle's per-sample schedule."""
    wl = W.WORKLOADS[name] if shape is None else W.WORKLOADS[name].scaled(shape)
    batch = wl.shape[0]
    inputs = W.draw_inputs(wl)
    pert = (lambda s_, b_: W.draw_perturbation(wl, s_, b_)) if wl.perturb_std else None
    ref = O.run_sampler(wl, inputs, perturb=pert, batch=batch)
    x0, states = _batched_run(wl, inputs, cuda, batch)
    if wl.dtype == "f32":
        assert float(np.max(np.abs(x0 - ref.x0))) <= 1e-5
        mtol = 1e-6
    else:
        assert np.linalg.norm(x0 - ref.x0) <= 2e-2 * np.linalg.norm(ref.x0)
        assert np.max(np.abs(x0 - ref.x0)) <= 2e-2 * np.max(np.abs(ref.x0))
        mtol = 1e-3
    for b, got in enumerate(states):
        assert np.max(np.abs(got["M"] / ref.M_samples[:, b] - 1)) <= mtol, b
        assert {k: got[k] for k in ref.sched_samples[b].as_dict()} == ref.sched_samples[b].as_dict(), b
        assert np.array_equal(got["phase"], ref.sched_samples[b].phase)
        assert got["n_seen"] == wl.n_steps and got["flags"] == 0


def test_batched_arguments_validated(cuda):
    x = torch.zeros(64, dtype=torch.bfloat16, device=cuda)
    ws = cs.new_workspace(64, cs.CFG_BF16, cuda, batch=2)
    with pytest.raises(cs.CfgError):                  # workspace for 2 samples, 4 asked
        cs.ddim_step(x, x, x, x, w=2.0, abar_t=0.5, abar_prev=0.6, workspace=ws, batch=4)
    with pytest.raises(ValueError):                   # 64 elements do not split into 3 samples
        cs.ddim_step(x, x, x, x, w=2.0, abar_t=0.5, abar_prev=0.6, workspace=ws, batch=3)
    assert cs.lib.cfg_ddim_step_batched(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 32,
                                        0, cs.CFG_BF16, 2.0, 0.5, 0.6, 0.0, 0, 0, None, None,
                                        None, ws.data_ptr(), ws.numel(), None) == -1
