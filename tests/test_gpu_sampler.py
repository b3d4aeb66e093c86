"""Whole-run parity: cfg_sampler_run on the device against the oracle's run (needs a GPU).

Each workload is run end to end by the library's native sampler loop with the
device-side synthetic denoiser, and by the oracle in float64 from the same
stored x_T, means and perturbations.  Checked:

* x_0: fp32 storage max abs error <= 1e-5; bf16 storage
  max |g - o| / max(|o|, 1) <= 2e-2;
* the rel-MAE trace: fp32 abs <= 1e-5 and rel <= 1e-6; bf16 rel <= 1e-3
  (the trajectories differ only by rare 1-ulp rounding disagreements);
* tau1', tau_cap, tau1, tau2, decided_at and the phases: exactly equal to
  the oracle's, and the oracle's rule applied to the device's own M trace
  reproduces the device's G values bit for bit.

Small shapes (several blocks, ragged tails) run first; the full workload
sizes follow, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_harness import rel_err, run_workload
from oracle import cfg_oracle as O

pytestmark = pytest.mark.gpu

SMALL = [
    ("sd_point_mass_f32", (1, 3, 17, 19)),
    ("sd_point_mass_f32", (1, 4, 64, 64)),
    ("sdxl_1024_b8_bf16", (3, 4, 17, 19)),
    ("sd_3840px_eta1_bf16", (1, 4, 61, 67)),
    ("dit_flow_b4_bf16", (2, 16, 37, 41)),
    ("video_b2_bf16", (1, 16, 3, 17, 19)),
]


def _check(wl, inputs, gpu, ref):
    if wl.dtype == "f32":
        err = float(np.max(np.abs(gpu.x0 - ref.x0)))
        assert err <= 1e-5, err
        assert float(np.max(np.abs(gpu.state["M"] - ref.M))) <= 1e-5
        assert float(np.max(np.abs(gpu.state["M"] / ref.M - 1))) <= 1e-6
    else:
        assert rel_err(gpu.x0, ref.x0) <= 2e-2
        assert float(np.max(np.abs(gpu.state["M"] / ref.M - 1))) <= 1e-3
    st = gpu.state
    assert st["n_seen"] == wl.n_steps and st["flags"] == 0
    for key, val in ref.sched.as_dict().items():
        assert st[key] == val, (key, st[key], val)
    assert np.array_equal(st["phase"], ref.sched.phase)
    # the rule applied by the oracle to the device's own trace gives the device's numbers
    same = O.schedule(st["M"], wl.L, wl.g_slope, wl.k, wl.tau_cap)
    assert np.array_equal(same.G, st["G"], equal_nan=True)
    assert {k: st[k] for k in same.as_dict()} == same.as_dict()


def _perturb(wl):
    return (lambda s, b: W.draw_perturbation(wl, s, b)) if wl.perturb_std else None


@pytest.mark.parametrize("name,shape", SMALL, ids=[f"{n}-{'x'.join(map(str, s))}" for n, s in SMALL])
def test_small_runs_match_oracle(cuda, name, shape):
    wl = W.WORKLOADS[name].scaled(shape)
    inputs = W.draw_inputs(wl)
    gpu = run_workload(wl, inputs, cuda)
    ref = O.run_sampler(wl, inputs, perturb=_perturb(wl))
    _check(wl, inputs, gpu, ref)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_full_size_runs_match_oracle(cuda, name):
    wl = W.WORKLOADS[name]
    inputs = W.draw_inputs(wl)
    gpu = run_workload(wl, inputs, cuda)
    ref = O.run_sampler(wl, inputs, perturb=_perturb(wl))
    _check(wl, inputs, gpu, ref)


def test_point_mass_run_lands_on_guided_mean(cuda):
    """fp32 point-mass DDIM: x_0 = mu_u + w (mu_c - mu_u) up to the storage rounding of the
    predictions, amplified by w (|err| <= 14 * ulp(|eps|)/2 * sqrt(1 - abar_0) < 5e-5)."""
    wl = W.WORKLOADS["sd_point_mass_f32"]
    inputs = W.draw_inputs(wl)
    gpu = run_workload(wl, inputs, cuda)
    mc = inputs["mean_c"].reshape(-1).astype(np.float64)
    mu = inputs["mean_u"].reshape(-1).astype(np.float64)
    assert float(np.max(np.abs(gpu.x0 - (mu + wl.w * (mc - mu))))) < 5e-5


def test_run_is_deterministic(cuda):
    wl = W.WORKLOADS["sd_3840px_eta1_bf16"].scaled((1, 4, 96, 96))
    inputs = W.draw_inputs(wl)
    a = run_workload(wl, inputs, cuda)
    b = run_workload(wl, inputs, cuda)
    assert np.array_equal(a.x0, b.x0)
    assert np.array_equal(a.state["M"], b.state["M"])


def test_resume_from_saved_state(cuda):
    """Stopping after step 20 and resuming from the saved (x, state) reproduces a full run."""
    wl = W.WORKLOADS["sdxl_1024_b8_bf16"].scaled((2, 4, 32, 32))
    inputs = W.draw_inputs(wl)
    full = run_workload(wl, inputs, cuda)
    part = run_workload(wl, inputs, cuda, stop_after=20)
    resumed = run_workload(wl, inputs, cuda, start_from=(part.state["x"], part.state["st"], 20))
    assert np.array_equal(full.x0, resumed.x0)
    assert np.array_equal(full.state["M"], resumed.state["M"])
    assert full.state["tau1"] == resumed.state["tau1"]


def test_callback_error_stops_the_run(cuda):
    import cfg_guided_sampler_step_b300 as cs
    wl = W.WORKLOADS["sdxl_1024_b8_bf16"].scaled((1, 4, 8, 8))
    x = torch.zeros(wl.n, dtype=torch.bfloat16, device=cuda)
    seen = []

    def bad(step, timestep, t):
        seen.append(step)
        if step == 3:
            raise ValueError("denoiser failed")

    with pytest.raises(ValueError, match="denoiser failed"):
        cs.sampler_run(x, mode=cs.CFG_MODE_DDIM, n_steps=wl.n_steps, w=5.0, denoise=bad,
                       pred_c=torch.zeros_like(x), pred_u=torch.zeros_like(x),
                       sched=cs.SchedParams(n_steps=wl.n_steps), state=cs.new_sched_state(cuda),
                       workspace=cs.new_workspace(wl.n, cs.CFG_BF16, cuda),
                       abar_table=cs.abar_linear(), timesteps=cs.ddim_timesteps(wl.n_steps))
    assert seen == [0, 1, 2, 3]
