"""The DDIM step on the library's static scratch (cfg_ddim_step_static_ws), for callers
that cannot allocate device memory (no workspace argument).

It must give what cfg_ddim_step gives with a caller-owned workspace, on two calls in a
row that share the static scratch (the second call sees whatever the first left in it).
Tolerances are those of the single-step parity tests: fp32 within 1 ulp (or 1e-9 after
cancellation), bf16 within 1 bf16 ulp (or 2^-17), rel-MAE within 1e-6 relative; the
schedule state must agree.  Called through the C ABI directly.  This file is collected
last, so a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import cfg_guided_sampler_step_b300 as cs
import workloads as W
from gpu_harness import to_device_stored, to_host_f64, ulp_distance_bf16, ulp_distance_f32
from oracle import cfg_oracle as O

pytestmark = pytest.mark.gpu

# (n, step, eta): a large ragged bf16/fp32 step with noise, then a smaller one without
CALLS = [(1_000_003, 3, 1.0), (65_536 + 7, 4, 0.0)]


def _close(got, ref, dtype):
    diff = np.abs(got - ref)
    if dtype == "f32":
        ok = (ulp_distance_f32(got, ref) <= 1) | (diff <= 1e-9)
    else:
        ok = (ulp_distance_bf16(got, ref) <= 1) | (diff <= 2.0**-17)
    return bool(ok.all())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_static_scratch_step_matches_workspace_step(cuda, dtype):
    code = cs.CFG_F32 if dtype == "f32" else cs.CFG_BF16
    abar = O.abar_linear()
    sp = cs.SchedParams(n_steps=10, L=1, g_slope=1.0, k=2)
    st_ref, st_new = cs.new_sched_state(cuda), cs.new_sched_state(cuda)
    stream = torch.cuda.current_stream().cuda_stream
    for call, (n, step, eta) in enumerate(CALLS):
        d = W.draw_prediction_pair(n, dtype, 500 + call)
        x, c, u = (to_device_stored(d[k], dtype, cuda) for k in ("x", "c", "u"))
        ab, abp = float(abar[600 - 20 * call]), float(abar[580 - 20 * call])
        ref_out, new_out = torch.empty_like(x), torch.empty_like(x)
        ref_M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        new_M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        cs.ddim_step(ref_out, x, c, u, w=6.0, abar_t=ab, abar_prev=abp, eta=eta, seed=11,
                     step=step, M_out=ref_M, state=st_ref, sched=sp,
                     workspace=cs.new_workspace(n, code, cuda))
        rc = cs.lib.cfg_ddim_step_static_ws(
            new_out.data_ptr(), x.data_ptr(), c.data_ptr(), u.data_ptr(), n, code, 6.0, ab, abp,
            eta, 11, step, new_M.data_ptr(), st_new.data_ptr(), ctypes.byref(sp.c), stream)
        assert rc == 0, cs.lib.cfg_last_error().decode()
        torch.cuda.synchronize()
        assert _close(to_host_f64(new_out), to_host_f64(ref_out), dtype), call
        assert abs(new_M.item() / ref_M.item() - 1) <= 1e-6, call
    a, b = cs.read_sched_state(st_ref), cs.read_sched_state(st_new)
    for key in ("n_seen", "tau1p", "argmin", "flags"):
        assert a[key] == b[key], key
    assert np.allclose(a["M"], b["M"], rtol=1e-6, atol=0)


def test_static_scratch_rejects_deferral(cuda):
    x = torch.zeros(64, dtype=torch.bfloat16, device=cuda)
    sp = cs.SchedParams(n_steps=10, defer=True)
    rc = cs.lib.cfg_ddim_step_static_ws(
        x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 64, cs.CFG_BF16, 2.0, 0.5, 0.6,
        0.0, 0, 0, None, cs.new_sched_state(cuda).data_ptr(), ctypes.byref(sp.c), None)
    assert rc == -1
    assert "workspace" in cs.lib.cfg_last_error().decode()
