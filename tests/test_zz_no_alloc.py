"""The DDIM step on the library's static scratch (cfg_ddim_step_static_ws), for callers
that cannot allocate device memory (no workspace argument): code inside a host framework
that owns every device allocation, or a real-time path that may not allocate after start-up.

Checked on two or more calls in a row that share the static scratch (each call sees whatever
the one before left in it):

* against the CPU oracle's step (``O.ddim_step``) on the same stored inputs, at the
  single-step tolerances: fp32 max |error| <= 1e-5 and, for eta = 0, every element within
  1 ulp (or 1e-9 after cancellation); bf16 max |g - o| / max(|o|, 1) <= 2e-2 and every
  element within 1 bf16 ulp (or 2^-17 after cancellation), and with CFG_BF16_EXACT every
  noise-free result equal to the oracle's; rel-MAE within 1e-6 relative; the schedule state
  against the oracle's rule on the oracle's rel-MAE trace;
* against cfg_ddim_step on a caller-owned workspace, bit for bit (x, M and the state).

Called through the C ABI directly and through the Python wrapper, and back to back on one
non-blocking stream with no host synchronisation between the calls.  This file is collected
last, so a run that stops at the first failure has already run every other test; it also
passes alone in a fresh process (the first call on the device then happens here).
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

# (n, eta) of consecutive steps 0, 1, 2: a large ragged step with noise, a smaller one
# without, and a last step (abar_prev = 1)
CALLS = [(1_000_003, 1.0), (65_536 + 7, 0.0), (4097, 1.0)]
W_SCALE, SEED = 6.0, 11


def _check_oracle(got, ref, dtype, eta, exact=False, last=False):
    diff = np.abs(got - ref)
    if exact and (eta == 0.0 or last):
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, bad[:10]
    if dtype == "f32":
        assert float(diff.max()) <= 1e-5, float(diff.max())
        if eta == 0.0:
            ok = (ulp_distance_f32(got, ref) <= 1) | (diff <= 1e-9)
            assert ok.all(), np.flatnonzero(~ok)[:10]
    else:
        assert float(np.max(diff / np.maximum(np.abs(ref), 1.0))) <= 2e-2
        ok = (ulp_distance_bf16(got, ref) <= 1) | (diff <= 2.0**-17)
        assert ok.all(), np.flatnonzero(~ok)[:10]


def _abar_pair(call):
    abar = O.abar_linear()
    last = call == len(CALLS) - 1
    return float(abar[600 - 20 * call]), (1.0 if last else float(abar[580 - 20 * call]))


@pytest.mark.parametrize("storage", ["bf16", "f32", "bf16_exact"])
def test_static_scratch_step_matches_oracle_and_workspace_step(cuda, storage):
    """Independent inputs per call, through the C ABI, each call synchronised."""
    dtype, exact = ("f32", False) if storage == "f32" else ("bf16", storage == "bf16_exact")
    code = cs.CFG_F32 if dtype == "f32" else (cs.CFG_BF16_EXACT if exact else cs.CFG_BF16)
    sp = cs.SchedParams(n_steps=len(CALLS), L=1, g_slope=1.0, k=2)
    st_ref, st_new = cs.new_sched_state(cuda), cs.new_sched_state(cuda)
    stream = torch.cuda.current_stream().cuda_stream
    oracle_M = []
    for call, (n, eta) in enumerate(CALLS):
        d = W.draw_prediction_pair(n, dtype, 500 + call)
        x, c, u = (to_device_stored(d[k], dtype, cuda) for k in ("x", "c", "u"))
        ab, abp = _abar_pair(call)
        ref_out, new_out = torch.empty_like(x), torch.empty_like(x)
        ref_M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        new_M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        cs.ddim_step(ref_out, x, c, u, w=W_SCALE, abar_t=ab, abar_prev=abp, eta=eta, seed=SEED,
                     step=call, M_out=ref_M, state=st_ref, sched=sp,
                     workspace=cs.new_workspace(n, code, cuda), exact_rounding=exact)
        rc = cs.lib.cfg_ddim_step_static_ws(
            new_out.data_ptr(), x.data_ptr(), c.data_ptr(), u.data_ptr(), n, code, W_SCALE, ab,
            abp, eta, SEED, call, new_M.data_ptr(), st_new.data_ptr(), ctypes.byref(sp.c), stream)
        assert rc == 0, cs.lib.cfg_last_error().decode()
        torch.cuda.synchronize()
        got = to_host_f64(new_out)
        assert np.array_equal(got, to_host_f64(ref_out)), call
        assert new_M.item() == ref_M.item(), call
        f64 = {k: W.stored_to_f64(d[k], dtype) for k in ("x", "c", "u")}
        ref, refM = O.ddim_step(f64["x"], f64["c"], f64["u"], dtype, W_SCALE, ab, abp, eta, SEED,
                                call, last=(abp == 1.0))
        _check_oracle(got, ref, dtype, eta, exact=exact, last=(abp == 1.0))
        assert abs(new_M.item() / refM - 1) <= 1e-6, call
        oracle_M.append(refM)
    a, b = cs.read_sched_state(st_ref), cs.read_sched_state(st_new)
    assert np.array_equal(a["M"], b["M"])
    for key in ("n_seen", "tau1p", "argmin", "tau_cap", "tau1", "tau2", "decided_at", "flags"):
        assert a[key] == b[key], key
    want = O.schedule(np.array(oracle_M), 1, 1.0, 2)
    assert b["flags"] == 0 and b["n_seen"] == len(CALLS)
    for key, val in want.as_dict().items():
        assert b[key] == val, (key, b[key], val)


def _chain(step_fn, x0, preds, stream, M, st, sp):
    """Steps 0..len(preds)-1 in a row on `stream`, x_{s+1} = step(x_s), no host sync."""
    xs = [x0]
    with torch.cuda.stream(stream):
        for s, (c, u) in enumerate(preds):
            n_eta = CALLS[min(s, len(CALLS) - 1)][1]
            ab, abp = _abar_pair(s)
            out = torch.empty_like(x0)
            step_fn(out, xs[-1], c, u, w=W_SCALE, abar_t=ab, abar_prev=abp, eta=n_eta, seed=SEED,
                    step=s, M_out=M[s:s + 1], state=st, sched=sp, stream=stream)
            xs.append(out)
    return xs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_static_scratch_back_to_back_on_a_nonblocking_stream(cuda, dtype):
    """Three chained steps through the Python wrapper, issued in a row on a torch stream
    (created non-blocking) with no host synchronisation between them, so each launch
    overlaps the previous one's tail (programmatic dependent launch) while both use the
    static scratch; equal bit for bit to the same chain on a caller-owned workspace, and
    each step within the oracle's tolerance on the device's own input to that step."""
    code = cs.CFG_F32 if dtype == "f32" else cs.CFG_BF16
    n = 300_001
    d = W.draw_prediction_pair(n, dtype, 900)
    x0 = to_device_stored(d["x"], dtype, cuda)
    preds = []
    for s in range(len(CALLS)):
        p = W.draw_prediction_pair(n, dtype, 910 + s)
        preds.append((to_device_stored(p["c"], dtype, cuda), to_device_stored(p["u"], dtype, cuda)))
    sp = cs.SchedParams(n_steps=len(CALLS), L=1, g_slope=1.0, k=2)
    stream = torch.cuda.Stream(cuda)
    stream.wait_stream(torch.cuda.current_stream(cuda))

    M_new = torch.full((len(CALLS),), -1.0, dtype=torch.float64, device=cuda)
    st_new = cs.new_sched_state(cuda)
    new = _chain(cs.ddim_step_static_ws, x0, preds, stream, M_new, st_new, sp)

    ws = cs.new_workspace(n, code, cuda)
    M_ref = torch.full((len(CALLS),), -1.0, dtype=torch.float64, device=cuda)
    st_ref = cs.new_sched_state(cuda)

    def with_ws(*args, **kw):
        cs.ddim_step(*args, workspace=ws, **kw)
    ref = _chain(with_ws, x0, preds, stream, M_ref, st_ref, sp)
    stream.synchronize()

    for s in range(1, len(CALLS) + 1):
        assert np.array_equal(to_host_f64(new[s]), to_host_f64(ref[s])), s
    assert torch.equal(M_new, M_ref)
    a, b = cs.read_sched_state(st_ref), cs.read_sched_state(st_new)
    assert np.array_equal(a["M"], b["M"])
    for key in ("n_seen", "tau1p", "argmin", "tau_cap", "tau1", "tau2", "decided_at", "flags"):
        assert a[key] == b[key], key

    # each step against the oracle, teacher-forced on the device's own x_s
    oracle_M = []
    for s, (c, u) in enumerate(preds):
        ab, abp = _abar_pair(s)
        eta = CALLS[s][1]
        ref_x, refM = O.ddim_step(to_host_f64(new[s]), to_host_f64(c), to_host_f64(u), dtype,
                                  W_SCALE, ab, abp, eta, SEED, s, last=(abp == 1.0))
        _check_oracle(to_host_f64(new[s + 1]), ref_x, dtype, eta)
        assert abs(M_new[s].item() / refM - 1) <= 1e-6, s
        oracle_M.append(refM)
    want = O.schedule(np.array(oracle_M), 1, 1.0, 2)
    assert b["flags"] == 0
    for key, val in want.as_dict().items():
        assert b[key] == val, (key, b[key], val)


def test_static_scratch_rejects_deferral(cuda):
    x = torch.zeros(64, dtype=torch.bfloat16, device=cuda)
    sp = cs.SchedParams(n_steps=10, defer=True)
    rc = cs.lib.cfg_ddim_step_static_ws(
        x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 64, cs.CFG_BF16, 2.0, 0.5, 0.6,
        0.0, 0, 0, None, cs.new_sched_state(cuda).data_ptr(), ctypes.byref(sp.c), None)
    assert rc == -1
    assert "workspace" in cs.lib.cfg_last_error().decode()
