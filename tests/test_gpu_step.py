"""Single-call parity of the CUDA library against the CPU oracle (needs a GPU).

Every call goes through the C ABI (via the ctypes binding) on stored inputs
drawn by ``workloads``; the oracle computes the same step in float64 on the
same stored values.  Tolerances:

* fp32 storage: max abs error <= 1e-5, and for eta = 0 every element within
  1 ulp of the oracle's rounded value (the library uses compensated
  arithmetic for fp32 storage); with eta > 0 the noise itself is an fp32
  Box-Muller value (relative error ~4e-7), so only the 1e-5 bound applies;
* bf16 storage: max |g - o| / max(|o|, 1) <= 2e-2, and every element within
  1 bf16 ulp unless cancellation left a result below the fp32 arithmetic's
  absolute error (2^-17); correctly rounded (CFG_BF16_EXACT) and without
  noise, every element equal to the oracle's bf16 value (the oracle's fp64
  step rounded once: the library decides its near-midpoint elements with the
  same fp64 evaluation);
* rel-MAE: relative error <= 1e-6 (fp32 L1 partial sums with Kahan
  compensation, fp64 combine).
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import cfg_guided_sampler_step_b300 as cs
import workloads as W
from oracle import cfg_oracle as O
from gpu_harness import (TORCH_DTYPE, certify_bf16_mismatches, ddim_exact, flow_exact, rel_err,
                         to_device_stored, to_host_f64, ulp_distance_bf16, ulp_distance_f32)

pytestmark = pytest.mark.gpu
GOLDEN = Path(__file__).parent / "golden"

SIZES = [0, 1, 7, 9, 4097, 65536 + 3, 1 << 20, 3 * (1 << 20) + 5]


def _code(dtype):
    return cs.CFG_F32 if dtype == "f32" else cs.CFG_BF16


def _inputs(n, dtype, seed, cuda, offset=0):
    """Stored x, pred_c, pred_u on the device (optionally starting `offset` elements into
    their allocation, so the pointers are not 16-byte aligned) and their exact fp64 values."""
    d = W.draw_prediction_pair(n, dtype, seed)
    out = {}
    for k in ("x", "c", "u"):
        arr = d[k]
        if offset:
            full = to_device_stored(np.concatenate([np.zeros(offset, dtype=arr.dtype), arr]), dtype,
                                    cuda)
            out[k] = full[offset:]
        else:
            out[k] = to_device_stored(arr, dtype, cuda)
        out[k + "64"] = W.stored_to_f64(arr, dtype)
    return out


def _compare(got, ref, dtype, strict_ulp, exact_bf16=None):
    """Stated tolerance, plus (strict_ulp) every element within 1 ulp of the oracle's stored
    value or, where the result is tiny after cancellation, within the arithmetic's absolute
    error bound (fp32 noise in the bf16 step: 2^-17; compensated fp32: <= 1e-9), plus
    (exact_bf16: the step's exact value, see gpu_harness.ddim_exact / flow_exact, used to
    describe any failure) every bf16 element equal to the oracle's."""
    if got.size == 0:
        return
    diff = np.abs(got - ref)
    if dtype == "f32":
        assert float(diff.max()) <= 1e-5, float(diff.max())
        if strict_ulp:
            ok = (ulp_distance_f32(got, ref) <= 1) | (diff <= 1e-9)
            assert ok.all(), np.flatnonzero(~ok)[:10]
    else:
        assert rel_err(got, ref) <= 2e-2
        if strict_ulp:
            ok = (ulp_distance_bf16(got, ref) <= 1) | (diff <= 2.0**-17)
            assert ok.all(), np.flatnonzero(~ok)[:10]
        if exact_bf16 is not None:
            bad = np.flatnonzero(got != ref)
            assert bad.size == 0, (bad[:10], got[bad[:10]], ref[bad[:10]],
                                   certify_bf16_mismatches(got, ref, exact_bf16)[:10])


# storage under test: fp32, bf16 with the default rounding, bf16 correctly rounded
STORAGES = [("f32", False), ("bf16", False), ("bf16", True)]
STORAGE_IDS = ["f32", "bf16", "bf16_exact"]


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("eta", [0.0, 1.0])
def test_ddim_step_matches_oracle(cuda, dtype, exact, n, eta):
    d = _inputs(n, dtype, seed=100 + n % 97, cuda=cuda)
    abar = O.abar_linear()
    ab, abp = float(abar[500]), float(abar[480])
    w, seed, step = 7.5, 0xC0FFEE_1234, 17
    x_out = torch.empty_like(d["x"])
    M = torch.zeros(1, dtype=torch.float64, device=cuda)
    ws = cs.new_workspace(n, _code(dtype), cuda)
    cs.ddim_step(x_out, d["x"], d["c"], d["u"], w=w, abar_t=ab, abar_prev=abp, eta=eta, seed=seed,
                 step=step, M_out=M, workspace=ws, exact_rounding=exact)
    torch.cuda.synchronize()
    ref, refM = O.ddim_step(d["x64"], d["c64"], d["u64"], dtype, w, ab, abp, eta, seed, step)
    _compare(to_host_f64(x_out), ref, dtype, strict_ulp=(eta == 0.0 or dtype == "bf16"),
             exact_bf16=ddim_exact(d["x64"], d["c64"], d["u64"], w, ab, abp)
             if (exact and eta == 0.0) else None)
    gotM = float(M.item())
    if n == 0:
        assert gotM == 0.0 and refM == 0.0
    else:
        assert abs(gotM - refM) <= 1e-6 * refM


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("n", [1, 9, 4097, 1 << 20])
def test_ddim_last_step_and_in_place(cuda, dtype, exact, n):
    """abar_prev = 1 returns the x0 prediction; x_out may alias x_in."""
    d = _inputs(n, dtype, seed=7, cuda=cuda)
    ab = float(O.abar_linear()[0])
    ws = cs.new_workspace(n, _code(dtype), cuda)
    x = d["x"].clone()
    cs.ddim_step(x, x, d["c"], d["u"], w=6.0, abar_t=ab, abar_prev=1.0, eta=1.0, seed=3, step=49,
                 workspace=ws, exact_rounding=exact)
    torch.cuda.synchronize()
    ref, _ = O.ddim_step(d["x64"], d["c64"], d["u64"], dtype, 6.0, ab, 1.0, 1.0, 3, 49, last=True)
    _compare(to_host_f64(x), ref, dtype, strict_ulp=True,
             exact_bf16=ddim_exact(d["x64"], d["c64"], d["u64"], 6.0, ab, 1.0) if exact else None)


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("offset", [1, 3])
@pytest.mark.parametrize("eta", [0.0, 1.0])
def test_misaligned_pointers_take_the_scalar_path(cuda, dtype, exact, offset, eta):
    n = 50_000 + 3
    d = _inputs(n, dtype, seed=11, cuda=cuda, offset=offset)
    assert d["x"].data_ptr() % 16 != 0
    abar = O.abar_linear()
    ab, abp = float(abar[700]), float(abar[680])
    x_out = torch.empty(n + 1, dtype=TORCH_DTYPE[dtype], device=cuda)[1:]
    M = torch.zeros(1, dtype=torch.float64, device=cuda)
    ws = cs.new_workspace(n, _code(dtype), cuda)
    cs.ddim_step(x_out, d["x"], d["c"], d["u"], w=5.0, abar_t=ab, abar_prev=abp, eta=eta, seed=5,
                 step=2, M_out=M, workspace=ws, exact_rounding=exact)
    torch.cuda.synchronize()
    ref, refM = O.ddim_step(d["x64"], d["c64"], d["u64"], dtype, 5.0, ab, abp, eta, 5, 2)
    _compare(to_host_f64(x_out), ref, dtype, strict_ulp=(eta == 0.0 or dtype == "bf16"),
             exact_bf16=ddim_exact(d["x64"], d["c64"], d["u64"], 5.0, ab, abp)
             if (exact and eta == 0.0) else None)
    assert abs(M.item() - refM) <= 1e-6 * refM


@pytest.mark.parametrize("dtype,exact", STORAGES, ids=STORAGE_IDS)
@pytest.mark.parametrize("n", [0, 1, 9, 4097, 1 << 20, 3 * (1 << 20) + 5])
def test_flow_step_matches_oracle(cuda, dtype, exact, n):
    d = _inputs(n, dtype, seed=200 + n % 13, cuda=cuda)
    t_cur, t_next = 1.0 - 3 / 28, 1.0 - 4 / 28
    x_out = torch.empty_like(d["x"])
    M = torch.zeros(1, dtype=torch.float64, device=cuda)
    ws = cs.new_workspace(n, _code(dtype), cuda)
    cs.flow_step(x_out, d["x"], d["c"], d["u"], w=3.5, t_cur=t_cur, t_next=t_next, M_out=M,
                 workspace=ws, exact_rounding=exact)
    torch.cuda.synchronize()
    ref, refM = O.flow_step(d["x64"], d["c64"], d["u64"], dtype, 3.5, t_cur, t_next)
    _compare(to_host_f64(x_out), ref, dtype, strict_ulp=True,
             exact_bf16=flow_exact(d["x64"], d["c64"], d["u64"], 3.5, t_cur, t_next) if exact else None)
    if n:
        assert abs(M.item() - refM) <= 1e-6 * refM


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [0, 1, 7, 4097, 1 << 20])
def test_relmae_reduce_matches_oracle(cuda, dtype, n):
    d = _inputs(n, dtype, seed=300 + n % 7, cuda=cuda)
    M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
    ws = cs.new_workspace(n, _code(dtype), cuda)
    cs.relmae_reduce(d["c"], d["u"], M_out=M, workspace=ws)
    torch.cuda.synchronize()
    refM = O.rel_mae(d["c64"], d["u64"])
    if n == 0:
        assert M.item() == 0.0
    else:
        assert abs(M.item() - refM) <= 1e-6 * refM


def test_relmae_degenerate_cases(cuda):
    ws = cs.new_workspace(64, cs.CFG_F32, cuda)
    M = torch.zeros(1, dtype=torch.float64, device=cuda)
    z = torch.zeros(64, device=cuda)
    one = torch.ones(64, device=cuda)
    cs.relmae_reduce(z, z, M_out=M, workspace=ws)
    assert M.item() == 0.0
    cs.relmae_reduce(one, z, M_out=M, workspace=ws)
    assert M.item() == math.inf
    cs.relmae_reduce(one, one, M_out=M, workspace=ws)
    assert M.item() == 0.0
    nan = one.clone()
    nan[5] = float("nan")
    cs.relmae_reduce(nan, one, M_out=M, workspace=ws)
    assert math.isnan(M.item())


def _with_inf(arr, dtype, positions, sign=1.0):
    """A copy of a stored array with +-inf at `positions` (storage form)."""
    out = np.array(arr, copy=True)
    if dtype == "f32":
        out[positions] = sign * np.inf
    else:
        out[positions] = 0x7F80 if sign > 0 else 0xFF80      # bf16 +-inf bits
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["ddim0", "ddim1", "flow", "reduce"])
def test_infinite_predictions(cuda, dtype, mode):
    """An infinite conditional prediction (u finite) makes the L1 sum infinite, so M = +inf as in
    the oracle; an infinite unconditional one makes M = inf/inf = NaN.  Elements away from the
    infinities match the oracle as usual; at them both sides are non-finite (the update's
    combined coefficients give +-inf where the pages' two-term DDIM form gives inf - inf = NaN)."""
    n = 70_003
    base = W.draw_prediction_pair(n, dtype, 77)
    pos = [5, 4096 * 3 + 1, n - 2]                  # vector path and ragged tail
    ab, abp = float(O.abar_linear()[600]), float(O.abar_linear()[580])
    ws = cs.new_workspace(n, _code(dtype), cuda)
    for which, sign, want in (("c", 1.0, "inf"), ("c", -1.0, "inf"), ("u", 1.0, "nan")):
        arrs = dict(base)
        arrs[which] = _with_inf(base[which], dtype, pos, sign)
        dev = {k: to_device_stored(arrs[k], dtype, cuda) for k in ("x", "c", "u")}
        f64 = {k: W.stored_to_f64(arrs[k], dtype) for k in ("x", "c", "u")}
        M = torch.zeros(1, dtype=torch.float64, device=cuda)
        out = torch.empty_like(dev["x"])
        with np.errstate(invalid="ignore", over="ignore"):     # the oracle's inf - inf
            if mode == "reduce":
                cs.relmae_reduce(dev["c"], dev["u"], M_out=M, workspace=ws)
                refM, ref = O.rel_mae(f64["c"], f64["u"]), None
            elif mode == "flow":
                cs.flow_step(out, dev["x"], dev["c"], dev["u"], w=3.5, t_cur=0.5, t_next=0.45,
                             M_out=M, workspace=ws)
                ref, refM = O.flow_step(f64["x"], f64["c"], f64["u"], dtype, 3.5, 0.5, 0.45)
            else:
                eta = 1.0 if mode == "ddim1" else 0.0
                cs.ddim_step(out, dev["x"], dev["c"], dev["u"], w=7.5, abar_t=ab, abar_prev=abp,
                             eta=eta, seed=5, step=3, M_out=M, workspace=ws)
                ref, refM = O.ddim_step(f64["x"], f64["c"], f64["u"], dtype, 7.5, ab, abp, eta,
                                        5, 3)
        torch.cuda.synchronize()
        got_M = M.item()
        if want == "inf":
            assert got_M == math.inf and refM == math.inf
        else:
            assert math.isnan(got_M) and math.isnan(refM)
        if ref is None:
            continue
        got = to_host_f64(out)
        fin = np.isfinite(ref)
        assert not fin[pos].any() and not np.isfinite(got[pos]).any()
        assert np.isfinite(got[fin]).all()
        _compare(got[fin], ref[fin], dtype, strict_ulp=(mode != "ddim1"))


def test_identical_branches_ignore_w(cuda):
    n = 10_001
    d = _inputs(n, "bf16", seed=13, cuda=cuda)
    ab, abp = float(O.abar_linear()[300]), float(O.abar_linear()[280])
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    outs = []
    for w in (0.0, 1.0, 7.5):
        o = torch.empty_like(d["x"])
        M = torch.zeros(1, dtype=torch.float64, device=cuda)
        cs.ddim_step(o, d["x"], d["u"], d["u"], w=w, abar_t=ab, abar_prev=abp, M_out=M, workspace=ws)
        torch.cuda.synchronize()
        assert M.item() == 0.0
        outs.append(o)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_step_is_deterministic(cuda):
    n = 3 * (1 << 20) + 5
    d = _inputs(n, "bf16", seed=17, cuda=cuda)
    ab, abp = float(O.abar_linear()[600]), float(O.abar_linear()[580])
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    res = []
    for _ in range(2):
        o = torch.empty_like(d["x"])
        M = torch.zeros(1, dtype=torch.float64, device=cuda)
        cs.ddim_step(o, d["x"], d["c"], d["u"], w=7.5, abar_t=ab, abar_prev=abp, eta=1.0, seed=1,
                     step=3, M_out=M, workspace=ws)
        torch.cuda.synchronize()
        res.append((o.clone(), M.item()))
    assert torch.equal(res[0][0], res[1][0])
    assert res[0][1] == res[1][1]


# ---------------------------------------------------------------------------
# Noise stream
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,seed,step,stream", [
    (1, 0, 0, 0), (7, 2, 5, 0), (4099, 0x123456789ABCDEF, 17, 0), (1 << 20, 2, 49, 3)])
def test_randn_matches_oracle(cuda, n, seed, step, stream):
    """The integer Philox stream is shared exactly (any word error moves z by O(1));
    the fp32 Box-Muller value is within 4 fp32 ulps of the fp64 one."""
    out = torch.empty(n, dtype=torch.float32, device=cuda)
    cs.randn(out, seed=seed, step=step, stream_id=stream)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = O.gaussian_noise(n, seed, step, stream)
    err = np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)
    assert err.max() <= 4 * 2.0**-23, err.max()


def test_randn_misaligned_output(cuda):
    n = 1001
    buf = torch.empty(n + 1, dtype=torch.float32, device=cuda)
    cs.randn(buf[1:], seed=4, step=1)
    torch.cuda.synchronize()
    ref = O.gaussian_noise(n, 4, 1)
    assert np.max(np.abs(buf[1:].cpu().numpy() - ref)) <= 4 * 2.0**-23 * 6


# ---------------------------------------------------------------------------
# Schedule rule on the device
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", json.loads((GOLDEN / "schedule_traces.json").read_text())["traces"],
                         ids=lambda c: c["name"])
def test_schedule_golden_on_device(cuda, case):
    M = [math.nan if v == "nan" else float(v) for v in case["M"]]
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=len(M), L=case["L"], g_slope=case["g_slope"], k=case["k"],
                        tau_cap=case["tau_cap"])
    for s, m in enumerate(M):
        cs.sched_observe(st, sp, s, m)
    got = cs.read_sched_state(st)
    for key, val in case["expect"].items():
        assert got[key] == val, (key, got[key], val)
    assert list(got["phase"]) == case["phase"]
    ref = O.schedule(np.array(M), case["L"], case["g_slope"], case["k"], case["tau_cap"])
    assert np.array_equal(got["G"], ref.G, equal_nan=True)
    assert got["flags"] == 0 and got["n_seen"] == len(M)


def test_schedule_random_traces_match_oracle(cuda):
    g = np.random.default_rng(21)
    for trial in range(20):
        N = int(g.integers(1, 80))
        M = np.abs(np.cumsum(g.standard_normal(N) * 0.01)) + 0.05
        L = int(g.integers(1, 8))
        gs = float(g.choice([1e-3, 5e-3, 0.0, 1.0]))
        k = int(g.integers(0, 20))
        cap = int(g.choice([-1, -1, int(g.integers(0, 100))]))
        st = cs.new_sched_state(cuda)
        sp = cs.SchedParams(n_steps=N, L=L, g_slope=gs, k=k, tau_cap=cap)
        for s in range(N):
            cs.sched_observe(st, sp, s, float(M[s]))
        got = cs.read_sched_state(st)
        ref = O.schedule(M, L, gs, k, cap)
        assert {k_: got[k_] for k_ in ref.as_dict()} == ref.as_dict(), trial
        assert np.array_equal(got["phase"], ref.phase)
        assert np.array_equal(got["G"], ref.G, equal_nan=True), trial


def test_schedule_signed_zero_inf_nan_traces(cuda):
    """The rule's comparisons on the device follow IEEE semantics exactly: negative M,
    -0.0 against +0.0, infinities and NaN (which compares false), against the oracle."""
    inf, nan = math.inf, math.nan
    traces = [
        [0.3, -0.0, 0.0, -0.0, 0.2, 0.2, -1.0, -1.0, 0.5, 0.5],
        [1.0, 2.0, inf, inf, 3.0, -inf, 0.0, 0.0, 1e-300, 0.0],
        [nan, 0.1, 0.1, nan, 0.1001, 0.1, -0.1, -0.1, 0.0, -0.0],
        [5.0, 4.0, 3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0],
    ]
    for L in (1, 2, 3):
        for gs in (1e-3, 0.0, -0.0, 1.0, 5e-324):
            for M in traces:
                M = np.array(M, dtype=np.float64)
                st = cs.new_sched_state(cuda)
                sp = cs.SchedParams(n_steps=len(M), L=L, g_slope=gs, k=2)
                for s_, m in enumerate(M):
                    cs.sched_observe(st, sp, s_, float(m))
                got = cs.read_sched_state(st)
                ref = O.schedule(M, L, gs, 2, -1)
                assert {k_: got[k_] for k_ in ref.as_dict()} == ref.as_dict(), (L, gs, M)
                assert np.array_equal(got["G"], ref.G, equal_nan=True)
                assert np.array_equal(got["phase"], ref.phase)


@pytest.mark.parametrize("L", [1, 2, 3, 5, 7, 10, 11, 13, 97, 1000])
def test_slope_is_ieee_division(cuda, L):
    """G_s on the device equals fp64 (M_s - M_{s-L}) / L bit for bit, over traces of
    widely varying magnitude (including exact repeats, i.e. zero differences)."""
    g = np.random.default_rng(1000 + L)
    N = 1024
    M = np.abs(g.standard_normal(N)) * 10.0 ** g.integers(-30, 30, N)
    M[L + 5] = M[5]                                  # a zero difference
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=N, L=L, g_slope=1e-3, k=3)
    for s_ in range(N):
        cs.sched_observe(st, sp, s_, float(M[s_]))
    got = cs.read_sched_state(st)["G"]
    ref = np.full(N, np.nan)
    ref[L:] = (M[L:] - M[:-L]) / float(L)
    assert np.array_equal(got, ref, equal_nan=True)


def test_schedule_flags_out_of_order(cuda):
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=10)
    cs.sched_observe(st, sp, 0, 1.0)
    cs.sched_observe(st, sp, 2, 1.0)
    got = cs.read_sched_state(st)
    assert got["flags"] & 1
    cs.sched_observe(st, sp, 0, 1.0)      # step 0 starts a new run
    assert cs.read_sched_state(st)["flags"] == 0


# ---------------------------------------------------------------------------
# Deferred reductions (CFG_SCHED_DEFER)
# ---------------------------------------------------------------------------
def _step_sequence(cuda, defer, n=200_003, N=12, dtype="bf16"):
    """N consecutive DDIM steps on fixed random inputs; returns (x, per-step M, state)."""
    code = _code(dtype)
    preds = [_inputs(n, dtype, seed=400 + s, cuda=cuda) for s in range(N)]
    abar = O.abar_linear()
    ts = O.ddim_timesteps(N)
    x = preds[0]["x"].clone()
    Mbuf = torch.full((N,), -1.0, dtype=torch.float64, device=cuda)
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=N, L=2, g_slope=0.01, k=3, defer=defer)
    ws = cs.new_workspace(n, code, cuda)
    for s in range(N):
        abp = 1.0 if s == N - 1 else float(abar[ts[s + 1]])
        cs.ddim_step(x, x, preds[s]["c"], preds[s]["u"], w=4.0, abar_t=float(abar[ts[s]]),
                     abar_prev=abp, eta=0.5, seed=9, step=s, M_out=Mbuf[s:s + 1], state=st,
                     sched=sp, workspace=ws)
    torch.cuda.synchronize()
    return x.clone(), Mbuf.cpu().numpy(), cs.read_sched_state(st), preds


def test_deferred_sequence_equals_synchronous(cuda):
    xs, Ms, sts, preds = _step_sequence(cuda, defer=False)
    xd, Md, std, _ = _step_sequence(cuda, defer=True)
    assert torch.equal(xs, xd)
    assert np.array_equal(Ms, Md) and np.all(Ms >= 0)
    for key in ("n_seen", "tau1p", "argmin", "tau_cap", "tau1", "tau2", "decided_at", "flags"):
        assert sts[key] == std[key], key
    assert np.array_equal(sts["M"], std["M"]) and np.array_equal(sts["phase"], std["phase"])
    # and the trace is the oracle's rel-MAE of each step's stored predictions
    for s, p in enumerate(preds):
        assert abs(Ms[s] / O.rel_mae(p["c64"], p["u64"]) - 1) <= 1e-6


def test_deferred_step_completed_by_flush(cuda):
    n = 70_001
    d = _inputs(n, "bf16", seed=41, cuda=cuda)
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=10, defer=True)
    M = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
    out = torch.empty_like(d["x"])
    ab, abp = float(O.abar_linear()[900]), float(O.abar_linear()[880])
    cs.ddim_step(out, d["x"], d["c"], d["u"], w=3.0, abar_t=ab, abar_prev=abp, step=0, M_out=M,
                 state=st, sched=sp, workspace=ws)
    torch.cuda.synchronize()
    assert M.item() == -1.0                      # deferred: not written yet
    cs.workspace_flush(ws)
    torch.cuda.synchronize()
    assert abs(M.item() / O.rel_mae(d["c64"], d["u64"]) - 1) <= 1e-6
    assert cs.read_sched_state(st)["n_seen"] == 1
    cs.workspace_flush(ws)                       # nothing pending: a no-op
    torch.cuda.synchronize()
    assert cs.read_sched_state(st)["n_seen"] == 1


def test_deferred_same_parity_clash_is_flagged(cuda):
    n = 30_000
    d = _inputs(n, "bf16", seed=43, cuda=cuda)
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=10, defer=True)
    out = torch.empty_like(d["x"])
    ab, abp = float(O.abar_linear()[900]), float(O.abar_linear()[880])
    for step in (0, 2):                          # step 1 skipped: both write slot 0
        cs.ddim_step(out, d["x"], d["c"], d["u"], w=3.0, abar_t=ab, abar_prev=abp, step=step,
                     state=st, sched=sp, workspace=ws)
    cs.workspace_flush(ws)
    torch.cuda.synchronize()
    got = cs.read_sched_state(st)
    assert got["flags"] & cs.SCHED_FLAG_DEFER_CLASH
    assert got["flags"] & cs.SCHED_FLAG_OUT_OF_ORDER     # step 2 recorded after step 0 was dropped


def test_deferred_results_lag(cuda):
    """In a run of deferring steps, step s's M is written by step s + 1's launch and its schedule
    update by step s + 2's: after steps 0..k, M[0..k-1] are final, M[k] is pending and the rule
    has seen steps 0..k-2, until a flush completes both."""
    N, k = 10, 5
    n = 50_000
    preds = [_inputs(n, "bf16", seed=600 + s, cuda=cuda) for s in range(k + 1)]
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=N, L=2, g_slope=0.01, k=3, defer=True)
    Ms = torch.full((k + 1,), -1.0, dtype=torch.float64, device=cuda)
    out = torch.empty_like(preds[0]["x"])
    ab, abp = float(O.abar_linear()[900]), float(O.abar_linear()[880])
    for s in range(k + 1):
        cs.ddim_step(out, preds[s]["x"], preds[s]["c"], preds[s]["u"], w=3.0, abar_t=ab,
                     abar_prev=abp, step=s, M_out=Ms[s:s + 1], state=st, sched=sp, workspace=ws)
    torch.cuda.synchronize()
    M = Ms.cpu().numpy()
    refs = [O.rel_mae(p["c64"], p["u64"]) for p in preds]
    for s in range(k):
        assert abs(M[s] / refs[s] - 1) <= 1e-6, s
    assert M[k] == -1.0
    assert cs.read_sched_state(st)["n_seen"] == k - 1
    cs.workspace_flush(ws)
    torch.cuda.synchronize()
    M = Ms.cpu().numpy()
    assert all(abs(M[s] / refs[s] - 1) <= 1e-6 for s in range(k + 1))
    got = cs.read_sched_state(st)
    assert got["n_seen"] == k + 1 and got["flags"] == 0


def test_reduce_call_mid_run_completes_pending_steps(cuda):
    """A rel-MAE call on the same workspace in the middle of a deferred run completes the pending
    work (the last step's reduction and the schedule update before it); the run then goes on
    and ends with the synchronous run's results and state."""
    N, n = 8, 40_003
    preds = [_inputs(n, "bf16", seed=700 + s, cuda=cuda) for s in range(N)]
    abar = O.abar_linear()
    ts = O.ddim_timesteps(N)

    def run(defer, interrupt):
        x = preds[0]["x"].clone()
        Mbuf = torch.full((N,), -1.0, dtype=torch.float64, device=cuda)
        Mr = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        st = cs.new_sched_state(cuda)
        sp = cs.SchedParams(n_steps=N, L=2, g_slope=0.01, k=3, defer=defer)
        ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
        for s in range(N):
            abp = 1.0 if s == N - 1 else float(abar[ts[s + 1]])
            cs.ddim_step(x, x, preds[s]["c"], preds[s]["u"], w=4.0, abar_t=float(abar[ts[s]]),
                         abar_prev=abp, eta=0.0, seed=9, step=s, M_out=Mbuf[s:s + 1], state=st,
                         sched=sp, workspace=ws)
            if interrupt and s == 3:
                cs.relmae_reduce(preds[0]["c"], preds[0]["u"], M_out=Mr, workspace=ws)
                torch.cuda.synchronize()
                assert np.all(Mbuf[:4].cpu().numpy() >= 0)      # steps 0..3 all complete
                assert cs.read_sched_state(st)["n_seen"] == 4
                assert abs(Mr.item() / O.rel_mae(preds[0]["c64"], preds[0]["u64"]) - 1) <= 1e-6
        torch.cuda.synchronize()
        return x.clone(), Mbuf.cpu().numpy(), cs.read_sched_state(st)

    xs, Ms, sts = run(False, False)
    xd, Md, std = run(True, True)
    assert torch.equal(xs, xd) and np.array_equal(Ms, Md)
    for key in ("n_seen", "tau1p", "argmin", "tau_cap", "tau1", "tau2", "decided_at", "flags"):
        assert sts[key] == std[key], key
    assert np.array_equal(sts["M"], std["M"]) and np.array_equal(sts["phase"], std["phase"])


def test_in_launch_call_completes_pending_step(cuda):
    n = 40_000
    d = _inputs(n, "f32", seed=47, cuda=cuda)
    ws = cs.new_workspace(n, cs.CFG_F32, cuda)
    st = cs.new_sched_state(cuda)
    sp = cs.SchedParams(n_steps=5, defer=True)
    M0 = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
    M1 = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
    out = torch.empty_like(d["x"])
    ab, abp = float(O.abar_linear()[900]), float(O.abar_linear()[880])
    cs.ddim_step(out, d["x"], d["c"], d["u"], w=3.0, abar_t=ab, abar_prev=abp, step=0, M_out=M0,
                 state=st, sched=sp, workspace=ws)
    cs.relmae_reduce(d["x"], d["u"], M_out=M1, workspace=ws)
    torch.cuda.synchronize()
    assert abs(M0.item() / O.rel_mae(d["c64"], d["u64"]) - 1) <= 1e-6
    assert abs(M1.item() / O.rel_mae(d["x64"], d["u64"]) - 1) <= 1e-6


def test_step_beyond_2_31_elements(cuda):
    """One bf16 step over n = 2^31 + 13 elements (64-bit indexing; ~17 GB of HBM).  M is known
    exactly by construction (u = +-2^k, c = u (1 + 2^-4) is exact in bf16, so every
    |c - u| = 2^-4 |u| and M = 2^-4); x_out is checked against the oracle's update on sampled
    elements, including both sides of 2^31 and the ragged tail, with eta = 1 noise."""
    free, _ = torch.cuda.mem_get_info(cuda)
    n = 2**31 + 13
    if free < 4 * 2 * n + (2 << 30):
        pytest.skip("needs ~18 GB of free device memory")
    g = torch.Generator(device=cuda)
    g.manual_seed(123)
    x = torch.empty(n, dtype=torch.bfloat16, device=cuda)
    u = torch.empty_like(x)
    chunk = 1 << 28
    for i0 in range(0, n, chunk):
        m = min(chunk, n - i0)
        x[i0:i0 + m] = torch.randn(m, generator=g, device=cuda).to(torch.bfloat16)
        e = torch.randint(-6, 6, (m,), generator=g, device=cuda).float()
        sgn = torch.randint(0, 2, (m,), generator=g, device=cuda).float() * 2 - 1
        u[i0:i0 + m] = (sgn * torch.exp2(e)).to(torch.bfloat16)
    c = torch.empty_like(u)
    for i0 in range(0, n, chunk):
        m = min(chunk, n - i0)
        c[i0:i0 + m] = (u[i0:i0 + m].float() * (1.0 + 2.0**-4)).to(torch.bfloat16)
    out = torch.empty_like(x)
    M = torch.zeros(1, dtype=torch.float64, device=cuda)
    abar = O.abar_linear()
    ab, abp = float(abar[300]), float(abar[280])
    cs.ddim_step(out, x, c, u, w=5.0, abar_t=ab, abar_prev=abp, eta=1.0, seed=77, step=4, M_out=M,
                 workspace=cs.new_workspace(n, cs.CFG_BF16, cuda))
    torch.cuda.synchronize()
    assert abs(M.item() - 2.0**-4) <= 1e-6 * 2.0**-4
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, n, 2000), np.arange(2**31 - 40, 2**31 + 13),
                                    np.arange(n - 20, n), np.arange(0, 20)]))
    it = torch.from_numpy(idx).to(cuda)
    xs, cs_, us, got = (t[it].float().cpu().numpy().astype(np.float64) for t in (x, c, u, out))
    z = np.array([O.gaussian_noise(1, 77, 4, start=int(i))[0] for i in idx])
    ref, _ = O.ddim_step(xs, cs_, us, "bf16", 5.0, ab, abp, 1.0, 77, 4, z=z)
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)) <= 2e-2
    # every sampled element within 1 bf16 ulp, or 2^-17 after cancellation (the single-step bound)
    ok = (ulp_distance_bf16(got, ref) <= 1) | (np.abs(got - ref) <= 2.0**-17)
    assert ok.all(), idx[~ok][:10]
    del x, u, c, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("exact", [False, True], ids=["bf16", "bf16_exact"])
def test_every_element_on_a_rounding_midpoint(cuda, exact):
    """A flow step whose exact result is a bf16 rounding midpoint at (nearly) every element:
    x = +-(1 + j 2^-7), v = c = -2^-6 (w = 1, u = 0) and dt = t_next - t_cur = -1/4, so
    x + dt v = x + 2^-8, half a bf16 ulp from x.  Ties go to even (the pages' fp64 step rounded
    once, as the oracle does), so even last bits stay and odd ones round to the neighbour.
    Correctly rounded, every element lies near a midpoint: each block's queue of near elements
    overflows, and the rest are recomputed by the thread that found them.  Every element must
    equal the oracle's in both roundings."""
    n = 3 * (1 << 20) + 5
    rng = np.random.default_rng(11)
    j = rng.integers(0, 128, n)
    x64 = np.where(rng.random(n) < 0.5, -1.0, 1.0) * (1.0 + j * 2.0**-7)
    c64, u64 = np.full(n, -2.0**-6), np.zeros(n)
    x, c, u = (torch.from_numpy(v).to(torch.bfloat16).to(cuda) for v in (x64, c64, u64))
    out = torch.empty_like(x)
    ws = cs.new_workspace(n, cs.CFG_BF16, cuda)
    cs.flow_step(out, x, c, u, w=1.0, t_cur=0.5, t_next=0.25, workspace=ws, exact_rounding=exact)
    torch.cuda.synchronize()
    ref, _ = O.flow_step(x64, c64, u64, "bf16", 1.0, 0.5, 0.25)
    got = to_host_f64(out)
    assert np.mean(np.abs(ref - x64) > 0) > 0.4          # about half the ties round away
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (bad[:10], got[bad[:10]], ref[bad[:10]], x64[bad[:10]])
