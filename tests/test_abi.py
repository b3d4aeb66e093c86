"""The C ABI without a GPU: exports, struct layout, argument validation, host helpers.

No call here launches anything: every invalid call is rejected by the library's
host-side checks, and the one test that passes validation (first calls from
several host threads) runs only where no CUDA device exists, so the library's
device lookup is the call that fails.
"""
import ctypes
import re
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

import cfg_guided_sampler_step_b300 as cs
from oracle import cfg_oracle as O

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "cfgstep.h"


def declared_symbols():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"CFG_API\s+[\w\s\*]+?\b(cfg_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("cfg_relmae_reduce", "cfg_ddim_step", "cfg_flow_step", "cfg_sampler_run",
                     "cfg_workspace_bytes", "cfg_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", str(cs.lib_path)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(cfg_\w+)", out))
    declared = set(declared_symbols())
    assert declared <= exported, declared - exported
    # nothing beyond the declared ABI is exported under the cfg_ prefix
    assert exported <= declared, exported - declared
    for name in declared:
        assert hasattr(cs.lib, name)


def test_struct_layout_matches_header(tmp_path):
    """sizeof/offsetof from a C compiler agree with the binding's ctypes mirrors."""
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "cfgstep.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m))
int main(void) {
  printf("cfg_sched_params %zu\n", sizeof(cfg_sched_params));
  printf("cfg_sched_state %zu\n", sizeof(cfg_sched_state));
  F(cfg_sched_params, L); F(cfg_sched_params, k); F(cfg_sched_params, g_slope);
  F(cfg_sched_params, tau_cap); F(cfg_sched_params, n_steps); F(cfg_sched_params, flags);
  F(cfg_sched_params, reserved);
  F(cfg_sched_state, n_seen); F(cfg_sched_state, tau1p); F(cfg_sched_state, argmin);
  F(cfg_sched_state, tau_cap); F(cfg_sched_state, tau1); F(cfg_sched_state, tau2);
  F(cfg_sched_state, decided_at); F(cfg_sched_state, flags); F(cfg_sched_state, min_M);
  F(cfg_sched_state, M); F(cfg_sched_state, G); F(cfg_sched_state, phase);
  F(cfg_sched_state, pad);
  printf("CFG_TAU_NONE %d\nCFG_SCHED_MAX_STEPS %d\n", CFG_TAU_NONE, CFG_SCHED_MAX_STEPS);
  printf("CFG_SCHED_DEFER %u\nCFG_SCHED_FLAG_DEFER_CLASH %u\n", CFG_SCHED_DEFER, CFG_SCHED_FLAG_DEFER_CLASH);
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", str(HEADER.parent), "-o", str(exe), str(src)],
                   check=True)
    c = dict(line.rsplit(" ", 1) for line in
             subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
             if line)
    c = {k: int(v) for k, v in c.items()}
    assert c["cfg_sched_params"] == ctypes.sizeof(cs.SchedParamsC)
    assert c["cfg_sched_state"] == ctypes.sizeof(cs.SchedStateC)
    assert c["cfg_sched_state"] % 16 == 0          # arrays of states stay 16-byte aligned
    for name, typ in (("cfg_sched_params", cs.SchedParamsC), ("cfg_sched_state", cs.SchedStateC)):
        for field, _ in typ._fields_:
            assert c[f"{name}.{field}"] == getattr(typ, field).offset, (name, field)
    assert c["CFG_TAU_NONE"] == cs.TAU_NONE == O.TAU_NONE
    assert c["CFG_SCHED_MAX_STEPS"] == cs.SCHED_MAX_STEPS
    assert c["CFG_SCHED_DEFER"] == cs.SCHED_DEFER
    assert c["CFG_SCHED_FLAG_DEFER_CLASH"] == cs.SCHED_FLAG_DEFER_CLASH


def test_version_and_workspace_size():
    assert "sm_103a" in cs.version()
    nb = cs.workspace_bytes(1 << 20, cs.CFG_BF16)
    assert nb > 0 and nb % 16 == 0
    assert cs.workspace_bytes(0, cs.CFG_F32) == nb          # independent of n and device
    assert cs.workspace_bytes(-1, cs.CFG_F32) == 0
    assert cs.workspace_bytes(10, 5) == 0


def test_host_helpers_match_oracle():
    for T, b0, b1 in ((1000, 1e-4, 0.02), (1, 0.01, 0.01), (37, 0.0, 0.5)):
        assert np.array_equal(cs.abar_linear(T, b0, b1), O.abar_linear(T, b0, b1))
    for N, T in ((50, 1000), (28, 1000), (1, 1000), (7, 10), (1000, 1000), (3, 4)):
        assert np.array_equal(cs.ddim_timesteps(N, T), O.ddim_timesteps(N, T))


FAKE = 0x100000  # a 16-byte aligned non-NULL address; never dereferenced (calls fail first)


def _ddim(**kw):
    a = dict(x_out=FAKE, x_in=FAKE, pc=FAKE, pu=FAKE, n=16, dtype=cs.CFG_BF16, w=5.0, ab=0.5,
             abp=0.6, eta=0.0, seed=0, step=0, M=None, st=None, sp=None, ws=FAKE,
             wsb=cs.workspace_bytes(16, 1), stream=None)
    a.update(kw)
    return cs.lib.cfg_ddim_step(a["x_out"], a["x_in"], a["pc"], a["pu"], a["n"], a["dtype"], a["w"],
                                a["ab"], a["abp"], a["eta"], a["seed"], a["step"], a["M"], a["st"],
                                a["sp"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), -2),
    (dict(n=-1), -1),
    (dict(pc=None), -1),
    (dict(x_in=None), -1),
    (dict(w=float("nan")), -1),
    (dict(w=float("inf")), -1),
    (dict(ab=0.0), -1),
    (dict(ab=1.0), -1),
    (dict(abp=0.0), -1),
    (dict(abp=1.5), -1),
    (dict(eta=-0.5), -1),
    (dict(eta=float("nan")), -1),
    (dict(eta=1.0, ab=0.7, abp=0.6), -1),       # eta > 0 needs abar_prev >= abar_t
    (dict(eta=3.0, ab=0.5, abp=0.6), -1),       # 1 - abar_prev - sigma^2 < 0
    (dict(step=-1), -1),
    (dict(ws=None), -3),
    (dict(ws=FAKE + 8), -3),
    (dict(wsb=100), -3),
])
def test_ddim_step_rejects_invalid_arguments(kw, code):
    assert _ddim(**kw) == code
    assert cs.lib.cfg_last_error().decode() != ""


def test_schedule_arguments_validated():
    st = FAKE
    for params, step in ((dict(L=0), 0), (dict(k=-1), 0), (dict(g_slope=float("nan")), 0),
                         (dict(tau_cap=-2), 0), (dict(n_steps=0), 0), (dict(n_steps=2000), 0),
                         (dict(), 50), (dict(), -1)):
        p = dict(n_steps=50, L=5, g_slope=1e-3, k=10, tau_cap=-1)
        p.update(params)
        sp = cs.SchedParams(**p)
        assert _ddim(st=st, sp=ctypes.byref(sp.c), step=step) == -1
        assert cs.lib.cfg_sched_observe(st, ctypes.byref(sp.c), step, 0.5, None) == -1
    bad = cs.SchedParams(n_steps=10)
    bad.c.flags = 4
    assert _ddim(st=st, sp=ctypes.byref(bad.c)) == -1          # unknown flag bit
    bad = cs.SchedParams(n_steps=10)
    bad.c.reserved = 1
    assert _ddim(st=st, sp=ctypes.byref(bad.c)) == -1
    sp = cs.SchedParams(n_steps=10)
    # state without parameters (or the reverse) is rejected
    assert _ddim(st=st, sp=None) == -1
    assert _ddim(st=None, sp=ctypes.byref(sp.c)) == -1
    assert _ddim(st=FAKE + 4, sp=ctypes.byref(sp.c)) == -1          # misaligned state
    assert _ddim(st=FAKE + 8, sp=ctypes.byref(sp.c)) == -1          # state needs 16 bytes


def test_other_entry_points_validate():
    L = cs.lib
    wsb = cs.workspace_bytes(16, 1)
    assert L.cfg_relmae_reduce(FAKE, FAKE, 16, 9, None, None, None, 0, FAKE, wsb, None) == -2
    assert L.cfg_relmae_reduce(None, FAKE, 16, 1, None, None, None, 0, FAKE, wsb, None) == -1
    assert L.cfg_flow_step(FAKE, FAKE, FAKE, FAKE, 16, 1, float("nan"), 1.0, 0.5, 0, None, None,
                           None, FAKE, wsb, None) == -1
    assert L.cfg_flow_step(FAKE, FAKE, FAKE, FAKE, 16, 1, 2.0, float("inf"), 0.5, 0, None, None,
                           None, FAKE, wsb, None) == -1
    assert L.cfg_randn(None, 16, 0, 0, 0, None) == -1
    assert L.cfg_randn(FAKE, -3, 0, 0, 0, None) == -1
    assert L.cfg_randn(None, 0, 0, 0, 0, None) == 0          # empty request: nothing to do
    assert L.cfg_workspace_init(None, wsb, None) == -3
    assert L.cfg_workspace_init(FAKE, 8, None) == -3
    assert L.cfg_workspace_flush(None, wsb, None) == -3
    assert L.cfg_workspace_flush(FAKE, wsb - 16, None) == -3
    assert L.cfg_abar_linear(None, 10, 0.1, 0.2) == -1
    out = np.empty(4)
    assert L.cfg_abar_linear(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), 4, 0.1, 1.5) == -1
    ts = np.empty(4, dtype=np.int32)
    assert L.cfg_ddim_timesteps(ts.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), 5, 4) == -1


def test_host_buffer_helpers_validate():
    """cfg_host_alloc / cfg_host_free / cfg_copy_async reject bad arguments before any CUDA call
    (so this runs without a GPU)."""
    ptr = ctypes.c_void_p(1)
    assert cs.lib.cfg_host_alloc(0, ctypes.byref(ptr)) == -1 and ptr.value is None
    assert cs.lib.cfg_host_alloc(16, None) == -1
    assert cs.lib.cfg_host_free(None) == 0
    assert cs.lib.cfg_copy_async(None, None, 0, None) == 0          # zero bytes: nothing to do
    assert cs.lib.cfg_copy_async(None, FAKE, 16, None) == -1
    assert cs.lib.cfg_copy_async(FAKE, None, 16, None) == -1
    with pytest.raises(ValueError):
        cs.copy_async(torch.empty(4), torch.empty(5))               # sizes differ
    with pytest.raises(ValueError):
        cs.copy_async(torch.empty(4, 2).t(), torch.empty(8))        # not contiguous


def test_sampler_run_validates_before_any_callback():
    called = []

    def denoise(*a):
        called.append(a)
        return 0

    cb = cs.DENOISE_FN(denoise)
    sp = cs.SchedParams(n_steps=4)
    abar = np.ascontiguousarray(O.abar_linear(10))
    bad_ts = np.array([9, 6, 3, 10], dtype=np.int32)      # 10 is outside [0, T)
    r = cs.lib.cfg_sampler_run(FAKE, 16, 1, cs.CFG_MODE_DDIM,
                               abar.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), 10,
                               bad_ts.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), None, 4, 5.0,
                               0.0, 0, cb, None, FAKE, FAKE, ctypes.byref(sp.c), FAKE, 0, FAKE,
                               cs.workspace_bytes(16, 1), None)
    assert r == -1 and not called
    r = cs.lib.cfg_sampler_run(FAKE, 16, 1, 7, None, 0, None, None, 4, 5.0, 0.0, 0, cb, None, FAKE,
                               FAKE, ctypes.byref(sp.c), FAKE, 0, FAKE, cs.workspace_bytes(16, 1),
                               None)
    assert r == -1 and not called
    sp5 = cs.SchedParams(n_steps=5)
    r = cs.lib.cfg_sampler_run(FAKE, 16, 1, cs.CFG_MODE_FLOW, None, 0, None, None, 4, 5.0, 0.0, 0,
                               cb, None, FAKE, FAKE, ctypes.byref(sp5.c), FAKE, 0, FAKE,
                               cs.workspace_bytes(16, 1), None)
    assert r == -1 and not called


def test_division_by_reciprocal_and_fma_is_correctly_rounded():
    """The schedule's slope G = d / L is formed on the device as q0 = RN(d * y),
    r = RN(d - q0 * L) (an FMA), G = RN(q0 + r * y) (an FMA) with y = RN(1/L);
    Markstein's theorem says this is the correctly rounded quotient.  Checked here
    with exact rational arithmetic (Fraction -> float rounds to nearest even) against
    Python's correctly rounded float division, on random and adversarial d and L."""
    from fractions import Fraction as F
    g = np.random.default_rng(77)
    Ls = [1, 2, 3, 5, 6, 7, 9, 10, 11, 13, 25, 97, 1000, 1023, 2**20 + 1, 2**31 - 1]
    ds = list(g.standard_normal(3000) * 10.0 ** g.integers(-250, 250, 3000))
    ds += [float(np.nextafter(1.0, 2.0)), 1.0 - 2.0**-53, 2.0**-890, 3.0 * 2.0**-880, 1e300]
    for L in Ls:
        y = F(1.0 / L)
        for d in ds:
            dF = F(d)
            q0 = float(dF * y)
            r = float(dF - F(q0) * L)
            assert F(r) == dF - F(q0) * L          # the residual is exact
            q = float(F(q0) + F(r) * y)
            assert q == d / L, (d, L, q, d / L)


def test_adjacent_sampler_tables_match_oracle():
    """The library's host tables (cosine abar, timestep spacings) equal the oracle's."""
    for T, s, mb in ((1000, 0.008, 0.999), (10, 0.0, 0.5), (1, 0.1, 0.9)):
        assert np.array_equal(cs.abar_cosine(T, s, mb), O.abar_cosine(T, s, mb))
    for N, T in ((50, 1000), (30, 1000), (7, 100), (1, 10), (10, 10)):
        for sp in ("linspace", "leading", "trailing"):
            assert np.array_equal(cs.timesteps(N, T, sp), O.timesteps(N, T, sp)), (N, T, sp)
    out = np.empty(4, dtype=np.int32)
    p = out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert cs.lib.cfg_timesteps(p, 4, 10, 3) == -1                 # unknown spacing
    assert cs.lib.cfg_timesteps(p, 11, 10, 1) == -1                # n_steps > T
    d = np.empty(4)
    pd = d.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    assert cs.lib.cfg_abar_cosine(pd, 4, -0.1, 0.999) == -1
    assert cs.lib.cfg_abar_cosine(pd, 4, 0.008, 1.0) == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_first_calls_from_many_threads_without_a_device():
    """Calls that pass argument validation reach the library's per-device lookups (SM count,
    static scratch address).  Made at once from several host threads with no device present,
    each must fail cleanly with CFG_ERR_CUDA and its own thread's message; the lookups are
    atomic, so concurrent first calls neither crash nor leave a bad cached value."""
    import threading
    sp = cs.SchedParams(n_steps=4)
    fake = 1 << 20                      # 16-byte aligned, never dereferenced on the host
    results = []
    lock = threading.Lock()
    start = threading.Barrier(8)

    def worker(i):
        start.wait()
        for _ in range(50):
            if i % 2:
                rc = cs.lib.cfg_ddim_step(fake, fake, fake, fake, 1024, cs.CFG_BF16, 2.0, 0.5, 0.6,
                                          0.0, 0, 0, None, fake, ctypes.byref(sp.c), fake,
                                          cs.workspace_bytes(1024, cs.CFG_BF16), None)
            else:
                rc = cs.lib.cfg_ddim_step_static_ws(fake, fake, fake, fake, 1024, cs.CFG_BF16, 2.0,
                                                    0.5, 0.6, 0.0, 0, 0, None, fake,
                                                    ctypes.byref(sp.c), None)
            msg = cs.lib.cfg_last_error().decode()
            with lock:
                results.append((rc, msg))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(60)
    assert len(results) == 8 * 50
    for rc, msg in results:
        assert cs.STATUS_NAMES[rc] == "CFG_ERR_CUDA", (rc, msg)
        assert "cudaGetDevice" in msg, msg
