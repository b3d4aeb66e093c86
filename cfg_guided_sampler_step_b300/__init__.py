"""Python binding of the CFG sampler-step library (``libcfgstep.so``).

Argument marshalling only: every entry point forwards device pointers, sizes
and the current CUDA stream to the C ABI declared in ``include/cfgstep.h``;
all arithmetic of the step runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.

The library must be built (``python cfg_guided_sampler_step_b300/_build.py``
or ``__graft_entry__.build()``); importing this package raises if it is
missing -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
from ctypes import (CFUNCTYPE, POINTER, Structure, c_char_p, c_double, c_float, c_int32, c_int64,
                    c_size_t, c_uint8, c_uint32, c_uint64, c_void_p)
from pathlib import Path
from typing import Callable, Dict, Optional

import numpy as np

__all__ = [
    "CFG_F32", "CFG_BF16", "CFG_BF16_EXACT", "CFG_MODE_DDIM", "CFG_MODE_FLOW", "TAU_NONE", "SCHED_MAX_STEPS",
    "CfgError", "SchedParams", "lib", "lib_path", "workspace_bytes", "new_workspace",
    "new_sched_state", "read_sched_state", "workspace_flush", "SCHED_DEFER", "relmae_reduce", "ddim_step", "flow_step",
    "sched_observe", "randn", "abar_linear", "ddim_timesteps", "abar_cosine", "timesteps",
    "sampler_run", "sampler_run_branches", "version", "pinned_empty", "copy_async",
]

CFG_F32, CFG_BF16, CFG_BF16_EXACT = 0, 1, 2
SCHED_DEFER = 1
SCHED_FLAG_OUT_OF_ORDER, SCHED_FLAG_DEFER_CLASH = 1, 2
CFG_MODE_DDIM, CFG_MODE_FLOW = 0, 1
TAU_NONE = 2**31 - 1
SCHED_MAX_STEPS = 1024
STATUS_NAMES = {0: "CFG_OK", -1: "CFG_ERR_INVALID_ARG", -2: "CFG_ERR_UNSUPPORTED_DTYPE",
                -3: "CFG_ERR_WORKSPACE", -4: "CFG_ERR_CUDA", -5: "CFG_ERR_CALLBACK"}

lib_path = Path(__file__).resolve().parent / "libcfgstep.so"


class CfgError(RuntimeError):
    """A negative status from the library, with its message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class SchedParamsC(Structure):
    _fields_ = [("L", c_int32), ("k", c_int32), ("g_slope", c_double), ("tau_cap", c_int32),
                ("n_steps", c_int32), ("flags", c_uint32), ("reserved", c_int32)]


class SchedStateC(Structure):
    _fields_ = [("n_seen", c_int32), ("tau1p", c_int32), ("argmin", c_int32), ("tau_cap", c_int32),
                ("tau1", c_int32), ("tau2", c_int32), ("decided_at", c_int32), ("flags", c_uint32),
                ("min_M", c_double), ("M", c_double * SCHED_MAX_STEPS),
                ("G", c_double * SCHED_MAX_STEPS), ("phase", c_uint8 * SCHED_MAX_STEPS),
                ("pad", c_uint8 * 8)]


DENOISE_FN = CFUNCTYPE(c_int32, c_void_p, c_int32, c_int32, c_double, c_void_p, c_void_p, c_void_p,
                       c_void_p)
BRANCH_FN = CFUNCTYPE(c_int32, c_void_p, c_int32, c_int32, c_int32, c_double, c_void_p, c_void_p,
                      c_void_p)


def _load() -> ctypes.CDLL:
    if not lib_path.exists():
        raise ImportError(
            f"{lib_path} is not built; run `python cfg_guided_sampler_step_b300/_build.py` "
            "(needs nvcc). There is no CPU fallback.")
    L = ctypes.CDLL(str(lib_path))
    vp = c_void_p
    sigs = {
        "cfg_last_error": (c_char_p, []),
        "cfg_version": (c_char_p, []),
        "cfg_workspace_bytes": (c_size_t, [c_int64, c_int32]),
        "cfg_workspace_init": (c_int32, [vp, c_size_t, vp]),
        "cfg_workspace_flush": (c_int32, [vp, c_size_t, vp]),
        "cfg_relmae_reduce": (c_int32, [vp, vp, c_int64, c_int32, vp, vp, POINTER(SchedParamsC),
                                        c_int32, vp, c_size_t, vp]),
        "cfg_ddim_step": (c_int32, [vp, vp, vp, vp, c_int64, c_int32, c_float, c_double, c_double,
                                    c_float, c_uint64, c_int32, vp, vp, POINTER(SchedParamsC), vp,
                                    c_size_t, vp]),
        "cfg_ddim_step_static_ws": (c_int32, [vp, vp, vp, vp, c_int64, c_int32, c_float, c_double,
                                              c_double, c_float, c_uint64, c_int32, vp, vp,
                                              POINTER(SchedParamsC), vp]),
        "cfg_flow_step": (c_int32, [vp, vp, vp, vp, c_int64, c_int32, c_float, c_double, c_double,
                                    c_int32, vp, vp, POINTER(SchedParamsC), vp, c_size_t, vp]),
        "cfg_relmae_reduce_batched": (c_int32, [vp, vp, c_int64, c_int32, c_int32, vp, vp,
                                                POINTER(SchedParamsC), c_int32, vp, c_size_t, vp]),
        "cfg_ddim_step_batched": (c_int32, [vp, vp, vp, vp, c_int64, c_int32, c_int32, c_float,
                                            c_double, c_double, c_float, c_uint64, c_int32, vp, vp,
                                            POINTER(SchedParamsC), vp, c_size_t, vp]),
        "cfg_flow_step_batched": (c_int32, [vp, vp, vp, vp, c_int64, c_int32, c_int32, c_float,
                                            c_double, c_double, c_int32, vp, vp,
                                            POINTER(SchedParamsC), vp, c_size_t, vp]),
        "cfg_workspace_init_batched": (c_int32, [vp, c_size_t, c_int32, vp]),
        "cfg_workspace_flush_batched": (c_int32, [vp, c_size_t, c_int32, vp]),
        "cfg_sched_observe": (c_int32, [vp, POINTER(SchedParamsC), c_int32, c_double, vp]),
        "cfg_sampler_run_branches": (c_int32, [vp, c_int64, c_int32, c_int32, POINTER(c_double),
                                               c_int32, POINTER(c_int32), POINTER(c_double),
                                               c_int32, c_float, c_float, c_uint64, BRANCH_FN,
                                               vp, vp, vp, vp, vp, POINTER(SchedParamsC), vp,
                                               c_int32, vp, c_size_t, vp]),
        "cfg_randn": (c_int32, [vp, c_int64, c_uint64, c_uint32, c_uint32, vp]),
        "cfg_host_alloc": (c_int32, [c_size_t, POINTER(c_void_p)]),
        "cfg_host_free": (c_int32, [vp]),
        "cfg_copy_async": (c_int32, [vp, vp, c_size_t, vp]),
        "cfg_abar_linear": (c_int32, [POINTER(c_double), c_int32, c_double, c_double]),
        "cfg_ddim_timesteps": (c_int32, [POINTER(c_int32), c_int32, c_int32]),
        "cfg_abar_cosine": (c_int32, [POINTER(c_double), c_int32, c_double, c_double]),
        "cfg_timesteps": (c_int32, [POINTER(c_int32), c_int32, c_int32, c_int32]),
        "cfg_sampler_run": (c_int32, [vp, c_int64, c_int32, c_int32, POINTER(c_double), c_int32,
                                      POINTER(c_int32), POINTER(c_double), c_int32, c_float,
                                      c_float, c_uint64, DENOISE_FN, vp, vp, vp,
                                      POINTER(SchedParamsC), vp, c_int32, vp, c_size_t, vp]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def version() -> str:
    return lib.cfg_version().decode()


def _check(status: int) -> None:
    if status != 0:
        raise CfgError(status, lib.cfg_last_error().decode())


# ---------------------------------------------------------------------------
# torch plumbing
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t, exact_rounding: bool = False) -> int:
    """Storage code of a tensor; ``exact_rounding`` selects CFG_BF16_EXACT for bf16 (the step
    rounds the exact value correctly; fp32 steps are compensated either way)."""
    torch = _torch()
    if t.dtype == torch.float32:
        return CFG_F32
    if t.dtype == torch.bfloat16:
        return CFG_BF16_EXACT if exact_rounding else CFG_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev_ptr(t, name: str) -> int:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class SchedParams:
    """tau1/tau2 rule parameters (L, k, g_slope, tau_cap, n_steps); see cfg_sched_params."""

    def __init__(self, n_steps: int, L: int = 5, g_slope: float = 1e-3, k: int = 10,
                 tau_cap: int = -1, defer: bool = False):
        self.c = SchedParamsC(L=L, k=k, g_slope=g_slope, tau_cap=tau_cap, n_steps=n_steps,
                              flags=SCHED_DEFER if defer else 0, reserved=0)

    def __repr__(self) -> str:
        c = self.c
        return (f"SchedParams(n_steps={c.n_steps}, L={c.L}, g_slope={c.g_slope}, k={c.k}, "
                f"tau_cap={c.tau_cap}, defer={bool(c.flags & SCHED_DEFER)})")


def _sp(sched: Optional[SchedParams]):
    return None if sched is None else ctypes.byref(sched.c)


def workspace_bytes(n: int, dtype_code: int) -> int:
    return int(lib.cfg_workspace_bytes(n, dtype_code))


def new_workspace(n: int = 0, dtype_code: int = CFG_BF16, device=None, batch: int = 1):
    """A zero-filled (hence prepared) device workspace for calls over n elements
    (``batch`` consecutive workspaces for the batched calls)."""
    torch = _torch()
    nb = workspace_bytes(n, dtype_code)
    if nb == 0:
        raise ValueError("invalid n / dtype for a workspace")
    return torch.zeros(nb * batch, dtype=torch.uint8, device=device or "cuda")


def new_sched_state(device=None, batch: int = 1):
    """Device memory for ``batch`` cfg_sched_state structs (contents are reset by step 0)."""
    torch = _torch()
    return torch.zeros(ctypes.sizeof(SchedStateC) * batch, dtype=torch.uint8,
                       device=device or "cuda")


def workspace_flush(workspace, stream=None, batch: int = 1) -> None:
    """Complete the work deferring steps left in the workspace (``batch`` regions)."""
    ws, wsb = _ws(workspace)
    _check(lib.cfg_workspace_flush_batched(ws, wsb, batch, _stream(stream)))


def read_sched_state(state, index: int = 0) -> Dict[str, object]:
    """Copy schedule state ``index`` of a device state array to the host (synchronises)."""
    size = ctypes.sizeof(SchedStateC)
    host = state.detach().view(-1)[index * size:(index + 1) * size].to("cpu").numpy().tobytes()
    s = SchedStateC.from_buffer_copy(host)
    n = max(0, min(s.n_seen, SCHED_MAX_STEPS))
    return {
        "n_seen": s.n_seen, "tau1p": s.tau1p, "argmin": s.argmin, "tau_cap": s.tau_cap,
        "tau1": s.tau1, "tau2": s.tau2, "decided_at": s.decided_at, "flags": s.flags,
        "min_M": s.min_M,
        "M": np.array(s.M[:n], dtype=np.float64),
        "G": np.array(s.G[:n], dtype=np.float64),
        "phase": np.array(s.phase[:n], dtype=np.uint8),
    }


def _ws(workspace):
    return _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------
def _per_sample(t, batch: int) -> int:
    if batch < 1 or t.numel() % batch:
        raise ValueError(f"{t.numel()} elements do not split into {batch} samples")
    return t.numel() // batch


def relmae_reduce(pred_c, pred_u, *, workspace, M_out=None, state=None, sched=None, step: int = 0,
                  stream=None, batch: int = 1) -> None:
    """rel-MAE of (pred_c, pred_u) into M_out (float64 device scalar, or ``batch`` of them,
    one per sample) and/or the schedule state(s)."""
    if pred_c.shape != pred_u.shape or pred_c.dtype != pred_u.dtype:
        raise ValueError("pred_c and pred_u must match in shape and dtype")
    ws, wsb = _ws(workspace)
    _check(lib.cfg_relmae_reduce_batched(
        _dev_ptr(pred_c, "pred_c"), _dev_ptr(pred_u, "pred_u"), _per_sample(pred_c, batch),
        batch, _dtype_code(pred_c), _dev_ptr(M_out, "M_out"), _dev_ptr(state, "state"),
        _sp(sched), step, ws, wsb, _stream(stream)))


def _same(x_out, x_in, pc, pu) -> None:
    for t in (x_in, pc, pu):
        if t.shape != x_out.shape or t.dtype != x_out.dtype:
            raise ValueError("x_out, x_in, pred_c, pred_u must share shape and dtype")


def ddim_step(x_out, x_in, pred_c, pred_u, *, w: float, abar_t: float, abar_prev: float,
              workspace, eta: float = 0.0, seed: int = 0, step: int = 0, M_out=None, state=None,
              sched=None, stream=None, batch: int = 1, exact_rounding: bool = False) -> None:
    """One fused CFG + DDIM step (see cfg_ddim_step; batch > 1: cfg_ddim_step_batched).
    ``exact_rounding``: bf16 results correctly rounded (CFG_BF16_EXACT)."""
    _same(x_out, x_in, pred_c, pred_u)
    ws, wsb = _ws(workspace)
    _check(lib.cfg_ddim_step_batched(
        _dev_ptr(x_out, "x_out"), _dev_ptr(x_in, "x_in"), _dev_ptr(pred_c, "pred_c"),
        _dev_ptr(pred_u, "pred_u"), _per_sample(x_out, batch), batch,
        _dtype_code(x_out, exact_rounding), w, abar_t, abar_prev, eta, seed, step, _dev_ptr(M_out, "M_out"), _dev_ptr(state, "state"),
        _sp(sched), ws, wsb, _stream(stream)))


def ddim_step_static_ws(x_out, x_in, pred_c, pred_u, *, w: float, abar_t: float,
                        abar_prev: float, eta: float = 0.0, seed: int = 0, step: int = 0,
                        M_out=None, state=None, sched=None, stream=None,
                        exact_rounding: bool = False) -> None:
    """ddim_step on the library's static device scratch (no workspace argument), for callers
    that cannot allocate device memory; calls on one device share that scratch."""
    _same(x_out, x_in, pred_c, pred_u)
    _check(lib.cfg_ddim_step_static_ws(
        _dev_ptr(x_out, "x_out"), _dev_ptr(x_in, "x_in"), _dev_ptr(pred_c, "pred_c"),
        _dev_ptr(pred_u, "pred_u"), x_out.numel(), _dtype_code(x_out, exact_rounding), w, abar_t,
        abar_prev, eta,
        seed, step, _dev_ptr(M_out, "M_out"), _dev_ptr(state, "state"), _sp(sched),
        _stream(stream)))


def flow_step(x_out, x_in, v_c, v_u, *, w: float, t_cur: float, t_next: float, workspace,
              step: int = 0, M_out=None, state=None, sched=None, stream=None,
              batch: int = 1, exact_rounding: bool = False) -> None:
    """One fused CFG + Euler flow step (see cfg_flow_step; batch > 1: cfg_flow_step_batched).
    ``exact_rounding``: bf16 results correctly rounded (CFG_BF16_EXACT)."""
    _same(x_out, x_in, v_c, v_u)
    ws, wsb = _ws(workspace)
    _check(lib.cfg_flow_step_batched(
        _dev_ptr(x_out, "x_out"), _dev_ptr(x_in, "x_in"), _dev_ptr(v_c, "v_c"),
        _dev_ptr(v_u, "v_u"), _per_sample(x_out, batch), batch,
        _dtype_code(x_out, exact_rounding), w, t_cur,
        t_next, step, _dev_ptr(M_out, "M_out"), _dev_ptr(state, "state"), _sp(sched), ws, wsb,
        _stream(stream)))


def sched_observe(state, sched: SchedParams, step: int, M: float, stream=None) -> None:
    """Record an externally computed rel-MAE value as step ``step`` of the schedule."""
    _check(lib.cfg_sched_observe(_dev_ptr(state, "state"), _sp(sched), step, M, _stream(stream)))


class _HostBlock:
    """Page-locked host memory from cfg_host_alloc, freed when the last tensor using it goes."""

    def __init__(self, nbytes: int):
        ptr = c_void_p()
        _check(lib.cfg_host_alloc(nbytes, ctypes.byref(ptr)))
        self.ptr, self.nbytes = ptr.value, nbytes

    def __del__(self):
        if getattr(self, "ptr", None) and lib is not None:
            lib.cfg_host_free(self.ptr)
            self.ptr = None


def pinned_empty(numel: int, dtype) -> "torch.Tensor":
    """A CPU tensor of `numel` elements on page-locked memory from cfg_host_alloc.

    Copies from/to it with :func:`copy_async` run asynchronously in stream order.  (torch's
    ``is_pinned()`` reports only its own pool, so it says False here, and ``Tensor.copy_``
    treats the memory as pageable; the CUDA driver knows it is page-locked.)
    """
    torch = _torch()
    itemsize = torch.empty((), dtype=dtype).element_size()
    nbytes = max(int(numel) * itemsize, 1)
    block = _HostBlock(nbytes)
    raw = (ctypes.c_char * nbytes).from_address(block.ptr)
    raw._owner = block                      # the buffer keeps the allocation alive
    t = torch.frombuffer(raw, dtype=torch.uint8)
    return t[: int(numel) * itemsize].view(dtype)


def copy_async(dst, src, *, stream=None) -> None:
    """Copy tensor `src` into `dst` (same number of bytes, both contiguous; host or device) with
    the library's cfg_copy_async on `stream` (default: the current stream).

    Unlike ``Tensor.copy_``, which treats host memory outside torch's own pool as pageable, this
    stays asynchronous for buffers from :func:`pinned_empty`.
    """
    for t, name in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(lib.cfg_copy_async(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)))


def randn(out, *, seed: int, step: int = 0, stream_id: int = 0, stream=None) -> None:
    """Fill a float32 device tensor with the library's Philox/Box-Muller N(0,1) stream."""
    torch = _torch()
    if out.dtype != torch.float32:
        raise TypeError("randn writes float32")
    _check(lib.cfg_randn(_dev_ptr(out, "out"), out.numel(), seed, step, stream_id, _stream(stream)))


def abar_linear(T: int = 1000, beta_start: float = 1e-4, beta_end: float = 0.02) -> np.ndarray:
    """Host table abar[t] of the linear-beta schedule (computed by the library)."""
    out = np.empty(T, dtype=np.float64)
    _check(lib.cfg_abar_linear(out.ctypes.data_as(POINTER(c_double)), T, beta_start, beta_end))
    return out


def ddim_timesteps(n_steps: int, T: int = 1000) -> np.ndarray:
    """DDIM timestep sequence, noisiest first (computed by the library)."""
    out = np.empty(n_steps, dtype=np.int32)
    _check(lib.cfg_ddim_timesteps(out.ctypes.data_as(POINTER(c_int32)), n_steps, T))
    return out


SPACING = {"linspace": 0, "leading": 1, "trailing": 2}


def abar_cosine(T: int = 1000, s: float = 0.008, max_beta: float = 0.999) -> np.ndarray:
    """Host table abar[t] of the cosine schedule (computed by the library)."""
    out = np.empty(T, dtype=np.float64)
    _check(lib.cfg_abar_cosine(out.ctypes.data_as(POINTER(c_double)), T, s, max_beta))
    return out


def timesteps(n_steps: int, T: int = 1000, spacing: str = "linspace") -> np.ndarray:
    """Timestep sequence, noisiest first, with the given spacing (computed by the library)."""
    out = np.empty(n_steps, dtype=np.int32)
    _check(lib.cfg_timesteps(out.ctypes.data_as(POINTER(c_int32)), n_steps, T, SPACING[spacing]))
    return out


def sampler_run(x, *, mode: int, n_steps: int, w: float, denoise: Callable, pred_c, pred_u,
                sched: SchedParams, state, workspace, abar_table: Optional[np.ndarray] = None,
                timesteps: Optional[np.ndarray] = None, t_grid: Optional[np.ndarray] = None,
                eta: float = 0.0, seed: int = 0, start_step: int = 0, stream=None,
                exact_rounding: bool = False) -> None:
    """Run a whole CFG sampler in the library's host loop (see cfg_sampler_run).

    ``denoise(step, timestep, t)`` must enqueue the two predictions for the
    current ``x`` into ``pred_c`` / ``pred_u`` on the current stream.  An
    exception raised by it stops the run and is re-raised here.
    """
    _same(x, x, pred_c, pred_u)
    err = []

    def _cb(user, step, timestep, t, x_t, out_c, out_u, strm):
        try:
            denoise(int(step), int(timestep), float(t))
            return 0
        except BaseException as e:  # noqa: BLE001 - re-raised after the C loop returns
            err.append(e)
            return 1

    cb = DENOISE_FN(_cb)
    ab = None
    ts = None
    tg = None
    if abar_table is not None:
        abar_table = np.ascontiguousarray(abar_table, dtype=np.float64)
        ab = abar_table.ctypes.data_as(POINTER(c_double))
    if timesteps is not None:
        timesteps = np.ascontiguousarray(timesteps, dtype=np.int32)
        ts = timesteps.ctypes.data_as(POINTER(c_int32))
    if t_grid is not None:
        t_grid = np.ascontiguousarray(t_grid, dtype=np.float64)
        tg = t_grid.ctypes.data_as(POINTER(c_double))
    ws, wsb = _ws(workspace)
    status = lib.cfg_sampler_run(
        _dev_ptr(x, "x"), x.numel(), _dtype_code(x, exact_rounding), mode, ab,
        0 if abar_table is None else int(abar_table.shape[0]), ts, tg, n_steps, w, eta, seed, cb,
        None, _dev_ptr(pred_c, "pred_c"), _dev_ptr(pred_u, "pred_u"), _sp(sched),
        _dev_ptr(state, "state"), start_step, ws, wsb, _stream(stream))
    if err:
        raise err[0]
    _check(status)


def sampler_run_branches(x, *, mode: int, n_steps: int, w: float, denoise_branch: Callable,
                         pred_c, pred_u, stream_c, stream_u, sched: SchedParams, state,
                         workspace, abar_table: Optional[np.ndarray] = None,
                         timesteps: Optional[np.ndarray] = None,
                         t_grid: Optional[np.ndarray] = None, eta: float = 0.0, seed: int = 0,
                         start_step: int = 0, stream=None, exact_rounding: bool = False) -> None:
    """A whole CFG sampler run with the two branches on two streams (see
    cfg_sampler_run_branches).

    ``denoise_branch(branch, step, timestep, t)`` must enqueue branch 0 (conditional, into
    ``pred_c``) or 1 (unconditional, into ``pred_u``); it is called with that branch's stream
    (``stream_c`` / ``stream_u``) as torch's current stream.
    """
    torch = _torch()
    _same(x, x, pred_c, pred_u)
    err = []
    streams = {0: stream_c, 1: stream_u}

    def _cb(user, branch, step, timestep, t, x_t, out, strm):
        try:
            with torch.cuda.stream(streams[int(branch)]):
                denoise_branch(int(branch), int(step), int(timestep), float(t))
            return 0
        except BaseException as e:  # noqa: BLE001 - re-raised after the C loop returns
            err.append(e)
            return 1

    cb = BRANCH_FN(_cb)
    ab = ts = tg = None
    if abar_table is not None:
        abar_table = np.ascontiguousarray(abar_table, dtype=np.float64)
        ab = abar_table.ctypes.data_as(POINTER(c_double))
    if timesteps is not None:
        timesteps = np.ascontiguousarray(timesteps, dtype=np.int32)
        ts = timesteps.ctypes.data_as(POINTER(c_int32))
    if t_grid is not None:
        t_grid = np.ascontiguousarray(t_grid, dtype=np.float64)
        tg = t_grid.ctypes.data_as(POINTER(c_double))
    ws, wsb = _ws(workspace)
    status = lib.cfg_sampler_run_branches(
        _dev_ptr(x, "x"), x.numel(), _dtype_code(x, exact_rounding), mode, ab,
        0 if abar_table is None else int(abar_table.shape[0]), ts, tg, n_steps, w, eta, seed, cb,
        None, _dev_ptr(pred_c, "pred_c"), _dev_ptr(pred_u, "pred_u"), _stream(stream_c),
        _stream(stream_u), _sp(sched), _dev_ptr(state, "state"), start_step, ws, wsb,
        _stream(stream))
    if err:
        raise err[0]
    _check(status)
