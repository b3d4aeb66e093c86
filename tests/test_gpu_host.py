"""Host-side parts of the C ABI on a GPU: page-locked host buffers (cfg_host_alloc /
cfg_host_free, cfg_copy_async) and first calls on a device made from several host threads at
once (needs a GPU)."""
import ctypes
import gc
import os
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest
import torch

import cfg_guided_sampler_step_b300 as cs

pytestmark = pytest.mark.gpu


def test_host_alloc_rejects_bad_arguments(cuda):
    ptr = ctypes.c_void_p(1)
    assert cs.STATUS_NAMES[cs.lib.cfg_host_alloc(0, ctypes.byref(ptr))] == "CFG_ERR_INVALID_ARG"
    assert ptr.value is None
    assert cs.lib.cfg_host_free(None) == 0


def test_pinned_empty_is_page_locked_and_round_trips(cuda):
    n = 3 * (1 << 20) + 5
    h = cs.pinned_empty(n, torch.bfloat16)
    assert h.device.type == "cpu" and h.dtype == torch.bfloat16 and h.numel() == n
    # page-locked as far as the CUDA driver is concerned (torch's is_pinned only knows its own pool)
    from cuda.bindings import runtime as cudart
    err, attr = cudart.cudaPointerGetAttributes(h.data_ptr())
    assert err == cudart.cudaError_t.cudaSuccess
    assert attr.type == cudart.cudaMemoryType.cudaMemoryTypeHost
    src = torch.randn(n).to(torch.bfloat16)
    h.copy_(src)
    d = torch.empty(n, dtype=torch.bfloat16, device=cuda)
    s = torch.cuda.Stream(cuda)
    back = cs.pinned_empty(n, torch.bfloat16)
    with torch.cuda.stream(s):
        d.copy_(h, non_blocking=True)
        d.mul_(2)
        back.copy_(d, non_blocking=True)
    s.synchronize()
    assert torch.equal(back, src * 2)


def test_pinned_empty_lifetime_follows_views(cuda):
    h = cs.pinned_empty(1000, torch.float32)
    v = h[10:20]
    h.fill_(3.0)
    del h
    gc.collect()
    assert np.all(v.numpy() == 3.0)          # the allocation lives while a view does
    d = torch.empty(10, device=cuda)
    d.copy_(v, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.all(d == 3.0)


def test_copy_async_round_trip_and_checks(cuda):
    n = (1 << 20) + 3
    h = cs.pinned_empty(n, torch.float32)
    h.copy_(torch.arange(n, dtype=torch.float32))
    d = torch.empty(n, dtype=torch.float32, device=cuda)
    back = cs.pinned_empty(n, torch.float32)
    s = torch.cuda.Stream(cuda)
    with torch.cuda.stream(s):
        cs.copy_async(d, h)                  # host -> device
        d.add_(1)
        cs.copy_async(back, d)               # device -> host
    s.synchronize()
    assert torch.equal(back, torch.arange(n, dtype=torch.float32) + 1)
    d2 = torch.empty_like(d)
    cs.copy_async(d2, d)                     # device -> device
    torch.cuda.synchronize()
    assert torch.equal(d2, d)
    with pytest.raises(ValueError):
        cs.copy_async(d[:10], h[:11])
    assert cs.lib.cfg_copy_async(None, None, 0, None) == 0            # zero bytes: a no-op
    assert cs.STATUS_NAMES[cs.lib.cfg_copy_async(None, h.data_ptr(), 4, None)] == "CFG_ERR_INVALID_ARG"


_FIRST_CALLS = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import cfg_guided_sampler_step_b300 as cs
import workloads as W
from gpu_harness import to_device_stored

dev = torch.device("cuda:0")
torch.cuda.init()
T = 8
n = 200_003
shared = torch.cuda.Stream(dev)
jobs = []
for i in range(T):
    d = W.draw_prediction_pair(n, "bf16", 700 + i)
    x, c, u = (to_device_stored(d[k], "bf16", dev) for k in ("x", "c", "u"))
    jobs.append(dict(x=x, c=c, u=u, ws_out=torch.empty_like(x), st_out=torch.empty_like(x),
                     ws=cs.new_workspace(n, cs.CFG_BF16, dev), own=torch.cuda.Stream(dev)))
torch.cuda.synchronize()
go = threading.Barrier(T)
errors = []

def worker(j):
    try:
        torch.cuda.set_device(dev)
        go.wait()
        # first calls on this device in this process: the per-device lookups race here
        cs.ddim_step(j["ws_out"], j["x"], j["c"], j["u"], w=5.0, abar_t=0.3, abar_prev=0.4,
                     eta=1.0, seed=3, step=2, workspace=j["ws"], stream=j["own"])
        # static scratch calls all go to one stream, so they never overlap on the GPU
        cs.ddim_step_static_ws(j["st_out"], j["x"], j["c"], j["u"], w=5.0, abar_t=0.3,
                               abar_prev=0.4, eta=1.0, seed=3, step=2, stream=shared)
    except Exception as e:  # noqa: BLE001
        errors.append(repr(e))

threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
for t in threads: t.start()
for t in threads: t.join(120)
torch.cuda.synchronize()
assert not errors, errors
for j in jobs:
    ref = torch.empty_like(j["x"])
    cs.ddim_step(ref, j["x"], j["c"], j["u"], w=5.0, abar_t=0.3, abar_prev=0.4, eta=1.0, seed=3,
                 step=2, workspace=cs.new_workspace(n, cs.CFG_BF16, dev))
    torch.cuda.synchronize()
    assert torch.equal(ref, j["ws_out"]) and torch.equal(ref, j["st_out"])
print("first calls ok")
"""


def test_first_calls_from_many_threads(cuda, tmp_path):
    """A fresh process (so every per-device lookup starts empty) in which eight host threads
    make their first step calls at the same moment: with their own workspaces and streams,
    and through the static scratch on one shared stream.  Every result equals a later
    single-threaded call bit for bit."""
    root = Path(__file__).resolve().parent.parent
    script = tmp_path / "first_calls.py"
    script.write_text(_FIRST_CALLS)
    env = dict(os.environ, PYTHONPATH=f"{root}:{root / 'tests'}")
    out = subprocess.run([sys.executable, str(script), str(root)], capture_output=True, text=True,
                         timeout=300, env=env)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "first calls ok" in out.stdout
