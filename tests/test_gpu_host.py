"""Page-locked host buffers of the C ABI (cfg_host_alloc / cfg_host_free) (needs a GPU)."""
import ctypes
import gc

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
    # page-locked as far as the driver is concerned (torch's is_pinned only knows its own pool)
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
