"""The C ABI from a plain C program (needs a GPU, gcc and the CUDA runtime).

`c_abi_consumer.c` includes only ``include/cfgstep.h`` and the CUDA runtime header, links
``libcfgstep.so`` and ``libcudart``, and runs one fp32 DDIM step and one rel-MAE reduction on
device buffers of its own. Its outputs are held to the oracle's step (zyxy.net DDIM sampler,
section 3) and rel-MAE (Hybridiff notes, key design 2) at the fp32 tolerances of the step
tests: every element within 1 ulp (or 1e-9 after cancellation), M within 1e-6.
"""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

import workloads as W
from cfg_guided_sampler_step_b300 import _build
from gpu_harness import ulp_distance_f32
from oracle import cfg_oracle as O

pytestmark = pytest.mark.gpu

SRC = Path(__file__).with_name("c_abi_consumer.c")


def _cuda_root() -> Path:
    return Path(_build.nvcc_path()).resolve().parent.parent


@pytest.fixture(scope="module")
def consumer(tmp_path_factory, cuda):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    exe = tmp_path_factory.mktemp("c_consumer") / "c_abi_consumer"
    cuda_root = _cuda_root()
    lib_dir = _build.LIB.parent
    cmd = ["gcc", "-std=c99", "-O2", "-I", str(_build.HEADER.parent),
           "-I", str(cuda_root / "include"), "-o", str(exe), str(SRC),
           "-L", str(lib_dir), "-lcfgstep", f"-Wl,-rpath,{lib_dir}",
           "-L", str(cuda_root / "lib64"), "-lcudart", f"-Wl,-rpath,{cuda_root / 'lib64'}"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-4000:]
    return exe


@pytest.mark.parametrize("n", [1, 4097, 3 * 65536 + 5])
def test_c_program_step_and_reduction_match_the_oracle(consumer, tmp_path, n):
    d = W.draw_prediction_pair(n, "f32", 41 + n % 7)
    abar = O.abar_linear()
    w, ab, abp = 7.5, float(abar[600]), float(abar[580])
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        np.array([n], dtype=np.int64).tofile(f)
        np.array([w, ab, abp], dtype=np.float64).tofile(f)
        for k in ("x", "c", "u"):
            np.asarray(d[k], dtype=np.float32).tofile(f)
    run = subprocess.run([str(consumer), str(inp), str(outp)], capture_output=True, text=True,
                         timeout=120)
    assert run.returncode == 0, run.stderr[-2000:]
    assert "sm_103a" in run.stdout
    raw = outp.read_bytes()
    got = np.frombuffer(raw[: 4 * n], dtype=np.float32).astype(np.float64)
    M_step, M_red = np.frombuffer(raw[4 * n:], dtype=np.float64)
    x64, c64, u64 = (W.stored_to_f64(d[k], "f32") for k in ("x", "c", "u"))
    ref, refM = O.ddim_step(x64, c64, u64, "f32", w, ab, abp, 0.0, 0, 0)
    diff = np.abs(got - ref)
    assert float(diff.max()) <= 1e-5
    ok = (ulp_distance_f32(got, ref) <= 1) | (diff <= 1e-9)
    assert ok.all(), np.flatnonzero(~ok)[:10]
    M_ref = O.rel_mae(c64, u64)
    for M in (M_step, M_red):
        assert abs(M - M_ref) <= 1e-6 * abs(M_ref), (M, M_ref)
