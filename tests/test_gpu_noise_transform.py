"""Exhaustive accuracy of the step's Gaussian transforms (needs a GPU and nvcc).

The noise uniforms are u = j / 2^24 with j odd in (0, 2^24): 2^23 values.  The
check program (``noise_transform_check.cu``) evaluates every factor of the
Box-Muller pair -- rho = sqrt(-2 ln u) and sin, cos of 2 pi u -- for all of
them, in both accuracies of ``csrc/cfg_noise.cuh``, against fp64.  From the
factor bounds, with |rho| <= sqrt(48 ln 2) < 5.78 and the final fp32 product
rounded (half an ulp of a value below 8: 2^-22), each normal's error is at
most |d rho| + 5.78 max(|d sin|, |d cos|) + 2^-22 (a cross term below 1e-12
aside):

* bf16-storage transform (the bf16 step's noise): at most 3.2e-6 absolute,
  the bound ``include/cfgstep.h`` states;
* full-accuracy transform (fp32 steps, cfg_randn): rho within 2 fp32 ulps,
  sin and cos within 2 ulps of their exact values.

The zyxy.net DDIM sampler (section 3) adds sigma_eta times standard normal
noise; the oracle draws it in fp64 from the same Philox words.
"""
import json
import math
import subprocess
from pathlib import Path

import pytest

from cfg_guided_sampler_step_b300 import _build

pytestmark = pytest.mark.gpu

CSRC = _build.PKG_DIR / "csrc"
CHECK = Path(__file__).with_name("noise_transform_check.cu")
RHO_MAX = math.sqrt(48.0 * math.log(2.0))


@pytest.fixture(scope="module")
def errors(tmp_path_factory, cuda):
    exe = tmp_path_factory.mktemp("noise") / "noise_transform_check"
    cmd = [_build.nvcc_path(), *_build.ARCH_FLAGS, "-O3", "-std=c++17", "-I", str(CSRC),
           "-o", str(exe), str(CHECK)]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-4000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr[-2000:]
    print("noise transform errors:", run.stdout.strip())
    return json.loads(run.stdout)


def test_bf16_transform_is_within_its_stated_bound(errors):
    e = errors["bf16"]
    assert e["rho_abs"] < 7.3e-7, e
    assert e["sin_abs"] < 3.5e-7 and e["cos_abs"] < 3.5e-7, e
    bound = e["rho_abs"] + RHO_MAX * max(e["sin_abs"], e["cos_abs"]) + 2.0**-22
    assert bound < 3.2e-6, (bound, e)


def test_full_accuracy_transform_is_within_two_ulps(errors):
    e = errors["full"]
    assert e["rho_ulp"] <= 2.0 and e["sin_ulp"] <= 2.0 and e["cos_ulp"] <= 2.0, e
    # and far tighter than the bf16 transform in absolute terms
    assert e["rho_abs"] < 1e-6 and e["sin_abs"] < 1.2e-7 and e["cos_abs"] < 1.2e-7, e
