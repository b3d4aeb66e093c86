"""Shared pytest setup: the ``gpu`` marker, import paths and the in-tree library build."""
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running parity case")


def _ensure_built():
    # loaded by path: importing the package needs the built library
    import importlib.util
    path = ROOT / "cfg_guided_sampler_step_b300" / "_build.py"
    spec = importlib.util.spec_from_file_location("cfg_guided_sampler_step_b300_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


# Build before any test module imports the binding (which raises when the
# library is missing).
_ensure_built()


def cuda_available() -> bool:
    import torch
    return torch.cuda.is_available()


@pytest.fixture(scope="session")
def cuda():
    if not cuda_available():
        pytest.skip("no CUDA device")
    import torch
    return torch.device("cuda:0")
