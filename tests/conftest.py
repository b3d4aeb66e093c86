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


_PARITY_ROWS = {}


@pytest.fixture(scope="session")
def parity_report():
    """Collects per-case parity figures (errors, margins) measured by the GPU tests; when the
    environment names a file in CFG_PARITY_REPORT, they are written there as JSON at the end
    of the session (the figures quoted in the design notes come from such a file)."""
    return _PARITY_ROWS


def pytest_sessionfinish(session, exitstatus):
    import json
    import os
    path = os.environ.get("CFG_PARITY_REPORT")
    if path and _PARITY_ROWS:
        Path(path).parent.mkdir(parents=True, exist_ok=True)
        Path(path).write_text(json.dumps(_PARITY_ROWS, indent=1, sort_keys=True, default=float))
