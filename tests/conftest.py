import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import importlib.util

import pytest


def _load_build_module():
    path = os.path.join(ROOT, "attention_ifa_fia_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("fia_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="session")
def built_lib():
    """Path of libfia_gb300.so, (re)built for sm_103a if missing or stale."""
    return _load_build_module().build()


@pytest.fixture(scope="session")
def F(built_lib):
    """The package binding (loads the built library)."""
    import attention_ifa_fia_gb300 as pkg
    return pkg


@pytest.fixture(scope="session")
def cuda(F):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Lists the softmax maxima that met their bound only through the near-zero absolute
    term (tests/parity.py); FIA_NEAR_ZERO_REPORT=<path> also writes them there as JSON."""
    try:
        from parity import NEAR_ZERO_MAX_ROWS
    except ImportError:
        return
    if not NEAR_ZERO_MAX_ROWS:
        return
    terminalreporter.write_line(f"softmax maxima accepted by the near-zero absolute term: {len(NEAR_ZERO_MAX_ROWS)}")
    for test, name, idx, mag, err in NEAR_ZERO_MAX_ROWS[:50]:
        terminalreporter.write_line(f"  {test} {name}[{idx}]: |max| {mag:.3g}, abs err {err:.3g}")
    path = os.environ.get("FIA_NEAR_ZERO_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([dict(test=t, quantity=n, index=i, abs_max=m, abs_err=e) for t, n, i, m, e in NEAR_ZERO_MAX_ROWS],
                      f, indent=1)
