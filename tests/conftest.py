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
