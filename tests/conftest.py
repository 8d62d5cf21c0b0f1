"""Test configuration: the `gpu` marker and the import path of the repository root."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def built_libraries():
    """Build whatever library is missing (the oracle, the generator, the CUDA library)."""
    import importlib.util

    import oracle
    import synth

    if not os.path.exists(oracle._SO):
        oracle.build()
    if not (os.path.exists(synth._HOST_SO) and os.path.exists(synth._DEV_SO)):
        synth.build()
    lib = os.path.join(ROOT, "fsdp_sharded_mixed_ss_gb300", "libss.so")
    if not os.path.exists(lib):
        spec = importlib.util.spec_from_file_location("ss_build", os.path.join(ROOT, "fsdp_sharded_mixed_ss_gb300", "_build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    yield

