import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def _lib_is_stale() -> bool:
    from packed_sequence_context_gb300 import build, thd_attn
    if not os.path.exists(thd_attn.LIB_PATH):
        return True
    t = os.path.getmtime(thd_attn.LIB_PATH)
    deps = build.sources() + [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(ROOT, "include", "thd_attn.h"))
    return any(os.path.getmtime(d) > t for d in deps)


@pytest.fixture(scope="session")
def thd_lib():
    """The built library (built in-tree first if missing or older than its sources)."""
    from packed_sequence_context_gb300 import build, thd_attn
    if _lib_is_stale():
        build.build()
    return thd_attn.lib()
