import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblce.so")
    config.addinivalue_line("markers", "slow: large workload, minutes of CPU oracle time")


def pytest_sessionstart(session):
    # LCE_TEST_GEMM_FORM=single|pair runs the whole suite with that GEMM form
    # instead of the library's default.
    form = os.environ.get("LCE_TEST_GEMM_FORM")
    if form:
        import lm_head_linear_chunked_gb300 as lce
        lce.lce_set_gemm_form(form)


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, where no GPU is present; the CPU
    # suite deselects them with -m "not gpu" anyway.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("LCE_PARITY_REPORT")
    if not path:
        return
    try:
        from tests import gpu_util
    except Exception:
        return
    import json
    with open(path, "w") as f:
        json.dump(gpu_util.RECORDS, f, indent=0)
