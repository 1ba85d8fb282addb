import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


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


def record_errors(name, reports):
    """Print the error measures of a parity comparison ({quantity: oracle.error_report})
    and, when SSM_PARITY_REPORT names a file, append them to it as one JSON line."""
    import json
    line = {"case": name, **{k: {m: float(f"{v:.4g}") for m, v in r.items()} for k, r in reports.items()}}
    print(json.dumps(line))
    path = os.environ.get("SSM_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")


@pytest.fixture(autouse=True)
def _bounds_checked_status(request):
    """Under SSM_EXPECT_BOUNDS_CHECK=1 (the bounds-checked library loaded through
    SSM_LIB_PATH), every GPU test must leave the device status clean: no store of any
    kernel it ran fell outside its buffer."""
    yield
    if os.environ.get("SSM_EXPECT_BOUNDS_CHECK") != "1" or "gpu" not in request.keywords:
        return
    import selective_state_space_143_b300 as ssm
    from selective_state_space_143_b300 import _lib
    assert ssm.bounds_check_enabled(), "SSM_EXPECT_BOUNDS_CHECK set but the library has no checks"
    import torch
    torch.cuda.synchronize()
    assert ssm.device_status(clear=True) == _lib.SSM_OK, "a bounds check fired"
