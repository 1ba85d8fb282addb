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
