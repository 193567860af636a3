import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


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


def pytest_sessionfinish(session, exitstatus):
    """With SINKATTN_PARITY_REPORT=<path>, write every oracle comparison the
    session made (per test: elements, max error, |ref| >= 4 count, elements
    passed by the one-ulp rule) to <path> as JSON."""
    path = os.environ.get("SINKATTN_PARITY_REPORT")
    if not path:
        return
    import json
    try:
        import tolerances
    except ImportError:
        return
    with open(path, "w") as f:
        json.dump(tolerances.RECORD, f, indent=1, sort_keys=True)
