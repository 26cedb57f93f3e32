import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


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


def pytest_terminal_summary(terminalreporter):
    """Print how far the bf16 attention rows of each parity test went past
    the flat 2e-2 tolerance (within their rounding allowances); with
    FUSEKV_PARITY_LOG set, also write the records there as JSON lines."""
    try:
        import rounding
    except Exception:  # pragma: no cover
        return
    if not rounding.RECORDS:
        return
    tr = terminalreporter
    tr.section("bf16 attention rows past the flat tolerance")
    for r in rounding.RECORDS:
        tr.write_line(f"{r['test']}: {r['over_flat']}/{r['pairs']} (row, head) pairs over 2e-2 "
                      f"(max {r['max_err_over_flat']:.3g}x), {r['widened']} widened, "
                      f"{r['widened_over_2x']} beyond 2x, {r['rows']} rows")
    path = os.environ.get("FUSEKV_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            for r in rounding.RECORDS:
                f.write(json.dumps(r) + "\n")
