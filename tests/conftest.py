import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the worst parity margin of every GPU parity test (the largest
    |gpu - oracle| / (atol + rtol |oracle|) it saw; 1.0 is the tolerance)."""
    mod = sys.modules.get("gpu_util")
    margins = getattr(mod, "MARGINS", None) if mod else None
    if not margins:
        return
    tr = terminalreporter
    tr.section("parity margins (worst err / (atol + rtol*|ref|) per test)")
    for test, (ratio, what) in sorted(margins.items(), key=lambda kv: -kv[1][0]):
        tr.write_line(f"{ratio:7.3f}  {test}  [{what}]")
    path = os.environ.get("PA_PARITY_MARGINS")
    if path:
        import json

        with open(path, "w") as f:
            json.dump({t: {"ratio": r, "case": w} for t, (r, w) in margins.items()}, f, indent=1, sort_keys=True)
