import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large full-size workload")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints every error a parity check measured, with the bound it was held
    to (tests record them through parity_util.record)."""
    mod = sys.modules.get("parity_util")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", f"measured errors ({len(recs)} checks): measured / bound")
    worst = max(recs, key=lambda r: r[2] / r[3] if r[3] > 0 else 0.0)
    for name, qty, got, bound in recs:
        ratio = got / bound if bound > 0 else float("nan")
        tr.write_line(f"{got:10.3e} / {bound:8.1e} ({ratio:5.2f})  {qty:28s} {name}")
    tr.write_line(f"closest to its bound: {worst[1]} of {worst[0]}: {worst[2]:.3e} / {worst[3]:.1e}")
