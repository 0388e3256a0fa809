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
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Worst error per test: raw max-abs, max-abs beyond bf16 output rounding
    (what the max-abs bound applies to) and mean-abs, each over its bound."""
    try:
        from tolerance import NOTES, RESULTS
    except ImportError:  # pragma: no cover
        return
    if not RESULTS and not NOTES:
        return
    worst = {}
    for name, raw, excess, mean, tol_max, tol_mean in RESULTS:
        test = name.rsplit("::", 1)[0]
        w = worst.setdefault(test, [0.0, 0.0, 0.0, 0.0, 0.0, 0])
        w[0] = max(w[0], raw)
        w[1] = max(w[1], excess)
        w[2] = max(w[2], mean)
        w[3] = max(w[3], excess / tol_max)
        w[4] = max(w[4], mean / tol_mean)
        w[5] += 1
    tr = terminalreporter
    for msg in NOTES:
        tr.write_line(msg)
    tr.write_sep("-", "parity errors (worst per test: raw max-abs | beyond bf16 rounding | mean-abs)")
    for test, (raw, excess, mean, fmax, fmean, n) in worst.items():
        tr.write_line(f"{test}: {n} checks, max-abs {raw:.3e} | {excess:.3e} ({fmax:.0%} of bound) | "
                      f"mean {mean:.3e} ({fmean:.0%} of bound)")
