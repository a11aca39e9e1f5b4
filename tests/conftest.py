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
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per test and in total: decisions compared with the oracle and how many
    of them the oracle flagged as too close to call (the parity rule's count)."""
    mod = sys.modules.get("parity")
    rows = getattr(mod, "SESSION", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "oracle parity: compared / flagged decisions")
    tot = {}
    for name, kind, compared, flagged in rows:
        tr.write_line(f"{kind:6s} {compared:8d} {flagged:4d}  {name}")
        c, f = tot.get(kind, (0, 0))
        tot[kind] = (c + compared, f + flagged)
    for kind, (c, f) in sorted(tot.items()):
        rate = f / c if c else 0.0
        tr.write_line(f"{kind:6s} total: {c} compared, {f} flagged (rate {rate:.2e})")
