import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size case, takes tens of seconds")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped cleanly when no GPU is present; the CPU suite is
    # selected with -m "not gpu".
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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # How often the output checks used the one-ulp slack of the tolerance.
    lib = sys.modules.get("flint_testlib")
    if lib is None or lib.SLACK_TOTALS["checks"] == 0:
        return
    t = lib.SLACK_TOTALS
    terminalreporter.write_line(
        f"output checks: {t['checks']}, elements {t['elements']}, beyond 2e-2*rms by at most one bf16 ulp: "
        f"{t['over_strict']} ({t['over_strict'] / max(1, t['elements']):.2e}); worst single check "
        f"{t['worst_fraction']:.2e} (limit 1e-2)")
