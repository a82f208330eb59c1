import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built specverify library")


def golden(name):
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def sv():
    """The CUDA binding, built in-tree; GPU tests fail loudly if it cannot load."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from serving_sampler_gb300 import _build

    _build.build()
    import serving_sampler_gb300 as m

    m.load()
    return m


def pytest_terminal_summary(terminalreporter):
    """The exempt-row counts of every sampling comparison (decision margin below 1e-6)."""
    try:
        from tests.sampling_parity import EXEMPT_LOG
    except Exception:
        return
    if not EXEMPT_LOG:
        return
    ex = sum(e for _, e, _, _ in EXEMPT_LOG)
    rows = sum(n for _, _, n, _ in EXEMPT_LOG)
    diff = sum(d for _, _, _, d in EXEMPT_LOG)
    worst = max(EXEMPT_LOG, key=lambda t: t[1] / max(t[2], 1))
    terminalreporter.write_line(
        f"exempt rows (decision margin < 1e-6): {ex} of {rows} rows in {len(EXEMPT_LOG)} comparisons "
        f"(rate {ex / max(rows, 1):.2e}); requests differing from the oracle: {diff}; "
        f"highest rate: {worst[0]} {worst[1]}/{worst[2]}")
