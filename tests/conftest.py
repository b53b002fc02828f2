import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvq8.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA binding, built in-tree; GPU tests fail loudly without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a host without CUDA")
    from int8_quantized_kv_gb300 import kvq8
    kvq8.load()
    return kvq8


def pytest_terminal_summary(terminalreporter):
    """The largest output errors against the oracle, per GPU test."""
    h = sys.modules.get("kvq8_harness")
    if h is None or not getattr(h, "ERRORS", None):
        return
    tr = terminalreporter
    tr.write_sep("-", "largest d = gpu - oracle per test: max |d|, max |d|/max(1,|oracle|), "
                      "max |d|/max |oracle|")
    for test, vals in sorted(h.ERRORS.items()):
        tr.write_line(" ".join(f"{v:10.3e}" for v in vals) + f"  {test}")
