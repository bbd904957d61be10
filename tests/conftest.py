import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly when no GPU is present: they must not be silently
    # skipped on a GPU box, so only deselection (-m "not gpu") keeps them out.
    pass


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Worst error / bound ratio of every floating-point parity check that
    ran (1.0 is the bound), or relative Frobenius error where marked."""
    gu = sys.modules.get("gpu_util")
    if gu is None or not getattr(gu, "WORST", None):
        return
    terminalreporter.write_sep("-", "worst parity ratios (1.0 = at the bound)")
    for name in sorted(gu.WORST):
        terminalreporter.write_line("%-60s %.4g" % (name, gu.WORST[name]))
