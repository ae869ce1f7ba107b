import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case (full-size workloads)")


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


def pytest_terminal_summary(terminalreporter):
    """Report the top-k pick pairs that GPU tests saw in the opposite order to the oracle's
    (their fp64 logit gap against the fp32 error window that allowed the swap)."""
    try:
        from tests.helpers import SWAP_LOG
    except ImportError:
        return
    if SWAP_LOG:
        gaps = sorted(SWAP_LOG, key=lambda gw: -gw[0])
        terminalreporter.write_line(f"top-k order swaps: {len(gaps)}; largest fp64 gap {gaps[0][0]:.3e} "
                                    f"(window {gaps[0][1]:.3e}); largest gap/window "
                                    f"{max(g / w for g, w in gaps):.3f}")
    else:
        terminalreporter.write_line("top-k order swaps: none")
