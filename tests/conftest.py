import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# Tests whose purpose is to make a bounded device wait give up.
_EXPECTS_TIMEOUTS = ("test_failure_gpu.py",)


@pytest.fixture(autouse=True)
def _no_device_wait_timeouts(request):
    """After every GPU test: no bounded wait in a kernel gave up.  A CTA that
    gives up returns early with its output incomplete while the call itself
    has already returned LA_OK, so the device counter is the only witness."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    if os.path.basename(str(request.node.fspath)) in _EXPECTS_TIMEOUTS:
        return
    la = sys.modules.get("kernelized_sequence_mixing_gb300")
    if la is None or getattr(la, "_lib", None) is None or not cuda_available():
        return
    import torch
    torch.cuda.synchronize()
    n = la.device_wait_timeouts(reset=True)
    assert n == 0, f"{n} bounded device wait(s) gave up during {request.node.nodeid}"


def pytest_terminal_summary(terminalreporter):
    from helpers import MARGINS
    if not MARGINS:
        return
    terminalreporter.section("parity margins (worst error / tolerance)")
    for name, (err, tol) in sorted(MARGINS.items()):
        terminalreporter.write_line(f"{name}: {err:.3e} / {tol:.0e} "
                                    f"(margin x{tol / err if err > 0 else float('inf'):.1f})")
