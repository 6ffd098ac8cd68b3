"""Failure detection without a GPU fault: the kernels' bounded waits give up
after their limit, count themselves in a device counter the host reads, and
leave the context usable.  The test makes one such wait run out (a barrier
that nothing arrives on, a 1e6-cycle limit) through the library's
diagnostic entry point; nothing traps, faults or hangs."""
import pytest
import torch

from helpers import max_row_error, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kernelized_sequence_mixing_gb300 import build
    build.build()
    import kernelized_sequence_mixing_gb300 as m
    return m


def test_bounded_wait_gives_up_and_reports(la, oracle_mod):
    torch.cuda.synchronize()
    la.device_wait_timeouts(reset=True)
    assert la.wait_selftest(1_000_000) is True
    assert la.device_wait_timeouts() == 1
    assert la.wait_selftest(2_000_000) is True
    assert la.device_wait_timeouts(reset=True) == 2
    assert la.device_wait_timeouts() == 0
    # the context is still usable: a forward pass on tensor cores is correct
    from kernelized_sequence_mixing_gb300.workloads import make_qkv
    q, k, v = make_qkv(1, 2, 300, 128, 128, torch.bfloat16, 3, 0.5)
    o = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    ref = oracle_mod.causal(to_np(q), to_np(k), to_np(v))
    assert max_row_error(to_np(o), ref) < 2e-2
    assert la.device_wait_timeouts() == 0
