"""Failure path of the kernels' pipeline waits, on the GPU, without a fault.

Every mbarrier wait in the attention kernels is bounded; when the limit runs
out the kernel records VH_ERR_TIMEOUT in the caller's flag and winds down.
Here a wait is made to run out on purpose (a barrier nothing arrives on, the
library's own self-test launch), the status is read on the host, and the
context is then used for a normal decode step, which must still match the
oracle.  Nothing here traps, faults or hangs: the wait gives up by itself."""
import time

import pytest
import torch

import gpu_harness as H
import workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    v = H.vh()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    v.vh_selftest_wait_timeout(err)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) == v.VH_ERR_TIMEOUT
    assert 0.2 < dt < 20.0, f"the wait gave up after {dt:.2f} s"


@pytest.mark.parametrize("path", H.PATHS)
def test_context_usable_after_a_timeout(path):
    v = H.vh()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v.vh_selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) & v.VH_ERR_TIMEOUT
    # the device is fine: a normal step runs and matches the oracle, with a clean flag
    H.full_check(workloads.make_inputs("tiny", device="cuda"), path=path)
