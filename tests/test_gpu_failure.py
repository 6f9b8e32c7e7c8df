"""Failure detection without a GPU fault: every kernel's waits are bounded
and, when a limit passes, raise HPC_FLAG_TIMEOUT and leave.  A self-test
kernel waits on a barrier nothing completes (the same wait helper, a short
limit); the flag is raised after the limit, the context stays usable and the
next decode step is correct."""

import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
from _gpu import assert_close, oracle_out, run_step
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, make_batch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [200, 2000])
def test_a_wait_that_runs_out_raises_the_flag_and_returns(limit_us):
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    hd.hpc_selftest_wait_timeout(flags, limit_us)
    e1.record()
    torch.cuda.synchronize()
    assert int(flags.item()) == hd.binding.HPC_FLAG_TIMEOUT
    waited_us = e0.elapsed_time(e1) * 1e3
    assert limit_us * 0.95 <= waited_us < limit_us + 50000


def test_the_context_stays_usable_after_a_timeout():
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    hd.hpc_selftest_wait_timeout(flags, 500)
    torch.cuda.synchronize()
    assert int(flags.item()) == hd.binding.HPC_FLAG_TIMEOUT
    batch = make_batch(WORKLOADS["tiny"], device="cuda")
    out, ws = run_step(batch)  # checks its own device flags and counters
    assert_close(out, oracle_out(batch), "bf16")
