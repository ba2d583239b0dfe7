"""The timeout path of the tcgen05 decode kernel, made to run out on purpose (no fault).

Every on-chip wait of the kernel (mbarriers between its roles and between the two CTAs of
a pair) is bounded.  A wait that runs out sets an abort word in both CTAs, every role
leaves its loop at the next wait (the 256 softmax threads only together, since they meet
at named barriers), the TMA loads and bulk copies already issued are waited for, the MMA
warps wait for their tensor-core operations, tensor memory is released, and the status
word gets MLA_STATUS_WAIT_TIMEOUT.  Here mla_set_test_stall makes one role of every
thread-block pair first wait for an arrival that never comes, with the limit set to
200 us through mla_set_wait_limit_ns: the call must return, report the timeout, and leave
the context usable -- the next call, with the default limit and no stall, must match the
oracle.  No wait is made to hang: each one gives up by itself, and nothing faults or
traps.
"""
import pytest
import torch

import mla_paged_decode_03_gb300 as M
import synth
from step_builder import step_from_workload

import gpu_helpers as H

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 8


@pytest.mark.parametrize("name,lengths,budget", [("cp2", None, M.BUDGET_AUTO),
                                                  ("long", [5000, 4097], M.BUDGET_WIDE)])
def test_wait_timeout_reports_and_recovers(name, lengths, budget):
    M.set_decode_kernel(M.KERNEL_AUTO)
    prev_b = M.set_rescale_budget(budget)
    w = synth.make_workload(name, lengths=lengths)
    step = step_from_workload(w, "cuda")
    assert M.device_status() == 0
    prev = M.set_wait_limit_ns(200_000)
    prev_stall = M.set_test_stall(True)
    try:
        step.run()
        torch.cuda.synchronize()
        bits = M.device_status()
    finally:
        M.set_test_stall(prev_stall)
        M.set_wait_limit_ns(prev)
    assert bits & TIMEOUT_BIT, f"no wait ran out (status {bits:#x})"
    assert bits & ~TIMEOUT_BIT == 0, f"unexpected status bits {bits:#x}"
    # the context is usable and the same step, with the default limit, is parity-green
    out, lse = step.run()
    torch.cuda.synchronize()
    assert M.device_status() == 0
    relative = name == "long"
    if relative:
        ro, rl, mo, ml, ra, ma, rd, md = H.oracle_shards(w, with_abs=True)
    else:
        ro, rl, mo, ml = H.oracle_shards(w)
        ma = md = None
    H.compare(out, lse, mo, ml, relative, f"{name} after a timed-out call", ma, md)
    M.set_rescale_budget(prev_b)


def test_wait_limit_setting_round_trips():
    prev = M.set_wait_limit_ns(123456)
    assert M.set_wait_limit_ns(prev) == 123456
    with pytest.raises(M.MlaError):
        M.set_wait_limit_ns(-1)
    assert M.set_test_stall(False) == 0


def test_tiny_wait_limit_returns():
    # with a 1 ns limit every wait that is not satisfied at once may run out (whether one
    # does depends on timing): the call returns either way and the status holds at most
    # the timeout bit; the next call with the default limit is clean
    w = synth.make_workload("cp2")
    step = step_from_workload(w, "cuda")
    prev = M.set_wait_limit_ns(1)
    try:
        step.run()
        torch.cuda.synchronize()
        bits = M.device_status()
    finally:
        M.set_wait_limit_ns(prev)
    assert bits & ~TIMEOUT_BIT == 0
    step.run()
    torch.cuda.synchronize()
    assert M.device_status() == 0
