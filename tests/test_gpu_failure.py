"""Failure detection on the GPU without a fault: the bounded device-side wait.

fa_selftest_wait_timeout runs the attention kernels' wait routine on
mbarriers that nothing arrives at; the waits must give up, report
FA_ERR_TIMEOUT through the workspace status word, and leave the context
usable.  Nothing here traps, asserts on the device or hangs.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_tiled_gb300 as fa
from exact_io_aware_tiled_gb300 import _lib
from exact_io_aware_tiled_gb300 import workloads as W
from tests.parity import check_head, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    fa.load()


def test_bounded_wait_gives_up_reports_timeout_and_propagates_the_abort():
    status, gave_up, waited_ns = fa.selftest_wait_timeout()
    assert status == _lib.FA_ERR_TIMEOUT
    assert gave_up == [1, 1]
    # the second warp began one second after the first; it left on the abort
    # flag raised by the first, not after its own two-second limit.  The first
    # polls (as the backward kernels wait), the second sleeps between tries
    # (as the forward kernels wait), so both forms of the wait give up.
    assert 0.5e9 < waited_ns < 1.6e9, waited_ns


def test_context_is_usable_after_a_timeout():
    fa.selftest_wait_timeout()
    wl = W.Workload("after_timeout", B=1, H=2, N=200, dtype="bf16", causal=True, seed=11)
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    for h in range(wl.H):
        check_head(wl, inp, got, 0, h)
    # a fresh call leaves a clean status word
    assert fa.check_status(fa.fwd.last_workspace) == 0
