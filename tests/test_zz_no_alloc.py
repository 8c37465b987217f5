"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Some callers cannot hand fa_bwd a workspace (they run inside a memory pool
they do not own, in a hook where allocation is forbidden, or from plain C
without a device allocator).  fa_bwd_noalloc takes its scratch from a fixed
array inside the library instead.  These tests call it through the C ABI
twice in a row and check both results against the ordinary fa_bwd, with the
gradient tolerance of the other parity tests; run a sequence of different
problems (block-sparse, head dimension 128, a smaller causal one) through
the one shared array, each against fa_bwd with its own workspace; check that
a timeout recorded in the array's status word is reported by
fa_noalloc_check_status and cleared by the next call; and check that a
problem too large for the fixed array is refused before anything runs.  The
file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_tiled_gb300 as fa
from exact_io_aware_tiled_gb300 import _lib
from exact_io_aware_tiled_gb300 import workloads as W
from tests.parity import TOL, kwargs_of, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    fa.load()


def _grads_match(a, b, tol):
    for x, y in zip(a, b):
        xn = x.float().cpu().numpy().astype(np.float64)
        yn = y.float().cpu().numpy().astype(np.float64)
        assert rel_frob(xn, yn) <= tol


def test_noalloc_backward_matches_fa_bwd_on_two_calls_in_a_row():
    wl = W.Workload("noalloc", B=2, H=3, N=700, dtype="bf16", causal=True, dropout_p=0.1, seed=11)
    inp = {k: v.cuda() for k, v in W.make_inputs(wl).items()}
    kw = kwargs_of(wl)
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], **kw)
    ref = fa.bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, **kw)
    tol = TOL[wl.dtype]["grad"]
    for _ in range(2):
        got = fa.bwd_noalloc(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, **kw)
        torch.cuda.synchronize()
        _grads_match(got, ref, tol)


def test_noalloc_backward_float32_path():
    wl = W.Workload("noalloc32", B=1, H=2, N=200, dtype="f32", seed=12)
    inp = {k: v.cuda() for k, v in W.make_inputs(wl).items()}
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"])
    ref = fa.bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse)
    for _ in range(2):
        got = fa.bwd_noalloc(inp["q"], inp["k"], inp["v"], o, inp["do"], lse)
        torch.cuda.synchronize()
        _grads_match(got, ref, TOL["f32"]["grad"])


def test_noalloc_reuses_the_array_across_different_problems():
    """The shared array keeps what the previous call left: block lists, the
    work counter, the dQ accumulator.  Each problem must still match fa_bwd
    with a fresh workspace of its own."""
    seq = [W.Workload("nz_sparse", B=1, H=2, N=640, dtype="bf16", sparse_butterfly=True, seed=21),
           W.Workload("nz_d128", B=1, H=2, N=300, d=128, dtype="bf16", seed=22),
           W.Workload("nz_causal", B=1, H=1, N=200, dtype="f16", causal=True, seed=23),
           W.Workload("nz_sparse_again", B=2, H=1, N=384, dtype="bf16", sparse_butterfly=True, causal=True,
                      seed=24)]
    for wl in seq:
        inp = {k: v.cuda() for k, v in W.make_inputs(wl).items()}
        kw = kwargs_of(wl)
        o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], **kw)
        ref = fa.bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, **kw)
        got = fa.bwd_noalloc(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, **kw)
        assert fa.noalloc_check_status() == 0, wl.name
        _grads_match(got, ref, TOL[wl.dtype]["grad"])


def test_noalloc_status_word_reports_a_timeout():
    addr, nbytes = fa.noalloc_scratch()
    assert nbytes == 64 << 20 and addr % 256 == 0
    # the bounded-wait self-test gives up and records FA_ERR_TIMEOUT at the
    # start of the fixed array, where fa_bwd_noalloc keeps its status word
    status, gave_up, _ = fa.selftest_wait_timeout(ws_ptr=addr)
    assert status == _lib.FA_ERR_TIMEOUT and gave_up == [1, 1]
    assert fa.noalloc_check_status() == _lib.FA_ERR_TIMEOUT
    # the next backward clears the word before it runs
    wl = W.Workload("nz_after", B=1, H=1, N=256, dtype="bf16", causal=True, seed=25)
    inp = {k: v.cuda() for k, v in W.make_inputs(wl).items()}
    o, lse = fa.fwd(inp["q"], inp["k"], inp["v"], causal=True)
    fa.bwd_noalloc(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, causal=True)
    assert fa.noalloc_check_status() == 0


def test_noalloc_refuses_problems_larger_than_its_array():
    lib = fa.load()
    fn = lib.fa_bwd_noalloc
    fn.argtypes = [ctypes.POINTER(_lib.fa_params)] + [ctypes.c_void_p] * 10
    fn.restype = ctypes.c_int
    p = _lib.fa_params()
    p.B, p.H, p.N, p.d, p.dtype = 64, 16, 1024, 64, 2      # needs ~280 MB of scratch
    p.stride_n, p.stride_h, p.stride_b = 64, 1024 * 64, 16 * 1024 * 64
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) > 64 << 20
    fake = ctypes.c_void_p(1 << 20)
    st = fn(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, None)
    assert st == _lib.FA_ERR_WORKSPACE
