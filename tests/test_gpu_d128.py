"""GPU parity at head dimension 128: the forward kernel (P overwrites S in
tensor memory, two 64-column boxes per tile) and the backward kernel (64-row
query steps, dQ formed transposed) against the float64 oracle on whole
heads, over ragged tails and every mask, and on sampled rows of the
GPT-2-medium-width workload with 8 heads of 128."""
import numpy as np
import pytest
import torch

from exact_io_aware_tiled_gb300 import workloads as W
import exact_io_aware_tiled_gb300 as fa
from tests.parity import check_head, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    fa.load()


def _wl(N, dtype="bf16", B=2, H=3, seed=11, **kw):
    return W.Workload("case_d128", B=B, H=H, N=N, d=128, dtype=dtype, seed=seed, **kw)


def _check_all_heads(wl, inp=None, layout="bhnd"):
    inp = W.make_inputs(wl) if inp is None else inp
    got = run_gpu(wl, inp, layout=layout)
    for b in range(wl.B):
        for h in range(wl.H):
            check_head(wl, inp, got, b, h)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N", [1, 127, 129, 300])
def test_dense(dtype, N):
    _check_all_heads(_wl(N, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N", [128, 129, 513])
def test_causal(dtype, N):
    _check_all_heads(_wl(N, dtype, causal=True))


def test_padding_dropout_and_causal():
    _check_all_heads(_wl(300, "bf16", B=3, seqlens=np.array([0, 1, 217], dtype=np.int32), dropout_p=0.2, causal=True))


def test_grouped_query_and_window():
    _check_all_heads(_wl(600, "f16", H=4, H_kv=2, causal=True, window=200))


def test_block_sparse_butterfly():
    _check_all_heads(_wl(1024, "bf16", B=1, H=2, sparse_butterfly=True))


def test_non_contiguous_layout():
    _check_all_heads(_wl(257, "bf16", causal=True), layout="bnhd")


def test_rescale_decided_per_row_within_a_warp():
    # neighbouring rows of one warp disagree on whether O must be rescaled
    # (see the d = 64 test of the same name); at d = 128 the rescale spans
    # four 32-column chunks of O
    wl = _wl(256, "bf16", B=1, H=2, seed=13)
    inp = W.make_inputs(wl)
    qs = torch.where(torch.arange(256) % 2 == 0, 4.0, 0.1).view(1, 1, 256, 1)
    ks = torch.where(torch.arange(256) < 128, 0.1, 4.0).view(1, 1, 256, 1)
    inp["q"] = (inp["q"].float() * qs).to(torch.bfloat16)
    inp["k"] = (inp["k"].float() * ks).to(torch.bfloat16)
    for w in (wl, wl.with_(causal=True)):
        _check_all_heads(w, inp)


def test_gpt2_medium_d128_causal_sampled():
    wl = W.CONFIGS["gpt2_medium_d128_causal"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    for b, h in [(0, 0), (63, 7)]:
        check_head(wl, inp, got, b, h)
    rows = sample_rows(wl.N, seed=128, extra=64)
    check_head(wl, inp, got, 31, 3, rows=rows, cols=rows)


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout(p):
    _check_all_heads(_wl(257, "f16", B=1, H=2, dropout_p=p))


def test_empty_key_tiles_and_ragged_half_steps():
    # keys past L_b leave whole 128-key items empty (dK = dV = 0 written
    # without a step), and N = 129 makes the last 128-row query tile's second
    # 64-row half start past N
    _check_all_heads(_wl(129 + 256, "bf16", B=3, H=2, seqlens=np.array([1, 129, 385], dtype=np.int32)))
    _check_all_heads(_wl(129, "bf16", B=1, H=2, causal=True))
