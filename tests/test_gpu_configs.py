"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times: the whole problem runs on the GPU; the oracle checks sampled
heads, rows (first / last 128, every tile boundary +-1, random) and key
columns one by one.  The tiny float32 workload is checked in full."""
import numpy as np
import pytest

from exact_io_aware_tiled_gb300 import workloads as W
import exact_io_aware_tiled_gb300 as fa
from tests.parity import check_head, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    fa.load()


def test_tiny_f32_full():
    wl = W.CONFIGS["tiny_f32"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    for h in range(wl.H):
        check_head(wl, inp, got, 0, h)


def test_gpt2_medium_causal():
    wl = W.CONFIGS["gpt2_medium_causal"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    for b, h in [(0, 0), (63, 15), (31, 7), (17, 3)]:          # whole heads
        check_head(wl, inp, got, b, h)
    rng = np.random.default_rng(0)
    for _ in range(6):                                         # sampled rows / columns elsewhere
        b, h = int(rng.integers(wl.B)), int(rng.integers(wl.H))
        rows = sample_rows(wl.N, seed=b * 100 + h, extra=64)
        check_head(wl, inp, got, b, h, rows=rows, cols=rows)


def test_bert_large_padding_dropout():
    wl = W.CONFIGS["bert_large_pad_dropout"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    L = np.asarray(wl.seqlens)
    for b in sorted({int(L.argmin()), int(L.argmax()), 0, wl.B - 1}):
        for h in (0, wl.H - 1):
            check_head(wl, inp, got, b, h)


def test_long_ragged_causal_f16():
    wl = W.CONFIGS["long_ragged_causal_f16"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    rows = sample_rows(wl.N, seed=4, extra=128)
    cols = np.unique(np.concatenate([np.arange(0, 64), np.arange(wl.N - 200, wl.N),
                                     np.random.default_rng(5).integers(0, wl.N, 64)]))
    check_head(wl, inp, got, 0, 11, rows=rows, cols=cols)


def test_butterfly_sparse_64k():
    wl = W.CONFIGS["butterfly_sparse_64k"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    rows = sample_rows(wl.N, seed=6, extra=128)
    cols = np.concatenate([np.arange(0, 40), np.arange(128 * 255 - 3, 128 * 255 + 40), np.arange(wl.N - 40, wl.N)])
    check_head(wl, inp, got, 0, 5, rows=rows, cols=cols)


def test_gqa8_gpt2_medium_causal():
    wl = W.CONFIGS["gqa8_gpt2_medium_causal"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    for b, h in [(0, 1), (63, 15), (40, 9)]:       # odd heads: each closes a K/V group (dK, dV checked)
        check_head(wl, inp, got, b, h)
    rows = sample_rows(wl.N, seed=66, extra=64)
    check_head(wl, inp, got, 21, 7, rows=rows, cols=rows)


def test_window512_8k():
    wl = W.CONFIGS["window512_8k"]
    inp = W.make_inputs(wl)
    got = run_gpu(wl, inp)
    rows = sample_rows(wl.N, seed=77, extra=128)
    cols = np.unique(np.concatenate([np.arange(0, 64), np.arange(4000, 4200), np.arange(wl.N - 128, wl.N)]))
    check_head(wl, inp, got, 3, 12, rows=rows, cols=cols)
    check_head(wl, inp, got, 0, 0, rows=rows[:200], cols=cols[:100])
