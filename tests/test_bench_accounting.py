"""The benchmark's FLOP accounting: bench.visible_pairs counts the visible
(query, key) pairs with its own tile-level arithmetic; here it is checked
against the oracle's element-level mask definition (oracle/masks.py) on small
problems with every mask, and against closed forms.  The metric's FLOP
counts (4 d per pair forward, 10 d backward) rest on this count."""
import numpy as np
import pytest

import bench
from exact_io_aware_tiled_gb300 import workloads as W
from oracle import masks


def brute_force_pairs(wl):
    total = 0
    rows = np.arange(wl.N)
    for b in range(wl.B):
        L = None if wl.seqlens is None else int(wl.seqlens[b])
        vis = masks.visible(rows, rows, causal=wl.causal, seqlen_k=L,
                            block_mask=None if wl.block_mask is None else wl.block_mask.astype(bool),
                            block_size=wl.block_size, window=wl.window)
        total += int(vis.sum()) * wl.H
    return total


@pytest.mark.parametrize("kw", [
    dict(N=300),
    dict(N=300, causal=True),
    dict(N=520, causal=True, window=200),
    dict(N=400, seqlen_range=(100, 400)),
    dict(N=640, sparse_butterfly=True),
    dict(N=640, sparse_butterfly=True, causal=True, window=300, seqlen_range=(200, 640)),
    dict(N=129, causal=True, window=1),
])
def test_visible_pairs_matches_the_oracle_masks(kw):
    wl = W.Workload("acct", B=3, H=2, seed=5, **kw)
    assert bench.visible_pairs(wl) == brute_force_pairs(wl)


def test_visible_pairs_closed_forms():
    # dense: B H N^2; causal: B H N (N + 1) / 2; the GPT-2-medium workload's
    # 64 * 16 * 524,800 pairs
    assert bench.visible_pairs(W.Workload("d", B=2, H=3, N=1000)) == 2 * 3 * 1000 * 1000
    assert bench.visible_pairs(W.Workload("c", B=2, H=3, N=1000, causal=True)) == 2 * 3 * 1000 * 1001 // 2
    assert bench.visible_pairs(W.CONFIGS["gpt2_medium_causal"]) == 64 * 16 * 524_800


def test_launch_counts_per_step():
    assert bench._launches_per_step(W.CONFIGS["gpt2_medium_causal"]) == 4            # fwd, prep, bwd, convert
    assert bench._launches_per_step(W.CONFIGS["butterfly_sparse_64k"]) == 6          # + block lists twice
    assert bench._launches_per_step(W.CONFIGS["tiny_f32"]) == 3                      # no dQ convert
    assert bench._launches_per_step(W.CONFIGS["gpt2_medium_causal_fp8"]) == 2        # quantiser, forward
