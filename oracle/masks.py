"""Mask definitions of the method (causal, sliding window, key padding,
block-sparse).

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Readings taken (the pages only say masks are applied to the score tile on chip,
agihunt.info summary of arXiv 2205.14135, paragraph on the fused kernel; causal
means a query never attends to the future, marketmaker.cc, section "O
mascaramento causal"; block-sparse keeps or skips whole blocks of a fixed
butterfly pattern, agihunt.info, paragraph on block-sparse):

* causal is top-left aligned on the square N x N score matrix: key j is
  visible to query i iff j <= i;
* key padding masks keys only: key j is visible iff j < L_b for batch b;
  query rows i >= L_b are computed normally;
* block-sparse keeps whole ``bs`` x ``bs`` blocks: (i, j) visible iff
  kept[i // bs, j // bs];
* a sliding window of ``w`` keys (lynx-cortex, "Problemas de práctica", the
  sliding-window exercise: each query tile then reads only the K/V tiles
  that overlap its window) is read as the local causal window: key j is
  visible to query i iff i - w < j, combined with the causal j <= i, so a
  query sees itself and the w - 1 keys before it;
* the masks combine by logical AND.
"""
from __future__ import annotations

import numpy as np


def butterfly_block_mask(nblocks):
    """kept[I, J] iff I == J or I XOR J is a power of two (fixed butterfly)."""
    I = np.arange(nblocks)[:, None]
    J = np.arange(nblocks)[None, :]
    x = I ^ J
    return (x == 0) | ((x & (x - 1)) == 0)


def visible(rows, cols, *, causal=False, seqlen_k=None, block_mask=None, block_size=128, window=0):
    """Boolean [len(rows), len(cols)] visibility of (query row, key col)."""
    rows = np.asarray(rows, dtype=np.int64)[:, None]
    cols = np.asarray(cols, dtype=np.int64)[None, :]
    m = np.ones((rows.shape[0], cols.shape[1]), dtype=bool)
    if causal:
        m &= cols <= rows
    if window:
        m &= cols > rows - int(window)
    if seqlen_k is not None:
        m &= cols < int(seqlen_k)
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        m &= bm[rows // block_size, cols // block_size]
    return m
