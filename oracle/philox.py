"""Philox4xW-R counter-based generator and the dropout keep-mask of the method.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Why it is here.  The pages state only that the dropout mask is *not stored*: the
backward pass regenerates it from the saved random-number-generator state
(FlashAttention, Dao et al. 2022: tonho.wtf summary, section "como funciona";
agihunt.info summary of arXiv 2205.14135, paragraph on the backward pass).
Regenerating a mask element-by-element in any tile order requires a
counter-based generator.  We take Philox4x32-10 from Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11), written here from
the paper's description of the round:

* the counter is four W-bit words (c0, c1, c2, c3) and the key two (k0, k1);
* one round multiplies c0 by M0 and c2 by M1 into double-width products
  (hi, lo), then emits (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1,
  lo(M0*c0));
* between rounds the key is bumped by the Weyl constants (k0 += W0, k1 += W1);
* ten rounds.

The round is written once, generically over the word width W; the 4x64
instantiation is pinned bit-for-bit against ``numpy.random.Philox`` (a
Philox4x64-10), which fixes the word permutation, which words are multiplied
and the key schedule.  The 4x32 constants are the SC'11 paper's.

The dropout mapping (a reading; the pages fix no RNG):
  key      = (lo32(seed), hi32(seed))
  row_g    = (b*H + h)*N + i                  (global query row, < 2**32)
  counter  = (j >> 3, row_g, lo32(offset), hi32(offset))
  slice t  = j & 7 selects 16-bit half (t & 1) of output word (t >> 1),
             low half for even t
  keep     iff slice >= T, T = dropout_threshold(p) = round(p * 65536)
One Philox call therefore serves the eight keys 8g..8g+7 of one query row.
The mapping depends only on (b, h, i, j), never on tiling.
"""
from __future__ import annotations

import numpy as np

# Multipliers and Weyl (key-bump) constants, Salmon et al. SC'11.
PHILOX_CONST = {
    32: dict(M0=0xD2511F53, M1=0xCD9E8D57, W0=0x9E3779B9, W1=0xBB67AE85),
    64: dict(M0=0xD2E7470EE14C6C93, M1=0xCA5A826395121157,
             W0=0x9E3779B97F4A7C15, W1=0xBB67AE8584CAA73B),
}


def philox_block(counter, key, width=32, rounds=10):
    """One Philox4x{width}-{rounds} evaluation with plain Python integers.

    ``counter`` is 4 words, ``key`` 2 words, each < 2**width.  Returns 4 words.
    Pinned by: tests/test_oracle_philox.py (4x64 against numpy.random.Philox).
    """
    c = dict(PHILOX_CONST[width])
    mask = (1 << width) - 1
    c0, c1, c2, c3 = (int(x) & mask for x in counter)
    k0, k1 = (int(x) & mask for x in key)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + c["W0"]) & mask
            k1 = (k1 + c["W1"]) & mask
        p0 = c["M0"] * c0
        p1 = c["M1"] * c2
        hi0, lo0 = p0 >> width, p0 & mask
        hi1, lo1 = p1 >> width, p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return [c0, c1, c2, c3]


def philox4x32_vec(c0, c1, c2, c3, k0, k1, rounds=10):
    """Vectorised Philox4x32 over numpy arrays of counters (same key for all).

    Same round as ``philox_block`` with width 32; products of two 32-bit words
    are exact in uint64.  Pinned by: equality with ``philox_block`` on random
    counters (tests/test_oracle_philox.py).
    """
    K = PHILOX_CONST[32]
    m32 = np.uint64(0xFFFFFFFF)
    c0 = np.asarray(c0, dtype=np.uint64) & m32
    c1 = np.asarray(c1, dtype=np.uint64) & m32
    c2 = np.asarray(c2, dtype=np.uint64) & m32
    c3 = np.asarray(c3, dtype=np.uint64) & m32
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    M0, M1 = np.uint64(K["M0"]), np.uint64(K["M1"])
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + K["W0"]) & 0xFFFFFFFF
            k1 = (k1 + K["W1"]) & 0xFFFFFFFF
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & m32
        hi1, lo1 = p1 >> np.uint64(32), p1 & m32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
    return c0, c1, c2, c3


def dropout_threshold(p):
    """16-bit threshold T with keep iff slice >= T; P(drop) = T / 65536."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(np.floor(p * 65536.0 + 0.5))


def keep_mask(B, H, N, b, h, rows, p, seed, offset, cols=None):
    """Dropout keep-mask Z[r, j] (bool) for query rows ``rows`` of head (b, h).

    ``cols`` defaults to all keys 0..N-1.  See the module docstring for the
    mapping.  Pinned by: philox pins above plus the keep-rate and independence
    statistics in tests/test_oracle_philox.py.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
    row_g = (np.int64(b) * H + h) * N + rows
    if row_g.size and int(row_g.max()) >= 2 ** 32:
        raise ValueError("B*H*N must stay below 2**32")
    T = dropout_threshold(p)
    seed = int(seed) & (2 ** 64 - 1)
    offset = int(offset) & (2 ** 64 - 1)
    k0, k1 = seed & 0xFFFFFFFF, seed >> 32
    g = (cols >> 3)[None, :]
    w = philox4x32_vec(g, row_g[:, None], offset & 0xFFFFFFFF, offset >> 32, k0, k1)
    words = np.stack(w, axis=0)                      # [4, R, C]
    t = (cols & 7)[None, :]
    word = np.take_along_axis(words, np.broadcast_to((t >> 1)[None], (1,) + words.shape[1:]), axis=0)[0]
    half = np.where((t & 1) == 1, word >> np.uint64(16), word) & np.uint64(0xFFFF)
    return half >= np.uint64(T)
