"""Pins for oracle.philox (CPU only)."""
import os

import numpy as np
import pytest

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "philox_kat.txt")


def _kat():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        f = lhs.split()
        width = int(f[0][len("philox4x"):])
        words = [int(x, 16) for x in f[2:]]
        out.append((width, int(f[1]), words[:4], words[4:6], [int(x, 16) for x in rhs.split()]))
    return out


def test_philox_known_answer_vectors():
    """The published known-answer vectors of Philox4x32-10 and Philox4x64-10
    (zero counter and key, all-ones, and the pi-digits case) pin the round,
    the multipliers and the Weyl key bumps of both widths."""
    kat = _kat()
    assert sorted({(w, r) for w, r, *_ in kat}) == [(32, 10), (64, 10)]
    assert len(kat) == 6
    for width, rounds, ctr, key, want in kat:
        assert philox.philox_block(ctr, key, width=width, rounds=rounds) == want, (width, ctr)
        if width == 32:
            got = philox.philox4x32_vec(*[np.array([c], dtype=np.uint64) for c in ctr], *key, rounds=rounds)
            assert [int(x[0]) for x in got] == want


def test_philox4x64_matches_numpy_bit_generator():
    # numpy.random.Philox is Philox4x64-10; it bumps the 256-bit counter by
    # one before producing each block of four words.
    rng = np.random.default_rng(7)
    for _ in range(20):
        ctr = [int(x) for x in rng.integers(0, 2**63, size=4, dtype=np.int64)]
        key = [int(x) for x in rng.integers(0, 2**63, size=2, dtype=np.int64)]
        bg = np.random.Philox(counter=ctr, key=key)
        got = [int(x) for x in bg.random_raw(8)]
        c = sum(w << (64 * i) for i, w in enumerate(ctr))
        for blk in range(2):
            cc = (c + 1 + blk) % (1 << 256)
            words = [(cc >> (64 * i)) & (2**64 - 1) for i in range(4)]
            assert philox.philox_block(words, key, width=64) == got[4 * blk:4 * blk + 4]


def test_philox4x32_vectorised_equals_generic():
    rng = np.random.default_rng(11)
    ctr = rng.integers(0, 2**32, size=(4, 200), dtype=np.uint64)
    k0, k1 = 0x12345678, 0x9ABCDEF0
    vec = philox.philox4x32_vec(*ctr, k0, k1)
    for n in range(200):
        ref = philox.philox_block([int(ctr[i, n]) for i in range(4)], [k0, k1], width=32)
        assert [int(vec[i][n]) for i in range(4)] == ref


def test_rounds_and_key_matter():
    a = philox.philox_block([1, 2, 3, 4], [5, 6], 32, 10)
    assert a != philox.philox_block([1, 2, 3, 4], [5, 6], 32, 9)
    assert a != philox.philox_block([1, 2, 3, 4], [5, 7], 32, 10)
    assert a != philox.philox_block([1, 2, 3, 5], [5, 6], 32, 10)


def test_threshold():
    assert philox.dropout_threshold(0.0) == 0
    assert philox.dropout_threshold(0.1) == 6554
    assert philox.dropout_threshold(0.5) == 32768
    with pytest.raises(ValueError):
        philox.dropout_threshold(1.0)


def test_mask_depends_only_on_element_index():
    B, H, N = 2, 3, 77
    full = philox.keep_mask(B, H, N, 1, 2, np.arange(N), 0.3, 99, 5)
    rows = np.array([0, 13, 76, 40])
    cols = np.array([75, 0, 8, 9, 15, 16, 31])
    sub = philox.keep_mask(B, H, N, 1, 2, rows, 0.3, 99, 5, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])
    # a different head, seed or offset gives a different mask
    assert not np.array_equal(full, philox.keep_mask(B, H, N, 0, 2, np.arange(N), 0.3, 99, 5))
    assert not np.array_equal(full, philox.keep_mask(B, H, N, 1, 2, np.arange(N), 0.3, 98, 5))
    assert not np.array_equal(full, philox.keep_mask(B, H, N, 1, 2, np.arange(N), 0.3, 99, 6))


def test_p_zero_keeps_everything():
    # T = 0: every 16-bit slice, including the ~32 zero slices among these
    # 2M draws, is >= T and kept.
    assert philox.keep_mask(1, 1, 2048, 0, 0, np.arange(1024), 0.0, 1, 0).all()


@pytest.mark.slow
def test_keep_rate_and_independence():
    # >= 10^7 draws: keep rate within 5 sigma of 1 - T/65536, and 2x2
    # contingency tables of horizontally / vertically adjacent elements show
    # no dependence (chi-square, 1 dof, far below 30).
    p = 0.1
    T = philox.dropout_threshold(p)
    q = 1.0 - T / 65536.0
    N = 4096
    kept = 0
    total = 0
    tabs_h = np.zeros((2, 2))
    tabs_v = np.zeros((2, 2))
    prev_last = None
    for r0 in range(0, 2560, 256):
        Z = philox.keep_mask(1, 1, N, 0, 0, np.arange(r0, r0 + 256), p, 0x5EED, 0)
        kept += int(Z.sum())
        total += Z.size
        a, b = Z[:, :-1].ravel(), Z[:, 1:].ravel()
        for x in (0, 1):
            for y in (0, 1):
                tabs_h[x, y] += np.sum((a == x) & (b == y))
        a, b = Z[:-1].ravel(), Z[1:].ravel()
        for x in (0, 1):
            for y in (0, 1):
                tabs_v[x, y] += np.sum((a == x) & (b == y))
    assert total >= 10**7
    sigma = np.sqrt(total * q * (1 - q))
    assert abs(kept - total * q) < 5 * sigma
    for t in (tabs_h, tabs_v):
        e = t.sum(1, keepdims=True) * t.sum(0, keepdims=True) / t.sum()
        chi2 = ((t - e) ** 2 / e).sum()
        assert chi2 < 30.0
