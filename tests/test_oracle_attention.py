"""Pins for oracle.attention (CPU only): invariants, closed forms, finite differences."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import masks


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _spec(N, d, **kw):
    return A.Spec(B=1, H=1, N=N, d=d, **kw)


MASK_CASES = [
    dict(),
    dict(causal=True),
    dict(seqlens_k=np.array([5])),
    dict(block_mask=np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], dtype=bool), block_size=4),
    dict(causal=True, seqlens_k=np.array([7]),
         block_mask=np.array([[1, 0, 1], [1, 1, 0], [1, 1, 1]], dtype=bool), block_size=4),
]


@pytest.mark.parametrize("mk", MASK_CASES)
def test_rows_are_distributions_and_masked_entries_zero(mk):
    # With V = I (N = d) the output is P itself.
    rng = np.random.default_rng(0)
    N = 12
    spec = _spec(N, N, **mk)
    q, k = _rand(rng, N, N), _rand(rng, N, N)
    P, lse = A.head_forward(spec, 0, 0, q, k, np.eye(N))
    vis = A.visible(spec, 0, np.arange(N), np.arange(N))
    assert np.all(P >= 0)
    assert np.all(P[~vis] == 0.0)
    has = vis.any(axis=1)
    assert np.allclose(P[has].sum(axis=1), 1.0, atol=1e-14, rtol=0)
    assert np.all(P[~has] == 0.0) and np.all(np.isneginf(lse[~has]))


def test_equal_scores_give_mean_of_visible_values():
    rng = np.random.default_rng(1)
    N, d = 9, 4
    v = _rand(rng, N, d)
    k = _rand(rng, N, d)
    q = np.zeros((N, d))
    O, lse = A.head_forward(_spec(N, d), 0, 0, q, k, v)
    assert np.allclose(O, v.mean(axis=0)[None, :], atol=1e-15)
    assert np.allclose(lse, math.log(N))
    O, _ = A.head_forward(_spec(N, d, causal=True), 0, 0, q, k, v)
    for i in range(N):
        assert np.allclose(O[i], v[:i + 1].mean(axis=0), atol=1e-15)
    assert np.array_equal(O[0], v[0])
    # all keys equal (instead of Q = 0) also gives equal scores
    O, _ = A.head_forward(_spec(N, d), 0, 0, _rand(rng, N, d), np.tile(k[:1], (N, 1)), v)
    assert np.allclose(O, v.mean(axis=0)[None, :], atol=1e-14)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(2)
    N, d = 6, 3
    q, k, v = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    O, lse = A.head_forward(_spec(N, d, seqlens_k=np.array([1])), 0, 0, q, k, v)
    assert np.array_equal(O, np.tile(v[0], (N, 1)))
    assert np.allclose(lse, (q @ k[0]) / math.sqrt(d))


def test_shift_invariance_of_the_softmax():
    # Adding w to every key adds tau q_i . w to the whole row i of S: P is
    # unchanged (living-dl-book, section 8, the pause on subtracting a constant).
    rng = np.random.default_rng(3)
    N, d = 10, 5
    q, k, v = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    w = 3.0 * _rand(rng, d)
    for mk in MASK_CASES[:3]:
        s = _spec(N, d, **mk)
        O1, l1 = A.head_forward(s, 0, 0, q, k, v)
        O2, l2 = A.head_forward(s, 0, 0, q, k + w, v)
        assert np.allclose(O1, O2, atol=1e-13)
        assert np.allclose(l2 - l1, (q @ w) / math.sqrt(d), atol=1e-12)


def test_two_keys_closed_form():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 2, 1), _rand(rng, 2, 1), _rand(rng, 2, 1)
    O, lse = A.head_forward(_spec(2, 1), 0, 0, q, k, v)
    for i in range(2):
        s0, s1 = q[i, 0] * k[0, 0], q[i, 0] * k[1, 0]
        sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        assert abs(O[i, 0] - (sig * v[0, 0] + (1 - sig) * v[1, 0])) < 1e-15
        assert abs(lse[i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-14


def test_lse_against_fsum():
    rng = np.random.default_rng(5)
    N, d = 7, 3
    q, k, v = 4 * _rand(rng, N, d), 4 * _rand(rng, N, d), _rand(rng, N, d)
    _, lse = A.head_forward(_spec(N, d), 0, 0, q, k, v)
    tau = 1 / math.sqrt(d)
    for i in range(N):
        s = [tau * sum(q[i, c] * k[j, c] for c in range(d)) for j in range(N)]
        ref = math.log(math.fsum(math.exp(x) for x in s))
        assert abs(lse[i] - ref) < 1e-13


def test_dropout_placement_one_hot_values():
    # Q = 0 (equal scores), V = I: O_ij = Z_ij / (n_visible (1 - p)).
    # Dropout acts on the normalised P, scaled by 1/(1-p); l uses undropped P.
    N = 16
    p = 0.25
    spec = A.Spec(B=2, H=3, N=N, d=N, dropout_p=p, seed=1234, offset=7, causal=True)
    O, lse = A.head_forward(spec, 1, 2, np.zeros((N, N)), np.ones((N, N)), np.eye(N))
    Z = A.keep(spec, 1, 2, np.arange(N), np.arange(N))
    nvis = np.arange(1, N + 1)[:, None]
    assert np.allclose(O, np.tril(Z) / (nvis * (1 - p)), atol=1e-15)
    assert np.allclose(lse, np.log(np.arange(1, N + 1)))
    assert 0 < Z.sum() < N * N


def _loss_grads(spec, q, k, v, do):
    O, _ = A.head_forward(spec, 0, 0, q, k, v)
    return float((O * do).sum()), A.head_backward(spec, 0, 0, q, k, v, do)


FD_CASES = MASK_CASES + [dict(dropout_p=0.3), dict(causal=True, dropout_p=0.5)]


@pytest.mark.parametrize("mk", FD_CASES)
def test_gradients_match_central_differences(mk):
    rng = np.random.default_rng(6)
    N, d = 12, 5
    mk = dict(mk)
    if "dropout_p" in mk:
        mk["fixed_keep"] = (rng.random((1, 1, N, N)) >= mk["dropout_p"])
    spec = _spec(N, d, **mk)
    q, k, v, do = (_rand(rng, N, d) for _ in range(4))
    _, g = _loss_grads(spec, q, k, v, do)
    h = 1e-6
    for name, x, gx in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = dict(q=q, k=k, v=v)
            args[name] = xp
            lp = float((A.head_forward(spec, 0, 0, **args)[0] * do).sum())
            args[name] = xm
            lm = float((A.head_forward(spec, 0, 0, **args)[0] * do).sum())
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - gx).max() / max(1e-12, np.abs(gx).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("mk", MASK_CASES + [dict(dropout_p=0.2, seed=3)])
def test_D_equals_rowwise_dO_dot_O(mk):
    # tonho.wtf, "como funciona": D_i = P_i . dP_i = dO_i . O_i.
    rng = np.random.default_rng(8)
    N, d = 12, 6
    spec = _spec(N, d, **mk)
    q, k, v, do = (_rand(rng, N, d) for _ in range(4))
    O, _ = A.head_forward(spec, 0, 0, q, k, v)
    g = A.head_backward(spec, 0, 0, q, k, v, do)
    assert np.allclose(g["D"], (do * O).sum(axis=1), atol=1e-13)


def test_row_and_column_sampling_is_consistent():
    rng = np.random.default_rng(9)
    N, d = 40, 4
    old = A.ROW_CHUNK
    A.ROW_CHUNK = 16
    try:
        spec = _spec(N, d, causal=True, seqlens_k=np.array([33]))
        q, k, v, do = (_rand(rng, N, d) for _ in range(4))
        Of, lf = A.head_forward(spec, 0, 0, q, k, v)
        rows = np.array([39, 0, 17, 16])
        Os, ls = A.head_forward(spec, 0, 0, q, k, v, rows=rows)
        assert np.allclose(Os, Of[rows]) and np.allclose(ls, lf[rows])
        gf = A.head_backward(spec, 0, 0, q, k, v, do)
        cols = np.array([5, 32, 33, 0])
        gs = A.head_backward(spec, 0, 0, q, k, v, do, rows=rows, cols=cols)
        assert np.allclose(gs["dq"], gf["dq"][rows], atol=1e-13)
        assert np.allclose(gs["dk"], gf["dk"][cols], atol=1e-13)
        assert np.allclose(gs["dv"], gf["dv"][cols], atol=1e-13)
        assert np.all(gf["dk"][33:] == 0) and np.all(gf["dv"][33:] == 0)
    finally:
        A.ROW_CHUNK = old


def test_butterfly_block_counts():
    bm = masks.butterfly_block_mask(512)
    assert bm.sum(axis=1).min() == 10 and bm.sum(axis=1).max() == 10
    assert bm.sum() == 5120
    assert np.array_equal(bm, bm.T)
