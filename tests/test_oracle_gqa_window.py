"""Pins for the grouped-query and sliding-window readings of the oracle (CPU only).

Grouped-query attention: living-dl-book, efficient attention, section 6 (h query
heads in h/g groups, one K head and one V head per group; g = 1 is multi-head,
g = h is multi-query).  Sliding window: lynx-cortex, "Problemas de práctica"
(the window exercise), read as the local causal window i - w < j <= i.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import masks
from oracle import tiled as T


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- window
def test_window_of_one_key_returns_own_value():
    # each query sees only itself: O_i = V_i and LSE_i = tau q_i . k_i
    rng = np.random.default_rng(20)
    N, d = 11, 4
    q, k, v = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    spec = A.Spec(B=1, H=1, N=N, d=d, causal=True, window=1)
    O, lse = A.head_forward(spec, 0, 0, q, k, v)
    assert np.array_equal(O, v)
    assert np.allclose(lse, (q * k).sum(axis=1) / math.sqrt(d), atol=1e-14)


def test_window_covering_the_sequence_is_plain_causal():
    rng = np.random.default_rng(21)
    N, d = 13, 3
    q, k, v = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    for w in (N, N + 5):
        O1, l1 = A.head_forward(A.Spec(B=1, H=1, N=N, d=d, causal=True, window=w), 0, 0, q, k, v)
        O2, l2 = A.head_forward(A.Spec(B=1, H=1, N=N, d=d, causal=True), 0, 0, q, k, v)
        assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("w", [2, 3, 7])
def test_window_against_a_scalar_loop(w):
    # independent restatement: query i averages V over keys max(0, i-w+1) .. i
    # with weights exp(s_ij), summed with math.fsum
    rng = np.random.default_rng(22 + w)
    N, d = 10, 3
    q, k, v = 2 * _rand(rng, N, d), 2 * _rand(rng, N, d), _rand(rng, N, d)
    O, lse = A.head_forward(A.Spec(B=1, H=1, N=N, d=d, causal=True, window=w), 0, 0, q, k, v)
    tau = 1 / math.sqrt(d)
    for i in range(N):
        js = range(max(0, i - w + 1), i + 1)
        s = {j: tau * math.fsum(q[i, c] * k[j, c] for c in range(d)) for j in js}
        m = max(s.values())
        wts = {j: math.exp(s[j] - m) for j in js}
        z = math.fsum(wts.values())
        for c in range(d):
            assert abs(O[i, c] - math.fsum(wts[j] * v[j, c] for j in js) / z) < 1e-14
        assert abs(lse[i] - (m + math.log(z))) < 1e-14


def test_window_mask_counts():
    # a causal window of w keys leaves min(i + 1, w) visible keys in row i
    N, w = 300, 37
    vis = masks.visible(np.arange(N), np.arange(N), causal=True, window=w)
    assert np.array_equal(vis.sum(axis=1), np.minimum(np.arange(N) + 1, w))
    # and combines with key padding by AND
    vis2 = masks.visible(np.arange(N), np.arange(N), causal=True, window=w, seqlen_k=100)
    assert np.array_equal(vis2, vis & (np.arange(N)[None, :] < 100))


@pytest.mark.parametrize("Br,Bc", [(4, 4), (3, 5), (16, 2)])
def test_tiled_recurrence_with_window_matches_definition(Br, Bc):
    rng = np.random.default_rng(23)
    N, d, w = 17, 4, 6
    q, k, v = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    spec = A.Spec(B=1, H=1, N=N, d=d, causal=True, window=w)
    vis = lambda r, c: A.visible(spec, 0, r, c)
    O_ref, _ = A.head_forward(spec, 0, 0, q, k, v)
    for fn in (T.kv_outer_normalised, T.q_outer_normalised, T.q_outer_deferred):
        O = fn(q, k, v, Br, Bc, vis=vis)
        O = O[0] if isinstance(O, tuple) else O
        assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-12), fn.__name__


# ---------------------------------------------------------------- grouped-query
def _problem(rng, B, H, Hkv, N, d):
    return (_rand(rng, B, H, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d), _rand(rng, B, H, N, d))


@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1), (4, 4)])
def test_grouped_query_gradients_match_central_differences(H, Hkv):
    # the loss sum(O * dO) over all query heads; a shared K/V entry moves the
    # outputs of every query head of its group, so its finite difference pins
    # the summation over the group (and the head mapping h -> h // g)
    rng = np.random.default_rng(30 + H + Hkv)
    B, N, d = 1, 6, 3
    spec = A.Spec(B=B, H=H, N=N, d=d, causal=True, H_kv=Hkv, window=4)
    q, k, v, do = _problem(rng, B, H, Hkv, N, d)
    _, dk, dv, _ = A.attention_bwd(spec, q, k, v, do)
    dq = A.attention_bwd(spec, q, k, v, do)[0]
    h = 1e-6
    loss = lambda qq, kk, vv: float((A.attention_fwd(spec, qq, kk, vv)[0] * do).sum())
    for name, x, gx in (("k", k, dk), ("v", v, dv), ("q", q, dq)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = dict(qq=q, kk=k, vv=v)
            args[name * 2] = xp
            lp = loss(**args)
            args[name * 2] = xm
            lm = loss(**args)
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - gx).max() / max(1e-12, np.abs(gx).max())
        assert err < 1e-6, (name, err)


def test_multi_query_equal_scores_average_the_single_value_head():
    # g = h (one K/V head): with Q = 0 every query head averages V of that head
    rng = np.random.default_rng(40)
    B, H, N, d = 2, 3, 7, 4
    spec = A.Spec(B=B, H=H, N=N, d=d, H_kv=1)
    q = np.zeros((B, H, N, d))
    k, v = _rand(rng, B, 1, N, d), _rand(rng, B, 1, N, d)
    O, lse = A.attention_fwd(spec, q, k, v)
    for b in range(B):
        for hh in range(H):
            assert np.allclose(O[b, hh], v[b, 0].mean(axis=0)[None, :], atol=1e-15)
    assert np.allclose(lse, math.log(N))


def test_group_must_divide_heads():
    with pytest.raises(AssertionError):
        _ = A.Spec(B=1, H=5, N=4, d=2, H_kv=2).group
