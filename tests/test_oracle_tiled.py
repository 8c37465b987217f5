"""Pins for oracle.tiled: the three printed loop orders equal the one-shot softmax."""
import itertools

import numpy as np
import pytest

from oracle import attention as A
from oracle import tiled


def _case(N, d, seed):
    rng = np.random.default_rng(seed)
    return [2.0 * rng.standard_normal((N, d)) for _ in range(3)]


@pytest.mark.parametrize("variant", sorted(tiled.VARIANTS))
@pytest.mark.parametrize("N,d", [(1, 1), (2, 3), (5, 4), (9, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_all_tile_sizes_match_one_shot(variant, N, d, causal):
    q, k, v = _case(N, d, N * 10 + d)
    spec = A.Spec(B=1, H=1, N=N, d=d, causal=causal)
    O_ref, lse_ref = A.head_forward(spec, 0, 0, q, k, v)
    vis = (lambda r, c: c[None, :] <= r[:, None]) if causal else None
    for Br, Bc in itertools.product(range(1, N + 1), repeat=2):
        O, l, m = tiled.VARIANTS[variant](q, k, v, Br, Bc, vis=vis)
        assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-13), (Br, Bc)
        assert np.allclose(m + np.log(l), lse_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("variant", sorted(tiled.VARIANTS))
def test_ragged_tiles_n17(variant):
    N, d = 17, 4
    q, k, v = _case(N, d, 170)
    spec = A.Spec(B=1, H=1, N=N, d=d)
    O_ref, _ = A.head_forward(spec, 0, 0, q, k, v)
    for Br, Bc in [(1, 17), (17, 1), (4, 5), (16, 3), (8, 8), (6, 16), (17, 17)]:
        O, _, _ = tiled.VARIANTS[variant](q, k, v, Br, Bc)
        assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-13)


def test_bc_one_is_the_serial_running_max_and_sum():
    # lynx-cortex, practice problem 4: B_c -> 1 degenerates to a serial pass.
    N, d = 11, 3
    q, k, v = _case(N, d, 5)
    tau = 1 / np.sqrt(d)
    _, l, m = tiled.q_outer_deferred(q, k, v, Br=N, Bc=1)
    for i in range(N):
        mm, ll = -np.inf, 0.0
        for j in range(N):
            s = tau * float(q[i] @ k[j])
            mn = max(mm, s)
            ll = ll * np.exp(mm - mn) + np.exp(s - mn)
            mm = mn
        assert m[i] == pytest.approx(mm, abs=1e-14)
        assert l[i] == pytest.approx(ll, rel=1e-13)
