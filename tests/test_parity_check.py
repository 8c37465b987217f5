"""The gradient check of the GPU parity tests tests what it claims (CPU only).

The bound on dQ, dK and dV is a relative Frobenius error of 1e-2 (16-bit)
or 1e-5 (fp32) against the plain norm of the exact gradient.  A floor on the
denominator is allowed only where the exact gradient vanishes identically
(rows that see a single key: dS = P (dP - D) = 0).  These tests pin that:
ordinary heads get no floor, a 1.5e-2 relative error is rejected on them, and
the floor is taken exactly in the cases whose exact gradient is zero.
"""
import numpy as np
import pytest

from exact_io_aware_tiled_gb300 import workloads as W
from oracle import attention as A
from tests import parity as PT


def _head(wl, b=0, h=0):
    inp = W.make_inputs(wl)
    spec = PT.spec_of(wl)
    q, k, v, do = (PT.np64(inp[n][b, h]) for n in ("q", "k", "v", "do"))
    return spec, q, k, v, do


@pytest.mark.parametrize("causal", [True, False])
def test_ordinary_head_has_no_floor_and_rejects_a_1p5e2_error(causal):
    wl = W.Workload("ord", B=1, H=1, N=1024, dtype="bf16", causal=causal, seed=11)
    spec, q, k, v, do = _head(wl)
    gr = A.head_backward(spec, 0, 0, q, k, v, do)
    rows = np.arange(wl.N)
    assert not PT.rows_all_single_key(spec, 0, rows)
    assert not PT.cols_fed_by_single_key_rows(spec, 0, rows)
    # The uncancelled-magnitude floor the old check applied everywhere is
    # several times ||dQ|| on such a head: that is why it must not apply here.
    old_floor = 0.1 * spec.tau * np.linalg.norm(do) * PT._rms_row(v) * PT._rms_row(k)
    assert old_floor > 3 * np.linalg.norm(gr["dq"])
    rng = np.random.default_rng(5)
    for name in ("dq", "dk", "dv"):
        ref = gr[name]
        noise = rng.standard_normal(ref.shape)
        noise *= np.linalg.norm(ref) / np.linalg.norm(noise)
        rep = {}
        PT.grad_check(rep, name, ref + 0.005 * noise, ref, old_floor, 1e-2, False)
        assert rep[name + "_floored"] == 0.0
        assert abs(rep[name] - 0.005) < 1e-9
        with pytest.raises(AssertionError):
            PT.grad_check({}, name, ref + 0.015 * noise, ref, old_floor, 1e-2, False)


@pytest.mark.parametrize("kind", ["window1", "seqlen1", "n1_causal"])
def test_floor_only_where_the_exact_gradient_vanishes(kind):
    kw = dict(window1=dict(N=200, causal=True, window=1),
              seqlen1=dict(N=200, seqlen_range=(1, 1)),
              n1_causal=dict(N=1, causal=True))[kind]
    wl = W.Workload("deg", B=1, H=1, dtype="bf16", seed=12, **kw)
    spec, q, k, v, do = _head(wl)
    rows = np.arange(wl.N)
    assert PT.rows_all_single_key(spec, 0, rows)
    assert PT.cols_fed_by_single_key_rows(spec, 0, rows)
    gr = A.head_backward(spec, 0, 0, q, k, v, do)
    scale = np.linalg.norm(do) * PT._rms_row(v) * PT._rms_row(k)
    assert np.linalg.norm(gr["dq"]) <= 1e-12 * scale
    assert np.linalg.norm(gr["dk"]) <= 1e-12 * scale
    assert np.linalg.norm(gr["dv"]) > 0        # dV does not cancel


def test_one_two_key_row_turns_the_floor_off():
    """Causal rows 0 and 1: row 0 sees one key, row 1 two, so dQ of the pair
    does not vanish and the check must use ||dQ_ref||."""
    wl = W.Workload("two", B=1, H=1, N=64, dtype="bf16", causal=True, seed=13)
    spec, q, k, v, do = _head(wl)
    assert PT.rows_all_single_key(spec, 0, [0])
    assert not PT.rows_all_single_key(spec, 0, [0, 1])
    assert PT.cols_fed_by_single_key_rows(spec, 0, [wl.N - 1]) is False  # row N-1 sees N keys
