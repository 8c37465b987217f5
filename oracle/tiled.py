"""CPU simulations of the three tiled online-softmax loop orders on the pages.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Each function takes one head (q, k, v: [N, d]), any tile sizes Br (query rows
per tile) and Bc (key rows per tile), ragged last tiles included, and an
optional visibility function vis(rows, cols) -> bool matrix.  They follow the
pages' own order of steps and notation:

* ``kv_outer_normalised`` -- tonho.wtf, section "como funciona": outer loop over
  K/V blocks, inner loop over Q blocks; block max m~, P~ = exp(S - m~),
  l_new = e^(m - m_new) l + e^(m~ - m_new) rowsum(P~), and O renormalised and
  written back (with l, m) every inner step.
* ``q_outer_normalised`` -- marketmaker.cc, section "O algoritmo de atenção do
  Flash": outer loop over Q blocks, inner over K/V blocks, the same running
  statistics with O renormalised every step.
* ``q_outer_deferred`` -- lynx-cortex, section "El algoritmo Flash (forward)":
  outer loop over Q blocks; m_new = max(m, rowmax S); alpha = e^(m - m_new);
  P = e^(S - m_new); l = alpha l + rowsum P; O = alpha O + P V; O / l once at
  the end.

The convention e^(-inf) = 0 covers rows of a block that are fully masked (a
guard the pages do not need because they have no masks; a reading).

``hbm`` is an optional ``oracle.traffic.Counter``; every load from / store to
the arrays that live in HBM (Q, K, V, O, l, m) is counted in elements, in the
order the page's loop performs them.

Pinned by tests/test_oracle_tiled.py: every variant agrees with the one-shot
softmax of ``oracle.attention`` for all (Br, Bc) on brute-force tiny inputs,
and Bc = 1 reproduces the serial running max / sum over keys.
"""
from __future__ import annotations

import numpy as np


def _exp0(x):
    """exp with exp(-inf) = 0 and exp(nan from -inf - -inf) = 0."""
    return np.where(np.isnan(x), 0.0, np.exp(x))


def _quiet(fn):
    """Run a loop variant with numpy's -inf - -inf warnings silenced."""
    def wrapped(*a, **kw):
        with np.errstate(invalid="ignore"):
            return fn(*a, **kw)
    wrapped.__name__, wrapped.__doc__ = fn.__name__, fn.__doc__
    return wrapped


def _blocks(n, b):
    return [(s, min(s + b, n)) for s in range(0, n, b)]


def _scores(q, k, rows, cols, tau, vis):
    S = tau * (q[rows[0]:rows[1]] @ k[cols[0]:cols[1]].T)
    if vis is not None:
        S = np.where(vis(np.arange(*rows), np.arange(*cols)), S, -np.inf)
    return S


class _NoCount:
    def read(self, n):
        pass

    def write(self, n):
        pass


@_quiet
def kv_outer_normalised(q, k, v, Br, Bc, tau=None, vis=None, hbm=None):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    N, d = q.shape
    tau = 1.0 / np.sqrt(d) if tau is None else tau
    hbm = hbm or _NoCount()
    O = np.zeros((N, v.shape[1]))          # lives in HBM
    l = np.zeros(N)                         # lives in HBM
    m = np.full(N, -np.inf)                 # lives in HBM
    for cj in _blocks(N, Bc):
        hbm.read(2 * (cj[1] - cj[0]) * d)                      # K_j, V_j
        Kj, Vj = k[cj[0]:cj[1]], v[cj[0]:cj[1]]
        for ri in _blocks(N, Br):
            nr = ri[1] - ri[0]
            hbm.read(nr * d + nr * v.shape[1] + 2 * nr)        # Q_i, O_i, l_i, m_i
            Oi, li, mi = O[ri[0]:ri[1]], l[ri[0]:ri[1]], m[ri[0]:ri[1]]
            S = _scores(q, k, ri, cj, tau, vis)
            m_til = S.max(axis=1)
            P_til = _exp0(S - m_til[:, None])
            m_new = np.maximum(mi, m_til)
            a_old = _exp0(mi - m_new)
            a_til = _exp0(m_til - m_new)
            l_new = a_old * li + a_til * P_til.sum(axis=1)
            safe = np.where(l_new > 0, l_new, 1.0)
            O[ri[0]:ri[1]] = ((li * a_old)[:, None] * Oi + a_til[:, None] * (P_til @ Vj)) / safe[:, None]
            l[ri[0]:ri[1]] = l_new
            m[ri[0]:ri[1]] = m_new
            hbm.write(nr * v.shape[1] + 2 * nr)                # O_i, l_i, m_i
    return O, l, m


@_quiet
def q_outer_normalised(q, k, v, Br, Bc, tau=None, vis=None, hbm=None):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    N, d = q.shape
    tau = 1.0 / np.sqrt(d) if tau is None else tau
    hbm = hbm or _NoCount()
    O = np.zeros((N, v.shape[1]))
    l_out = np.zeros(N)
    m_out = np.full(N, -np.inf)
    for ri in _blocks(N, Br):
        nr = ri[1] - ri[0]
        Oi = np.zeros((nr, v.shape[1]))
        li = np.zeros(nr)
        mi = np.full(nr, -np.inf)
        hbm.read(nr * d)                                       # Q_i
        for cj in _blocks(N, Bc):
            hbm.read(2 * (cj[1] - cj[0]) * d)                  # K_j, V_j
            S = _scores(q, k, ri, cj, tau, vis)
            m_ij = S.max(axis=1)
            P = _exp0(S - m_ij[:, None])
            l_ij = P.sum(axis=1)
            m_new = np.maximum(mi, m_ij)
            l_new = li * _exp0(mi - m_new) + l_ij * _exp0(m_ij - m_new)
            safe = np.where(l_new > 0, l_new, 1.0)
            Oi = Oi * (li * _exp0(mi - m_new) / safe)[:, None] \
                + (P @ v[cj[0]:cj[1]]) * (_exp0(m_ij - m_new) / safe)[:, None]
            mi, li = m_new, l_new
        O[ri[0]:ri[1]] = Oi
        l_out[ri[0]:ri[1]], m_out[ri[0]:ri[1]] = li, mi
        hbm.write(nr * v.shape[1])                             # O_i
    return O, l_out, m_out


@_quiet
def q_outer_deferred(q, k, v, Br, Bc, tau=None, vis=None, hbm=None):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    N, d = q.shape
    tau = 1.0 / np.sqrt(d) if tau is None else tau
    hbm = hbm or _NoCount()
    O = np.zeros((N, v.shape[1]))
    l_out = np.zeros(N)
    m_out = np.full(N, -np.inf)
    for ri in _blocks(N, Br):
        nr = ri[1] - ri[0]
        hbm.read(nr * d)                                       # Q_i
        Oi = np.zeros((nr, v.shape[1]))
        mi = np.full(nr, -np.inf)
        li = np.zeros(nr)
        for cj in _blocks(N, Bc):
            hbm.read(2 * (cj[1] - cj[0]) * d)                  # K_j, V_j
            S = _scores(q, k, ri, cj, tau, vis)
            m_new = np.maximum(mi, S.max(axis=1))
            alpha = _exp0(mi - m_new)
            P = _exp0(S - m_new[:, None])
            li = alpha * li + P.sum(axis=1)
            Oi = alpha[:, None] * Oi + P @ v[cj[0]:cj[1]]
            mi = m_new
        O[ri[0]:ri[1]] = Oi / np.where(li > 0, li, 1.0)[:, None]
        l_out[ri[0]:ri[1]], m_out[ri[0]:ri[1]] = li, mi
        hbm.write(nr * v.shape[1])                             # O_i
    return O, l_out, m_out


VARIANTS = {
    "kv_outer_normalised": kv_outer_normalised,
    "q_outer_normalised": q_outer_normalised,
    "q_outer_deferred": q_outer_deferred,
}
