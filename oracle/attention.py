"""Exact scaled-dot-product attention, forward and backward, by definition.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

This is the plain definition that the tiled method reaches up to rounding
(exactness: tonho.wtf, "o que fica" item 2; marketmaker.cc, section "A
recorrência do softmax online"; lynx-cortex, "Por qué Flash es exacto").  It
materialises the N x N score matrix S and probability matrix P of one (b, h)
head in float64, exactly as the "standard attention" the pages describe
(lynx-cortex, "El algoritmo naive de attention" steps 1-3; marketmaker.cc,
"Por que a atenção está ligada à memória"):

  1. S = tau * Q K^T, tau = 1/sqrt(d) unless given.
  2. S_ij = -inf where (i, j) is masked (``oracle.masks``).
  Grouped-query attention (living-dl-book, efficient attention, section 6:
  the h query heads form h_kv = h / g groups, each sharing one K head and one
  V head): query head h reads K and V head h // g, and the gradient of a
  shared K or V head is the sum of its g query heads' contributions
  (``attention_fwd`` / ``attention_bwd``; the per-head functions take the
  head's own K and V rows).
  3. m_i = max_j S_ij;  P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i);
     LSE_i = m_i + ln sum_j exp(S_ij - m_i)  (natural log, tau-scaled units).
     A row with no visible key has P_i = 0, O_i = 0, LSE_i = -inf and zero
     gradients (a reading; the pages have no such row).
  4. Dropout (reading: on the normalised P, inverted scaling):
     P~ = Z o P / (1 - p), Z from ``oracle.philox.keep_mask``.  The softmax
     statistics use the undropped P.
  5. O = P~ V.
  6. Backward for an upstream gradient dO (chain rule; the pages give the
     recomputation and the identity D_i = dO_i . O_i, tonho.wtf "como
     funciona"):
       dV = P~^T dO;  dP~ = dO V^T;  dP = Z o dP~ / (1 - p);
       D_i = sum_j P_ij dP_ij;  dS = P o (dP - D);
       dQ = tau dS K;  dK = tau dS^T Q.

Rows are processed in chunks of ``ROW_CHUNK`` only to bound memory for long
sequences; the arithmetic per element is the definition above.

Pinned by tests/test_oracle_attention.py: row sums, masked zeros, equal-score
means, single-key rows, shift invariance, the d=1/N=2 closed form, a
``math.fsum`` log-sum-exp, a one-hot dropout placement case, central finite
differences of every gradient (with each mask and a fixed dropout mask) and
the D_i = dO_i . O_i identity.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import masks as _masks
from . import philox as _philox

ROW_CHUNK = 2048


@dataclass
class Spec:
    """Problem description shared by every oracle entry point."""
    B: int
    H: int
    N: int
    d: int
    scale: Optional[float] = None          # None -> 1/sqrt(d)
    causal: bool = False
    seqlens_k: Optional[np.ndarray] = None  # [B] ints or None
    block_mask: Optional[np.ndarray] = None  # [nb, nb] bool or None
    block_size: int = 128
    dropout_p: float = 0.0
    seed: int = 0
    offset: int = 0
    fixed_keep: Optional[np.ndarray] = field(default=None, repr=False)  # [B,H,N,N] test hook
    H_kv: Optional[int] = None               # K/V heads (grouped-query); None -> H
    window: int = 0                          # sliding window of keys (0 = none)

    @property
    def tau(self) -> float:
        return float(1.0 / np.sqrt(self.d)) if self.scale is None else float(self.scale)

    @property
    def hkv(self) -> int:
        return self.H if self.H_kv is None else int(self.H_kv)

    @property
    def group(self) -> int:
        """Query heads per K/V head (g); query head h reads K/V head h // g."""
        assert self.H % self.hkv == 0, "H must be a multiple of H_kv"
        return self.H // self.hkv


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def visible(spec: Spec, b, rows, cols):
    L = None if spec.seqlens_k is None else int(spec.seqlens_k[b])
    return _masks.visible(rows, cols, causal=spec.causal, seqlen_k=L,
                          block_mask=spec.block_mask, block_size=spec.block_size, window=spec.window)


def keep(spec: Spec, b, h, rows, cols):
    """Dropout keep-mask Z for (rows x cols) of head (b, h); ones if no dropout."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    if spec.fixed_keep is not None:
        return spec.fixed_keep[b, h][np.ix_(rows, cols)].astype(bool)
    if spec.dropout_p == 0.0:
        return np.ones((rows.size, cols.size), dtype=bool)
    return _philox.keep_mask(spec.B, spec.H, spec.N, b, h, rows, spec.dropout_p,
                             spec.seed, spec.offset, cols=cols)


def _softmax_rows(S, vis):
    """P, LSE of masked score rows S (visible entries only)."""
    S = np.where(vis, S, -np.inf)
    m = S.max(axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.where(vis, np.exp(S - m_safe[:, None]), 0.0)
    ell = E.sum(axis=1)
    P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, ell)[:, None])
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, ell)))
    return P, lse


def head_forward(spec: Spec, b, h, q, k, v, rows=None):
    """O and LSE of one head for query ``rows`` (default all).

    q, k, v: [N, d] arrays of the head (any float dtype; decoded to float64).
    Returns (O [len(rows), d], LSE [len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    N = k.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(N)
    tau = spec.tau
    O = np.zeros((rows.size, v.shape[1]))
    lse = np.zeros(rows.size)
    for s in range(0, rows.size, ROW_CHUNK):
        r = rows[s:s + ROW_CHUNK]
        S = tau * (q[r] @ k.T)
        P, lse[s:s + ROW_CHUNK] = _softmax_rows(S, visible(spec, b, r, cols))
        Pt = keep(spec, b, h, r, cols) * P / (1.0 - spec.dropout_p)
        O[s:s + ROW_CHUNK] = Pt @ v
    return O, lse


def _row_stats(spec, b, h, q, k, v, do, r, cols):
    """P, Z, dP and D for query rows r (all keys)."""
    S = spec.tau * (q[r] @ k.T)
    P, lse = _softmax_rows(S, visible(spec, b, r, cols))
    Z = keep(spec, b, h, r, cols)
    dPt = do[r] @ v.T
    dP = Z * dPt / (1.0 - spec.dropout_p)
    D = (P * dP).sum(axis=1)
    return P, Z, dP, D, lse


def head_backward(spec: Spec, b, h, q, k, v, do, rows=None, cols=None):
    """Gradients of one head.

    Returns a dict with ``dq`` for query ``rows`` (default all), ``dk``/``dv``
    for key ``cols`` (default all), and ``D`` / ``lse`` (D_i = sum_j P_ij
    dP_ij) for every row that the requested outputs depend on (NaN elsewhere).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N, d = q.shape
    tau = spec.tau
    allc = np.arange(N)
    rows = allc if rows is None else np.asarray(rows, dtype=np.int64)
    cols = allc if cols is None else np.asarray(cols, dtype=np.int64)
    # D_i and LSE_i for every row that sees one of ``cols`` or is in ``rows``
    # (any other row has P = 0 against the selected columns and contributes
    # nothing to them); NaN marks rows that were not needed.
    need = np.zeros(N, dtype=bool)
    need[rows] = True
    for s in range(0, N, ROW_CHUNK):
        r = allc[s:s + ROW_CHUNK]
        need[r] |= visible(spec, b, r, cols).any(axis=1)
    D = np.full(N, np.nan)
    lse = np.full(N, np.nan)
    nr = allc[need]
    for s in range(0, nr.size, ROW_CHUNK):
        r = nr[s:s + ROW_CHUNK]
        _, _, _, D[r], lse[r] = _row_stats(spec, b, h, q, k, v, do, r, allc)
    # dQ rows: dQ_i = tau sum_j dS_ij K_j with dS = P o (dP - D).
    dq = np.zeros((rows.size, d))
    for s in range(0, rows.size, ROW_CHUNK):
        r = rows[s:s + ROW_CHUNK]
        P, Z, dP, Dr, _ = _row_stats(spec, b, h, q, k, v, do, r, allc)
        dS = P * (dP - Dr[:, None])
        dq[s:s + ROW_CHUNK] = tau * (dS @ k)
    # dK, dV columns: sums over every row i.
    dk = np.zeros((cols.size, d))
    dv = np.zeros((cols.size, d))
    for s in range(0, nr.size, ROW_CHUNK):
        r = nr[s:s + ROW_CHUNK]
        vis = visible(spec, b, r, cols)
        S = tau * (q[r] @ k[cols].T)
        lr = lse[r][:, None]
        P = np.where(vis & np.isfinite(lr), np.exp(np.where(vis, S, 0.0) - np.where(np.isfinite(lr), lr, 0.0)), 0.0)
        Z = keep(spec, b, h, r, cols)
        Pt = Z * P / (1.0 - spec.dropout_p)
        dv += Pt.T @ do[r]
        dP = Z * (do[r] @ v[cols].T) / (1.0 - spec.dropout_p)
        dS = P * (dP - D[r][:, None])
        dk += tau * (dS.T @ q[r])
    return dict(dq=dq, dk=dk, dv=dv, D=D, lse=lse)


def attention_fwd(spec: Spec, q, k, v):
    """O [B,H,N,d] and LSE [B,H,N] for the whole problem (k, v: [B,H_kv,N,d])."""
    O = np.zeros((spec.B, spec.H, spec.N, spec.d))
    L = np.zeros((spec.B, spec.H, spec.N))
    g = spec.group
    for b in range(spec.B):
        for h in range(spec.H):
            O[b, h], L[b, h] = head_forward(spec, b, h, q[b, h], k[b, h // g], v[b, h // g])
    return O, L


def attention_bwd(spec: Spec, q, k, v, do):
    """dQ [B,H,N,d], dK and dV [B,H_kv,N,d] and D [B,H,N] for the whole problem.

    The gradient of a K/V head shared by g query heads sums their contributions.
    """
    shp = (spec.B, spec.H, spec.N, spec.d)
    dq = np.zeros(shp)
    dk = np.zeros((spec.B, spec.hkv, spec.N, spec.d))
    dv = np.zeros_like(dk)
    D = np.zeros(shp[:3])
    g = spec.group
    for b in range(spec.B):
        for h in range(spec.H):
            r = head_backward(spec, b, h, q[b, h], k[b, h // g], v[b, h // g], do[b, h])
            dq[b, h], D[b, h] = r["dq"], r["D"]
            dk[b, h // g] += r["dk"]
            dv[b, h // g] += r["dv"]
    return dq, dk, dv, D
