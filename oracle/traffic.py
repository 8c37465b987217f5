"""Instrumented HBM traffic counts of the naive and tiled attention algorithms.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

The pages account HBM traffic in elements read and written (lynx-cortex,
sections "El algoritmo naive de attention" and "Bytes movidos por Flash";
tonho.wtf, "como funciona", the Theta(N^2 d^2 / M) count).  Rather than retype
their closed forms, this module *executes* each algorithm on real data and
counts every element that crosses the HBM boundary:

* ``naive_counts``: step 1 reads Q, K and writes S; step 2 reads S and writes
  P; step 3 reads P, V (and writes O, which the page leaves out of its total
  because both algorithms write it; reported separately here).
* ``tiled_counts``: runs one of ``oracle.tiled.VARIANTS`` with a counter.

Pinned by tests/test_oracle_traffic.py against the page's worked numbers
(tests/golden/roofline_byte_accounting.json) and the M-scaling of the
KV-outer order.
"""
from __future__ import annotations

import numpy as np

from . import tiled as _tiled


class Counter:
    def __init__(self):
        self.reads = 0
        self.writes = 0

    def read(self, n):
        self.reads += int(n)

    def write(self, n):
        self.writes += int(n)

    @property
    def total(self):
        return self.reads + self.writes


def naive_counts(q, k, v):
    """Run standard attention step by step, counting HBM element traffic.

    Returns (counter_without_O, o_write_elements, O).
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    N, d = q.shape
    c = Counter()
    # step 1: S = Q K^T / sqrt(d), written to HBM
    c.read(q.size)
    c.read(k.size)
    S = (q @ k.T) / np.sqrt(d)
    c.write(S.size)
    # step 2: P = softmax_rowwise(S), read back and written to HBM
    c.read(S.size)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    P = E / E.sum(axis=1, keepdims=True)
    c.write(P.size)
    # step 3: O = P V
    c.read(P.size)
    c.read(v.size)
    O = P @ v
    return c, O.size, O


def tiled_counts(variant, q, k, v, Br, Bc):
    c = Counter()
    out = _tiled.VARIANTS[variant](q, k, v, Br, Bc, hbm=c)
    return c, out
