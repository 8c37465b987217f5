"""Pins for oracle.traffic against the pages' HBM byte accounting."""
import json
import os

import numpy as np

from oracle import traffic

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "roofline_byte_accounting.json")))
MiB = 2.0 ** 20


def _qkv(N, d):
    rng = np.random.default_rng(0)
    return [rng.standard_normal((N, d)) for _ in range(3)]


def test_naive_count_matches_worked_numbers():
    N, d, e = GOLD["N"], GOLD["d"], GOLD["bytes_per_element"]
    q, k, v = _qkv(N, d)
    c, o_elems, O = traffic.naive_counts(q, k, v)
    assert o_elems == N * d
    total_b = c.total * e
    assert total_b == 68_681_728
    nn_part = (c.total - 3 * q.size) * e            # S and P traffic only
    assert nn_part / MiB == GOLD["page_naive_NxN_part_MiB"]
    assert round((3 * q.size * e) / 1e6, 1) == GOLD["page_naive_Nd_part_M"]
    assert abs(total_b / MiB - GOLD["page_naive_total_MiB"]) <= 0.1 + 1e-9


def test_q_outer_flash_count_matches_worked_numbers():
    N, d, e, Br = GOLD["N"], GOLD["d"], GOLD["bytes_per_element"], GOLD["B_r"]
    q, k, v = _qkv(N, d)
    c, _ = traffic.tiled_counts("q_outer_deferred", q, k, v, Br=Br, Bc=64)
    assert c.total * e == 34_603_008
    assert round(c.total * e / MiB) == GOLD["page_flash_total_MiB"]
    cn, _, _ = traffic.naive_counts(q, k, v)
    assert round(cn.total / c.total) == GOLD["page_ratio"]


def test_kv_outer_dominant_term_halves_when_sram_doubles():
    # tonho.wtf, "como funciona": Theta(N^2 d^2 / M) with B_c = ceil(M / 4d),
    # B_r = min(ceil(M / 4d), d).
    N, d = 1024, 16
    q, k, v = _qkv(N, d)
    tot = []
    for M in (1024, 2048, 4096):
        Bc = -(-M // (4 * d))
        Br = min(Bc, d)
        c, _ = traffic.tiled_counts("kv_outer_normalised", q, k, v, Br=Br, Bc=Bc)
        tot.append(c.total - 2 * N * d)   # minus the single read of K and V
    assert abs(tot[0] / tot[1] - 2.0) < 1e-9
    assert abs(tot[1] / tot[2] - 2.0) < 1e-9
