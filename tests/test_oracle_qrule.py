"""Pins for oracle.qrule: the integer miss split and the fraction forms."""
import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import qrule as Q


def brute_force_q(m, f_q16):
    """Exhaustive argmin over q in [1, m] of the Q16 exposed-time cost
    max(q*(1-f), (m-q)*f), smallest q on ties (no neighbour shortcut)."""
    best, best_q = None, None
    for q in range(1, m + 1):
        c = max(q * (65536 - f_q16), (m - q) * f_q16)
        if best is None or c < best:
            best, best_q = c, q
    return best_q


@pytest.mark.parametrize("row", read_golden("q_rule_worked_examples.txt"))
def test_worked_examples(row):
    m, bp, bh, q = int(row[0]), float(row[1]), float(row[2]), int(row[3])
    assert Q.q_rule(m, Q.split_from_bandwidth(bp, bh)) == q


def test_naive_rounding_loss_on_5090_desktop():
    (m, bp, bh, q_naive, q_best, loss), = read_golden("qiita_rounding_loss.txt")
    m, bp, bh = int(m), float(bp), float(bh)
    assert round(Q.q_star_continuous(m, bp, bh)) == int(q_naive)
    lat = {q: Q.exposed_latency(q, m, bp, bh) for q in range(1, m + 1)}
    assert min(lat, key=lat.get) == int(q_best)
    assert Q.q_rule(m, Q.split_from_bandwidth(bp, bh)) == int(q_best)
    got = lat[int(q_naive)] / lat[int(q_best)] - 1
    assert abs(100 * got - float(loss)) < 0.05
    assert abs((bh - bp) - 4.8) < 1e-9


def test_rule_equals_exhaustive_argmin():
    fs = sorted(set(list(range(1, 65537, 97)) + [1, 16281, 16384, 32768, 35747, 43691,
                                                 59689, 65535, 65536]))
    for m in range(1, 97):
        for f in fs:
            assert Q.q_rule(m, f) == brute_force_q(m, f), (m, f)


def test_rule_is_optimal_for_real_bandwidths():
    # [QIITA §8]: checked against brute force for m in {4, 8, 16, 32} over ratio
    # steps of 0.01.  The Q16 rounding of f may move q only where two choices are
    # within that rounding of each other.
    bp = 10.0
    for m in (4, 8, 16, 32):
        for r in np.arange(0.01, 1.0, 0.01):
            bh = bp / r
            q = Q.q_rule(m, Q.split_from_bandwidth(bp, bh))
            best = min(Q.exposed_latency(x, m, bp, bh) for x in range(1, m + 1))
            assert Q.exposed_latency(q, m, bp, bh) <= best * (1 + 1e-3), (m, r)


def test_machine_table_is_optimal():
    for name, bp, bh in read_golden("machine_bandwidths.txt"):
        bp, bh = float(bp), float(bh)
        for m in range(1, 33):
            q = Q.q_rule(m, Q.split_from_bandwidth(bp, bh))
            best = min(Q.exposed_latency(x, m, bp, bh) for x in range(1, m + 1))
            assert Q.exposed_latency(q, m, bp, bh) <= best * (1 + 1e-3), (name, m)


def test_closed_form_neighbourhood():
    # the integer q lies within one of q* = m*B_P/B_H clamped to [1, m]
    for m in range(1, 64):
        for f in (0.05, 0.25, 1 / 3, 0.5, 2 / 3, 0.91, 1.0):
            q = Q.q_rule(m, Q.f_to_q16(f))
            assert abs(q - min(m, max(1.0, m * f))) < 1.0 + 1e-9


def test_full_fraction_fills_everything_and_zero_misses():
    for m in range(0, 200):
        assert Q.q_rule(m, 65536) == m
    assert Q.q_rule(0, 12345) == 0
    # B_H <= B_P: the residual host bandwidth is zero, every miss goes to the GPU
    assert Q.split_from_bandwidth(60.0, 50.0) == 65536
    assert Q.split_from_bandwidth(50.0, 50.0) == 65536


def test_at_least_one_fill():
    for f in (1, 100, 4000, 16384):
        for m in range(1, 4):
            assert Q.q_rule(m, f) >= 1


def test_half_fraction_ties_go_low():
    # m*f = x.5 at f = 1/2 for odd m: both neighbours cost the same; the lower wins
    got = [Q.q_rule(m, 32768) for m in range(17)]
    assert got == [0, 1, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6, 7, 7, 8]


def test_overlap_form_reduces_to_bandwidth_form():
    # [BWRATIO "实测版本"]: with c_ov = B_H - B_P and p_ov = B_P the two forms agree
    for _, bp, bh in read_golden("machine_bandwidths.txt"):
        bp, bh = float(bp), float(bh)
        a = Q.split_from_overlap(bp, bh - bp)
        b = Q.split_from_bandwidth(bp, bh)
        assert abs(a - b) <= 1
    assert Q.split_from_overlap(50.0, 50.0) == Q.split_from_bandwidth(50.0, 100.0) == 32768
    assert Q.split_from_overlap(48.0, 40.0) == 35747


def test_capacity_clamp():
    assert Q.q_for_call(10, 5, 8, True, 65536) == 3
    assert Q.q_for_call(10, 8, 8, True, 65536) == 0
    assert Q.q_for_call(4, 0, 8, False, 16384) == 1
