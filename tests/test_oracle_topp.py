"""Pins for the oracle's top-p block selection and LPT over given costs.

Checked against closed forms (uniform and two-block softmax), the limiting
thresholds, a brute-force search over all block sets on tiny rows, and the
reduction of LPT-over-costs to the budget-based LPT schedule.
"""
import itertools
import math

import numpy as np

from oracle import attention as A
from oracle import plan as P


def test_block_probabilities_closed_forms():
    assert np.allclose(A.block_probabilities(np.zeros(9), 8), np.full(9, 1 / 9))
    d = 1.7
    pr = A.block_probabilities(np.array([0.0, d, 5.0]), 1)      # entries past i ignored
    assert abs(pr[1] - math.exp(d) / (1 + math.exp(d))) < 1e-15
    assert abs(pr.sum() - 1.0) < 1e-15


def test_topp_limits():
    r = np.random.default_rng(21)
    for i in range(0, 12):
        s = r.standard_normal(i + 1)
        assert A.select_row_topp(s, i, 1.0) == list(range(i + 1)) or i == 0
        assert A.select_row_topp(s, i, 0.0) == sorted({0, i})
    # a threshold the mandatory blocks already reach keeps only them
    s = np.array([9.0, 0.0, 0.0, 0.0, 9.0])
    assert A.select_row_topp(s, 4, 0.99) == [0, 4]


def test_topp_is_the_smallest_set_reaching_p_with_the_most_mass():
    r = np.random.default_rng(22)
    for _ in range(40):
        i = int(r.integers(2, 9))
        s = r.standard_normal(i + 1) * 2.0
        p = float(r.uniform(0.2, 0.999))
        prob = A.block_probabilities(s, i)
        got = A.select_row_topp(s, i, p)
        mand = sorted({0, i})
        best = None
        for n in range(0, i):
            for c in itertools.combinations(range(1, i), n):
                sel = mand + list(c)
                mass = prob[sel].sum()
                if mass >= p - 1e-15:
                    if best is None or len(sel) < len(best[0]) or (
                            len(sel) == len(best[0]) and mass > best[1] + 1e-15):
                        best = (sel, mass)
            if best is not None and len(best[0]) == n + len(mand):
                break
        assert best is not None
        assert len(got) == len(best[0])
        assert abs(prob[got].sum() - best[1]) < 1e-12


def test_topp_rows_are_well_formed():
    r = np.random.default_rng(23)
    Hq, nb = 3, 20
    scores = np.tril(r.standard_normal((Hq, nb, nb))) + np.triu(np.full((nb, nb), -np.inf), 1)
    idx, cnt = A.select_all_topp(scores, 0.7, nb)
    for h in range(Hq):
        for i in range(nb):
            sel = list(idx[h, i, :cnt[h, i]])
            assert sel == sorted(set(sel)) and 0 in sel and i in sel
            assert A.block_probabilities(scores[h, i], i)[sel].sum() >= 0.7 or cnt[h, i] == i + 1
            assert np.all(idx[h, i, cnt[h, i]:] == -1)


def test_lpt_over_costs_reduces_to_the_budget_schedule():
    r = np.random.default_rng(24)
    for _ in range(10):
        nb = int(r.integers(2, 30))
        budgets = [int(x) for x in r.integers(2, nb + 1, int(r.integers(1, 6)))]
        W = int(r.integers(1, 12))
        costs = P.item_costs(budgets, nb)
        assert P.schedule_from_costs(costs, W) == P.schedule(budgets, nb, W, "lpt")


def test_lpt_over_costs_is_a_partition_within_grahams_bound():
    r = np.random.default_rng(25)
    for _ in range(10):
        costs = [int(x) for x in r.integers(1, 50, int(r.integers(1, 9)))]
        W = int(r.integers(1, 4))
        wptr, items, loads = P.schedule_from_costs(costs, W)
        assert sorted(items) == list(range(len(costs)))
        for w in range(W):
            assert loads[w] == sum(costs[x] for x in items[wptr[w]:wptr[w + 1]])
        opt = min(max(sum(costs[x] for x in range(len(costs)) if a[x] == w) for w in range(W))
                  for a in itertools.product(range(W), repeat=len(costs)))
        assert max(loads) <= (4 / 3 - 1 / (3 * W)) * opt + 1e-9


def test_item_order_keeps_each_workers_set_and_sorts_it():
    r = np.random.default_rng(26)
    costs = [int(x) for x in r.integers(0, 40, 200)]
    a_wptr, a_items, a_loads = P.schedule_from_costs(costs, 7)
    i_wptr, i_items, i_loads = P.schedule_from_costs(costs, 7, within="item")
    assert a_wptr == i_wptr and a_loads == i_loads
    for w in range(7):
        lst = i_items[i_wptr[w]:i_wptr[w + 1]]
        assert lst == sorted(a_items[a_wptr[w]:a_wptr[w + 1]])
