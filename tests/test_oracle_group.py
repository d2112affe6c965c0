"""Pins for the oracle's group-shared selection (one block list per KV group).

Checked against what fixes it independently of its own formula: the identity
between averaging the heads' scores and scoring the averaged pooled query, the
reduction to per-head selection when G = 1 or when a group's heads agree, a
brute-force search over all valid block sets on tiny rows, and the budget rule
on a hand example.
"""
import itertools

import numpy as np

from oracle import attention as A
from oracle import plan as P


def test_group_budgets_hand_example():
    # groups demand [5, 4]: levelled at once, every head keeps 4
    assert P.group_budgets(4, [2, 5, 3, 4], 2, 2, 8) == [4, 4, 4, 4]
    # groups demand [7, 2]: the second gives until it reaches k_min (4->3->2)
    assert P.group_budgets(4, [1, 7, 2, 2], 2, 2, 8) == [6, 6, 2, 2]
    # a group's demand is its most demanding head's, not the sum or mean
    assert P.group_budgets(5, [9, 1, 1, 1, 2, 2, 2, 2], 4, 2, 16) == [8] * 4 + [2] * 4


def test_group_budgets_of_groups_of_one_are_the_per_head_budgets():
    r = np.random.default_rng(21)
    for _ in range(20):
        H, nb = int(r.integers(1, 9)), int(r.integers(4, 40))
        k_u = int(r.integers(2, nb + 1))
        demand = r.integers(0, nb + 1, H).tolist()
        assert P.group_budgets(k_u, demand, 1, 2, nb) == P.maxmin_shift(k_u, demand, 2, nb)


def test_group_budgets_conserve_the_total_and_follow_demand():
    r = np.random.default_rng(22)
    for _ in range(30):
        Hkv, G, nb = int(r.integers(1, 6)), int(r.choice([2, 4, 7])), int(r.integers(8, 64))
        k_u = int(r.integers(2, nb // 2 + 1))
        demand = r.integers(0, nb + 1, Hkv * G).tolist()
        k = P.group_budgets(k_u, demand, G, 2, nb)
        assert sum(k) == Hkv * G * k_u                       # conserved, as per head
        assert all(len(set(k[g * G:(g + 1) * G])) == 1 for g in range(Hkv))
        gd = [max(demand[g * G:(g + 1) * G]) for g in range(Hkv)]
        for a in range(Hkv):
            for b in range(Hkv):
                if gd[a] > gd[b]:
                    assert k[a * G] >= k[b * G]


def test_group_scores_equal_scores_of_the_mean_pooled_query():
    # mean_h (qbar_h . kbar) == (mean_h qbar_h) . kbar: the two routes share no code
    r = np.random.default_rng(11)
    Hq, G, nb, d = 6, 3, 9, 16
    qbar = r.standard_normal((Hq, nb, d))
    kbar = r.standard_normal((Hq // G, nb, d))
    per_head = A.block_scores(qbar, kbar, G)
    got = A.group_scores(per_head, G)
    qmean = qbar.reshape(Hq // G, G, nb, d).mean(axis=1)
    want = A.block_scores(qmean, kbar, 1)
    finite = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), finite)
    assert np.allclose(got[finite], want[finite], rtol=1e-12, atol=1e-12)


def test_grouped_selection_with_group_of_one_is_per_head_selection():
    r = np.random.default_rng(12)
    Hq, nb = 4, 12
    scores = np.tril(r.standard_normal((Hq, nb, nb))) + np.triu(np.full((nb, nb), -np.inf), 1)
    budgets = [2, 5, 7, 12]
    a = A.select_all(scores, budgets, 12)
    b = A.select_all_grouped(scores, budgets, 1, 12)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_grouped_selection_when_heads_agree_is_per_head_selection():
    r = np.random.default_rng(13)
    Hkv, G, nb = 2, 4, 10
    base = np.tril(r.standard_normal((Hkv, nb, nb))) + np.triu(np.full((nb, nb), -np.inf), 1)
    scores = np.repeat(base, G, axis=0)          # the G heads of a group have equal scores
    budgets = P.group_budgets(4, [3, 6, 2, 4, 5, 5, 8, 2], G, 2, nb)
    a = A.select_all(scores, budgets, nb)
    b = A.select_all_grouped(scores, budgets, G, nb)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_grouped_selection_is_the_best_valid_set_for_the_group():
    # the shared list maximises the group's summed score among all valid sets
    r = np.random.default_rng(14)
    G = 3
    for _ in range(15):
        i = int(r.integers(2, 9))
        nb = i + 1
        k = int(r.integers(2, i + 2))
        scores = np.full((G, nb, nb), -np.inf)
        scores[:, i, :i + 1] = r.standard_normal((G, i + 1))
        idx, cnt = A.select_all_grouped(scores, [k] * G, G, nb)
        keep = min(k, i + 1)
        total = scores[:, i, :].sum(axis=0)
        best = max(itertools.combinations(range(1, i), keep - 2),
                   key=lambda c: sum(total[j] for j in c))
        want = sorted({0, i} | set(best))
        for h in range(G):
            assert list(idx[h, i, :cnt[h, i]]) == want


def test_grouped_lists_are_shared_and_well_formed():
    r = np.random.default_rng(15)
    Hq, G, nb = 8, 4, 16
    scores = np.tril(r.standard_normal((Hq, nb, nb))) + np.triu(np.full((nb, nb), -np.inf), 1)
    budgets = P.group_budgets(6, [2, 9, 4, 3, 6, 6, 2, 16], G, 2, 16)
    kmax = max(budgets)
    idx, cnt = A.select_all_grouped(scores, budgets, G, kmax)
    for h in range(Hq):
        g = h // G
        for i in range(nb):
            n = cnt[h, i]
            assert n == min(budgets[h], i + 1)
            sel = list(idx[h, i, :n])
            assert sel == sorted(set(sel)) and 0 in sel and i in sel
            assert list(idx[g * G, i, :n]) == sel
            assert np.all(idx[h, i, n:] == -1)
