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
    assert P.group_budgets([2, 5, 3, 4, 7, 1, 1, 1], 4) == [5, 5, 5, 5, 7, 7, 7, 7]
    assert P.group_budgets([3, 9, 2], 1) == [3, 9, 2]
    assert P.group_budgets([4, 2, 6, 6], 2) == [4, 4, 6, 6]


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
    budgets = P.group_budgets([3, 6, 2, 4, 5, 5, 8, 2], G)
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
    budgets = P.group_budgets([2, 9, 4, 3, 6, 6, 2, 16], G)
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
