"""Pins for the oracle's budget and schedule code (no GPU).

Each check compares the oracle with something other than itself: a
hand-worked example, a closed form, brute-force enumeration, or Graham's
bound for longest-first scheduling.
"""
import itertools
import json
import os
import random

import pytest

from oracle import plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("nb", [1, 2, 7, 64, 256, 1024])
def test_kept_blocks_closed_form(nb):
    # sum_i min(k, i+1) = k(k+1)/2 + k(nb-k) for 1 <= k <= nb
    for k in sorted(x for x in {1, 2, 3, nb // 2 or 1, nb} if x <= nb):
        assert plan.kept_blocks(k, nb) == k * (k + 1) // 2 + k * (nb - k)
    assert plan.kept_blocks(nb, nb) == plan.causal_blocks(nb)


def test_budget_for_density_nearest():
    for nb, target in [(64, 0.25), (256, 0.10), (1024, 0.06), (100, 0.5)]:
        k = plan.budget_for_density(target, nb)
        # closed-form densities of the neighbours are no nearer
        def dens(kk):
            return (kk * (kk + 1) / 2 + kk * (nb - kk)) / (nb * (nb + 1) / 2)
        err = abs(dens(k) - target)
        for kk in range(1, nb + 1):
            assert abs(dens(kk) - target) >= err - 1e-15
            if abs(dens(kk) - target) == err:
                assert kk >= k
    # the uniform budgets of the prefill workloads
    assert plan.budget_for_density(0.25, 64) == 9
    assert plan.budget_for_density(0.10, 256) == 13
    assert plan.budget_for_density(0.06, 1024) == 31


def test_maxmin_hand_example():
    g = _golden("maxmin_hand.json")
    got = plan.maxmin_shift(g["k_uniform"], g["demand"], g["k_min"], g["nb"])
    assert got == g["budgets"]


def test_maxmin_equal_demands_unchanged():
    assert plan.maxmin_shift(7, [5] * 6, 2, 50) == [7] * 6
    assert plan.maxmin_shift(7, [30] * 3, 2, 50) == [7] * 3


def _brute_force_maxmin_value(k_uniform, demand, k_min, nb):
    H = len(demand)
    total = k_uniform * H
    best = None
    for ks in itertools.product(range(k_min, nb + 1), repeat=H):
        if sum(ks) != total:
            continue
        v = min(k - d for k, d in zip(ks, demand))
        best = v if best is None else max(best, v)
    return best


@pytest.mark.parametrize("seed", range(40))
def test_maxmin_brute_force(seed):
    r = random.Random(seed)
    H = r.randint(1, 4)
    nb = r.randint(2, 9)
    k_min = r.randint(1, 2)
    k_uniform = r.randint(k_min, nb)
    demand = [r.randint(1, nb) for _ in range(H)]
    got = plan.maxmin_shift(k_uniform, demand, k_min, nb)
    # conservation of the total and the bounds
    assert sum(got) == k_uniform * H
    assert all(k_min <= k <= nb for k in got)
    # the max-min objective equals brute-force enumeration
    assert min(k - d for k, d in zip(got, demand)) == \
        _brute_force_maxmin_value(k_uniform, demand, k_min, nb)


@pytest.mark.parametrize("seed", range(20))
def test_maxmin_monotone_and_levelled(seed):
    r = random.Random(100 + seed)
    H = r.randint(2, 64)
    nb = r.randint(16, 1024)
    k_min = 2
    k_uniform = r.randint(k_min, max(k_min, nb // 8))
    demand = [r.randint(1, nb) for _ in range(H)]
    got = plan.maxmin_shift(k_uniform, demand, k_min, nb)
    assert sum(got) == k_uniform * H
    for h in range(H):
        for g in range(H):
            if demand[h] > demand[g]:
                assert got[h] >= got[g]
    free = [k - d for k, d in zip(got, demand) if k_min < k < nb]
    if free:
        assert max(free) - min(free) <= 1


def test_lpt_hand_example():
    g = _golden("lpt_hand.json")
    wptr, items, loads = plan.schedule(g["budgets"], g["nb"], g["workers"], g["policy"])
    assert wptr == g["wptr"] and items == g["items"] and loads == g["loads"]


def _brute_force_opt(costs, W):
    best = None
    for assign in itertools.product(range(W), repeat=len(costs)):
        loads = [0] * W
        for c, w in zip(costs, assign):
            loads[w] += c
        m = max(loads)
        best = m if best is None else min(best, m)
    return best


@pytest.mark.parametrize("seed", range(30))
def test_lpt_graham_bound(seed):
    r = random.Random(seed)
    N = r.randint(1, 10)
    W = r.randint(1, 3)
    costs = [r.randint(1, 20) for _ in range(N)]
    order = sorted(range(N), key=lambda x: (-costs[x], x))
    lists, loads = plan.lpt_assign(order, costs, W)
    opt = _brute_force_opt(costs, W)
    # Graham (1969): LPT <= (4/3 - 1/(3W)) OPT
    assert max(loads) * 3 * W <= (4 * W - 1) * opt
    assert max(loads) >= max(max(costs), -(-sum(costs) // W))


@pytest.mark.parametrize("policy", ["lpt", "lpt_grouped", "head_order"])
def test_schedule_is_a_partition(policy):
    r = random.Random(7)
    H, nb, W, G = 8, 33, 5, 4
    budgets = [r.randint(2, nb) for _ in range(H)]
    wptr, items, loads = plan.schedule(budgets, nb, W, policy, G)
    assert len(wptr) == W + 1 and wptr[0] == 0 and wptr[-1] == H * nb
    assert sorted(items) == list(range(H * nb))
    costs = plan.item_costs(budgets, nb)
    for w in range(W):
        lst = items[wptr[w]:wptr[w + 1]]
        assert loads[w] == sum(costs[x] for x in lst)
        if policy == "head_order":
            assert lst == list(range(w * H * nb // W, (w + 1) * H * nb // W))
        if policy == "lpt_grouped":
            groups = [(x // nb) // G for x in lst]
            assert groups == sorted(groups)
    assert sum(loads) == sum(costs)


def test_lpt_grouped_assignment_and_run_order_by_hand():
    # two KV groups of two heads, two workers.  The greedy walks group 0 by
    # cost descending, ties by query block then head, each item to the
    # least-loaded worker (ties: the lower one); then group 1 from those
    # loads.  Each worker then runs its items by (group, query block, head).
    nb, G = 4, 2
    budgets = [3, 3, 2, 3]
    # costs: head 0 and 1: 1 2 3 3; head 2: 1 2 2 2; head 3: 1 2 3 3
    # group 0 walk: (0,2)3 (1,2)3 (0,3)3 (1,3)3 (0,1)2 (1,1)2 (0,0)1 (1,0)1
    #   w0: (0,2) [3] (0,3) [6] (0,1) [8] (0,0) [9]
    #   w1: (1,2) [3] (1,3) [6] (1,1) [8] (1,0) [9]
    # group 1 walk: (3,2)3 (3,3)3 (2,1)2 (3,1)2 (2,2)2 (2,3)2 (2,0)1 (3,0)1
    #   w0: (3,2) [12] (2,1) [14] (2,2) [16] (2,0) [17]
    #   w1: (3,3) [12] (3,1) [14] (2,3) [16] (3,0) [17]
    wptr, items, loads = plan.schedule(budgets, nb, 2, "lpt_grouped", G)
    assert wptr == [0, 8, 16] and loads == [17, 17]
    hi = [(x // nb, x % nb) for x in items]
    assert hi[:8] == [(0, 0), (0, 1), (0, 2), (0, 3), (2, 0), (2, 1), (2, 2), (3, 2)]
    assert hi[8:] == [(1, 0), (1, 1), (1, 2), (1, 3), (3, 0), (3, 1), (2, 3), (3, 3)]


def test_lpt_grouped_runs_a_groups_query_blocks_together():
    # every worker runs its items by group, query block, head
    r = random.Random(11)
    H, nb, W, G = 8, 40, 3, 4
    budgets = [r.randint(2, nb) for _ in range(H)]
    wptr, items, loads = plan.schedule(budgets, nb, W, "lpt_grouped", G)
    for w in range(W):
        lst = items[wptr[w]:wptr[w + 1]]
        keys = [((x // nb) // G, x % nb, x // nb) for x in lst]
        assert keys == sorted(keys)
    # the loads are the greedy's over the grouped walk
    costs = plan.item_costs(budgets, nb)
    order = sorted(range(H * nb), key=lambda x: ((x // nb) // G, -costs[x], x % nb, x // nb))
    lists, want = plan.lpt_assign(order, costs, W)
    assert loads == want
    assert [sorted(items[wptr[w]:wptr[w + 1]]) for w in range(W)] == [sorted(l) for l in lists]


def test_lpt_balances_better_than_head_order():
    r = random.Random(3)
    H, nb, W = 32, 256, 152
    budgets = [r.randint(2, 60) for _ in range(H)]
    _, _, l_lpt = plan.schedule(budgets, nb, W, "lpt")
    _, _, l_naive = plan.schedule(budgets, nb, W, "head_order")
    costs = plan.item_costs(budgets, nb)
    lower = max(max(costs), -(-sum(costs) // W))
    assert max(l_lpt) <= lower + max(costs)
    assert max(l_lpt) < max(l_naive)
