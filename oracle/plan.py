"""Oracle: per-head budgets (Max-Min shifting) and work schedules (LPT, naive).

Test infrastructure only (see the package docstring).  Integer arithmetic in
Python ints, written step by step as the pages describe it.

Budget unit (a reading; the pages speak of a "token budget"): k_h is the number
of KV blocks kept per query-block row, capped at the row's causal block count
i+1, with the two mandatory blocks (sink block 0 and the diagonal block i)
counted inside it.
"""
from __future__ import annotations

import heapq

import numpy as np


def causal_blocks(nb: int) -> int:
    """Number of (i, j) block pairs with j <= i in an nb x nb causal grid."""
    return nb * (nb + 1) // 2


def kept_blocks(k: int, nb: int) -> int:
    """Blocks kept over all rows when every row i keeps min(k, i+1) blocks."""
    return int(np.minimum(k, np.arange(1, nb + 1)).sum())


def density(k: int, nb: int) -> float:
    """Fraction of causal blocks kept by a per-row budget of k blocks."""
    return kept_blocks(k, nb) / causal_blocks(nb)


def density_table(nb: int) -> np.ndarray:
    """density(k, nb) for k = 1..nb (entry k-1)."""
    rows = np.arange(1, nb + 1)
    kept = np.minimum(rows[:, None], rows[None, :]).sum(axis=1)   # k along axis 0
    return kept / causal_blocks(nb)


def budget_for_density(target: float, nb: int) -> int:
    """The k in [1, nb] whose density is nearest the target; ties -> smaller k.

    This is how "X% of causal blocks" becomes an integer per-row budget (a
    reading: the pages give budgets only as fractions).
    """
    err = np.abs(density_table(nb) - target)
    return int(np.argmin(err)) + 1          # argmin takes the first (smaller k)


def maxmin_shift(k_uniform: int, demand: list[int], k_min: int, nb: int) -> list[int]:
    """Max-Min budget shifting (S-HPLB, "Strategia Max-Min (Budget Shifting)";
    Chinese summary 2.1 "最大-最小预算迁移策略").

    Every head starts at the uniform budget.  Budget then moves, one block at a
    time, from the head with the most budget to spare relative to its demand
    (a high-sparsity head) to the head that is shortest of its demand (a
    low-sparsity head); the total never changes.  Reading of the stopping
    rule: the donor is argmax_h (k_h - d_h) over heads above k_min, the
    receiver argmin_h (k_h - d_h) over heads below nb, ties to the lowest h;
    stop once the donor's surplus exceeds the receiver's by at most one.  The
    result maximises min_h (k_h - d_h) with surpluses levelled to within one.
    """
    H = len(demand)
    k = [k_uniform] * H
    while True:
        surplus = [k[h] - demand[h] for h in range(H)]
        donor = -1
        for h in range(H):
            if k[h] > k_min and (donor < 0 or surplus[h] > surplus[donor]):
                donor = h
        receiver = -1
        for h in range(H):
            if k[h] < nb and (receiver < 0 or surplus[h] < surplus[receiver]):
                receiver = h
        if donor < 0 or receiver < 0:
            break
        if surplus[donor] - surplus[receiver] <= 1:
            break
        k[donor] -= 1
        k[receiver] += 1
    return k


def group_budgets(k_uniform: int, demand: list[int], group: int, k_min: int,
                  nb: int) -> list[int]:
    """Budgets when the G query heads of a KV group share one block list.

    Fluxion models access at the level of the GQA group ("Riepilogo Tecnico:
    Fluxion", "Componenti di Sistema", "Selettore Granularità-Budget"; one KV
    block fetched serves every query head of its group).  Reading: the group
    is the unit the budget is shifted between.  Its demand is that of its most
    demanding head (the shared list has to cover that head), and Max-Min
    shifting runs over the groups from the uniform budget, so the groups'
    total stays Hkv * k_uniform and the heads' total Hq * k_uniform, as with
    per-head budgets.  Returned per query head (equal within a group).
    """
    H = len(demand)
    g_demand = [max(demand[g * group:(g + 1) * group]) for g in range(H // group)]
    k_g = maxmin_shift(k_uniform, g_demand, k_min, nb)
    return [k_g[h // group] for h in range(H)]


def item_costs(budgets: list[int], nb: int) -> list[int]:
    """Cost of work item (h, i), id h*nb+i: the blocks it attends, min(k_h, i+1).

    Reading: the pages balance by the per-head budget; on one GPU the work unit
    is a (head, query-block) item whose budget in blocks is capped by
    causality.
    """
    costs = []
    for h in range(len(budgets)):
        for i in range(nb):
            costs.append(min(budgets[h], i + 1))
    return costs


def lpt_assign(order: list[int], costs: list[int], workers: int):
    """Greedy longest-first assignment (S-HPLB "Algoritmo Greedy"; Chinese
    summary 2.2 "贪心启发式算法"): walk the items in the given order and give
    each to the currently least-loaded worker (ties: lowest worker id)."""
    heap = [(0, w) for w in range(workers)]
    lists = [[] for _ in range(workers)]
    loads = [0] * workers
    for item in order:
        load, w = heapq.heappop(heap)
        lists[w].append(item)
        loads[w] = load + costs[item]
        heapq.heappush(heap, (loads[w], w))
    return lists, loads


def schedule(budgets: list[int], nb: int, workers: int, policy: str, group: int = 1):
    """Work lists of (head, query-block) items for ``workers`` persistent workers.

    policy:
      "lpt"         items sorted by cost, descending (ties: lower item id), then
                    greedy least-loaded assignment -- the pages' heuristic.
      "lpt_grouped" the same greedy, but items are walked KV group by KV group
                    (g = h // group ascending; within a group cost descending,
                    ties by query block i, then head).  Each worker then runs
                    its items by (g, i, head): the assignment and the loads
                    are the greedy's, and all workers sweep a group's query
                    blocks together, its heads side by side.
      "head_order"  the naive baseline of the Chinese summary ("电脑 1 拿头
                    1-4"): items in id order cut into W contiguous chunks of
                    equal count; chunk w is [w*N//W, (w+1)*N//W).
    Returns (wptr, items, loads): CSR offsets [W+1], item ids in each worker's
    processing order, and per-worker total cost.
    """
    costs = item_costs(budgets, nb)
    n = len(costs)
    if policy == "head_order":
        lists = []
        for w in range(workers):
            lists.append(list(range(w * n // workers, (w + 1) * n // workers)))
        loads = [sum(costs[x] for x in lst) for lst in lists]
    elif policy == "lpt":
        order = sorted(range(n), key=lambda x: (-costs[x], x))
        lists, loads = lpt_assign(order, costs, workers)
    elif policy == "lpt_grouped":
        order = sorted(range(n), key=lambda x: ((x // nb) // group, -costs[x], x % nb, x // nb))
        lists, loads = lpt_assign(order, costs, workers)
        lists = [sorted(lst, key=lambda x: ((x // nb) // group, x % nb, x // nb))
                 for lst in lists]
    else:
        raise ValueError(policy)
    wptr = [0]
    items = []
    for lst in lists:
        items.extend(lst)
        wptr.append(len(items))
    return wptr, items, loads


def pair_schedule(budgets: list[int], nb: int, workers: int, policy: str, group: int):
    """Schedule of a group-shared plan whose KV groups have an even number of
    query heads: the heads 2p and 2p+1 share their block list, so the work
    item is (pair p, query block i), id p*nb + i, and one K/V block load
    serves both.  Reading: the greedy of ``schedule`` runs on the pairs'
    budgets with group/2 pairs per KV group; an item costs both heads'
    blocks, 2 * min(k_p, i+1), so loads count head-blocks as per-head plans
    do (the factor changes no decision of the greedy).
    """
    pair_budgets = [budgets[2 * x] for x in range(len(budgets) // 2)]
    wptr, items, loads = schedule(pair_budgets, nb, workers, policy, group // 2)
    return wptr, items, [2 * x for x in loads]


def schedule_from_costs(costs: list[int], workers: int, within: str = "assignment"):
    """LPT over given item costs (e.g. the block counts a data-dependent
    selection produced): items by cost descending, ties lower id, each to the
    least-loaded worker.  Each worker's list is in assignment order, or with
    within="item" in ascending item id.  Returns (wptr, items, loads) as
    schedule()."""
    order = sorted(range(len(costs)), key=lambda x: (-costs[x], x))
    lists, loads = lpt_assign(order, costs, workers)
    if within == "item":
        lists = [sorted(lst) for lst in lists]
    elif within != "assignment":
        raise ValueError(within)
    wptr = [0]
    items = []
    for lst in lists:
        items.extend(lst)
        wptr.append(len(items))
    return wptr, items, loads


def makespan(loads: list[int]) -> int:
    return max(loads) if loads else 0
