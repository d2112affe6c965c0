"""Oracle: per-head selection granularity for decode retrieval heads, chosen
together with the budget.

Test infrastructure only (see the package docstring).

"Riepilogo Tecnico: Fluxion" ("Intuizioni Chiave" 2; the granularity-budget
selector among its system components): retrieval heads pick blocks by top-k,
the cost of picking depends on the block size, and each retrieval head gets
its own selection granularity and KV budget, chosen together to meet an error
bound with the least data movement, the movement counted per GQA group.

Readings taken here (the pages give no formula):

* A retrieval head h selects blocks of g_h tokens and keeps k_h of them: the
  sink block 0 and the last block (which holds the new token), then the best
  of the rest.  Streaming heads keep their fixed sink + window list at the
  default block size.
* Error bound: on the calibration draw, head h must keep at least the
  attention mass that the default selection (block size g0, k0 blocks) keeps.
  The mass of a selection is that of the best k blocks, mandatory ones first:
  the pooled scores that rank blocks at run time are the estimate of it.
* Data movement per decode step and sequence: the keys and values of the
  selected tokens, k_h * g_h * d * 2 bytes each (bf16), plus the pooled keys
  the scores read, (L / g) * d * 4 bytes (fp32) for each block size g used by
  the group's retrieval heads -- once per group, since its heads share the
  pooled cache of one size.
* For each KV group the heads' sizes are chosen together over all
  combinations of the candidate sizes; ties go to the first combination in
  lexicographic order of the candidates (finer sizes, lower heads first).
* choose_granularity_time charges time instead of bytes: the attention's
  K/V bytes and the scoring's pooled bytes at their measured rates, a fixed
  time per scoring pass (one per block size in use), and the selection
  kernel's time for the longest row (its candidate count).  The rates are
  inputs, measured on the device the plan is for.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

STREAMING = 1
REL_TOL = 1e-12      # masses summed over different block sizes differ in rounding


def decode_block_mass(q_row: np.ndarray, k_head: np.ndarray, g: int) -> np.ndarray:
    """Softmax weight of one decode query over all L keys, summed per block
    of g tokens: m[j] for j < L / g (sums to 1)."""
    d = q_row.shape[0]
    logits = k_head.astype(np.float64) @ q_row.astype(np.float64) / math.sqrt(d)
    p = np.exp(logits - logits.max())
    p /= p.sum()
    return p.reshape(-1, g).sum(axis=1)


def _mandatory(nb: int) -> list[int]:
    return sorted({0, nb - 1})


def _rest_by_mass(mass: np.ndarray) -> np.ndarray:
    """Blocks other than the mandatory ones, by mass descending, ties to the
    lower index."""
    nb = len(mass)
    mand = set(_mandatory(nb))
    rest = np.array([j for j in range(nb) if j not in mand], dtype=np.int64)
    if len(rest) == 0:
        return rest
    return rest[np.lexsort((rest, -mass[rest]))]


def kept_mass(mass: np.ndarray, k: int) -> float:
    """Mass of the best selection of k blocks that keeps block 0 and the last
    block: those, then the heaviest of the rest."""
    mand = _mandatory(len(mass))
    take = max(0, k - len(mand))
    return float(mass[mand].sum() + mass[_rest_by_mass(mass)[:take]].sum())


def blocks_for_mass(mass: np.ndarray, target: float) -> int:
    """Fewest blocks k (at least the mandatory ones) with kept_mass >= target."""
    mand = _mandatory(len(mass))
    acc = float(mass[mand].sum())
    k = len(mand)
    if acc >= target:
        return k
    for j in _rest_by_mass(mass):
        acc += float(mass[j])
        k += 1
        if acc >= target:
            return k
    return len(mass)


def kv_bytes(k: int, g: int, d: int) -> int:
    """Keys and values of k blocks of g tokens, bf16."""
    return k * g * d * 2 * 2


def pooled_bytes(L: int, g: int, d: int) -> int:
    """Pooled keys of one KV head at block size g, fp32."""
    return (L // g) * d * 4


def choose_granularity(masses, kinds, group: int, g0: int, k0: int, candidates, L: int,
                       d: int):
    """Per-head (g_h, k_h) for the retrieval heads, chosen per KV group.

    masses[h][g]: decode_block_mass of retrieval head h at block size g, for g
    in ``candidates`` and g0.  Returns a dict with ``gran`` and ``budget``
    ([Hq]; streaming heads get g0 and 0), the per-head ``target`` mass (that of
    the default selection) and ``kept`` mass of the choice, and the bytes per
    step of the choice and of the default, summed over the groups.
    """
    Hq = len(kinds)
    gran = [g0] * Hq
    budget = [0] * Hq
    target = [0.0] * Hq
    kept = [0.0] * Hq
    total = default = 0
    for grp in range(Hq // group):
        heads = [h for h in range(grp * group, (grp + 1) * group) if kinds[h] != STREAMING]
        if not heads:
            continue
        need = {}
        for h in heads:
            target[h] = kept_mass(masses[h][g0], k0)
            for g in candidates:
                need[h, g] = blocks_for_mass(masses[h][g], target[h] * (1.0 - REL_TOL))
        best = None
        for combo in itertools.product(candidates, repeat=len(heads)):
            cost = sum(kv_bytes(need[h, g], g, d) for h, g in zip(heads, combo))
            cost += sum(pooled_bytes(L, g, d) for g in set(combo))
            if best is None or cost < best[0]:
                best = (cost, combo)
        total += best[0]
        default += len(heads) * kv_bytes(k0, g0, d) + pooled_bytes(L, g0, d)
        for h, g in zip(heads, best[1]):
            gran[h] = g
            budget[h] = need[h, g]
            kept[h] = kept_mass(masses[h][g], need[h, g])
    return {"gran": gran, "budget": budget, "target": target, "kept": kept,
            "bytes": total, "bytes_default": default}


def attn_rate(rates: dict, g: int) -> float:
    """Attention's K/V bytes per second at block size g: rates["attn_bps"] is
    one rate, or pairs (size, rate) ascending, the first with size >= g
    applying (the last beyond them)."""
    r = rates["attn_bps"]
    if isinstance(r, (int, float)):
        return float(r)
    for size, bps in r:
        if g <= size:
            return bps
    return r[-1][1]


def select_time(rates: dict, candidates: int) -> float:
    """Modelled time of the selection kernel when its longest row has
    ``candidates`` blocks: the first bin of rates["select_s"] (pairs of (max
    candidates, seconds), ascending) that holds it."""
    for top, sec in rates["select_s"]:
        if candidates <= top:
            return sec
    return rates["select_s"][-1][1]


def step_time(assign: dict, need: dict, kinds, group: int, g0: int, L: int, d: int,
              batch: int, rates: dict) -> float:
    """Modelled decode-step time (seconds) of the retrieval heads' choice
    assign[h] = g with need[h, g] blocks each, for ``batch`` sequences:

      sum over heads of batch * kv_bytes / attn_rate(rates, g_h)
      + per block size in use: rates["score_pass_s"] + batch * (pooled bytes
        of the groups that use it) / rates["score_bps"]   (one scoring pass
        per size, a group reading each size's cache once)
      + select_time(the longest row: L / the smallest size in use, streaming
        rows counting L / g0)

    The three kernels run one after another; the terms are their times."""
    Hq = len(kinds)
    t = 0.0
    for h, g in assign.items():
        t += batch * kv_bytes(need[h, g], g, d) / attn_rate(rates, g)
    used = {}
    for grp in range(Hq // group):
        for g in {assign[h] for h in range(grp * group, (grp + 1) * group) if h in assign}:
            used[g] = used.get(g, 0) + 1
    for g, ngroups in used.items():
        t += rates["score_pass_s"] + batch * ngroups * pooled_bytes(L, g, d) / rates["score_bps"]
    rows = [L // g for g in used]
    if any(kinds[h] == STREAMING for h in range(Hq)):
        rows.append(L // g0)
    t += select_time(rates, max(rows) if rows else 0)
    return t


def choose_granularity_time(masses, kinds, group: int, g0: int, k0: int, candidates, L: int,
                            d: int, batch: int, rates: dict):
    """Per-head (g_h, k_h) for the retrieval heads minimising step_time
    instead of bytes; the error bound (each head keeps at least the default
    selection's mass) and the budget for a size (the fewest blocks reaching
    it) are those of choose_granularity.

    The scoring passes and the selection kernel are shared by every group,
    so the choice is global.  For each set U of sizes allowed (every
    non-empty subset of the candidates, in ascending order of the sorted
    tuple), each group takes, among the combinations of sizes in U in
    lexicographic order, the first that minimises its own K/V time plus its
    pooled-key time; the assignment is then timed with the passes and the
    selection of the sizes it actually uses, and the best U wins (ties: the
    first).  This is the global minimum: at the optimum's own set of sizes
    every group does at least as well, and fewer sizes cost no more.
    Returns the dict of choose_granularity, with ``time_s`` and
    ``time_s_default`` in place of the byte totals' role."""
    Hq = len(kinds)
    heads_of = []
    need = {}
    target = [0.0] * Hq
    for grp in range(Hq // group):
        heads = [h for h in range(grp * group, (grp + 1) * group) if kinds[h] != STREAMING]
        heads_of.append(heads)
        for h in heads:
            target[h] = kept_mass(masses[h][g0], k0)
            for g in set(candidates) | {g0}:
                need[h, g] = blocks_for_mass(masses[h][g], target[h] * (1.0 - REL_TOL))
    cands = list(candidates)
    best = None
    for r in range(1, len(cands) + 1):
        for U in itertools.combinations(sorted(cands), r):
            assign = {}
            for heads in heads_of:
                if not heads:
                    continue
                pick = None
                for combo in itertools.product(U, repeat=len(heads)):
                    c = sum(batch * kv_bytes(need[h, g], g, d) / attn_rate(rates, g)
                            for h, g in zip(heads, combo))
                    c += sum(batch * pooled_bytes(L, g, d) / rates["score_bps"]
                             for g in set(combo))
                    if pick is None or c < pick[0]:
                        pick = (c, combo)
                for h, g in zip(heads, pick[1]):
                    assign[h] = g
            t = step_time(assign, need, kinds, group, g0, L, d, batch, rates)
            if best is None or t < best[0]:
                best = (t, assign)
    default = {h: g0 for heads in heads_of for h in heads}
    gran = [g0] * Hq
    budget = [0] * Hq
    kept = [0.0] * Hq
    for h, g in best[1].items():
        gran[h] = g
        budget[h] = need[h, g]
        kept[h] = kept_mass(masses[h][g], need[h, g])
    return {"gran": gran, "budget": budget, "target": target, "kept": kept,
            "time_s": best[0],
            "time_s_default": step_time(default, need, kinds, group, g0, L, d, batch, rates)}


def pool_cache(k: np.ndarray, g: int) -> np.ndarray:
    """Mean key of each block of g tokens: [Bt, Hkv, L, d] -> [Bt, Hkv, L/g, d]."""
    Bt, Hkv, L, d = k.shape
    return k.astype(np.float64).reshape(Bt, Hkv, L // g, g, d).mean(axis=3)


def decode_scores(q: np.ndarray, k: np.ndarray, kinds, gran):
    """scores[b][h] = q[b,h] . kbar_{g_h}[b, h/G, j] / sqrt(d) over the L/g_h
    blocks of head h's size, for retrieval heads (None for streaming heads)."""
    Bt, Hq, d = q.shape
    group = Hq // k.shape[1]
    caches = {g: pool_cache(k, g) for g in sorted({gran[h] for h in range(Hq)
                                                    if kinds[h] != STREAMING})}
    out = [[None] * Hq for _ in range(Bt)]
    for b in range(Bt):
        for h in range(Hq):
            if kinds[h] != STREAMING:
                kb = caches[gran[h]][b, h // group]
                out[b][h] = kb @ q[b, h].astype(np.float64) / math.sqrt(d)
    return out


def select_row(scores_row: np.ndarray, k: int) -> list[int]:
    """k blocks of a decode row: block 0 and the last block, then the
    highest-scoring of the rest, ties to the lower index; ascending."""
    nb = len(scores_row)
    mand = _mandatory(nb)
    if k >= nb:
        return list(range(nb))
    rest = np.array([j for j in range(nb) if j not in set(mand)], dtype=np.int64)
    order = rest[np.lexsort((rest, -scores_row[rest]))] if len(rest) else rest
    take = max(0, k - len(mand))
    return sorted(mand + [int(j) for j in order[:take]])


def decode_select(scores, kinds, budget, gran, window_blocks: int, L: int, B: int):
    """idx [Bt, Hq, kmax] (-1 padded; block indices at the head's own size) and
    cnt [Bt, Hq].  Retrieval heads keep budget[h] blocks of gran[h] tokens;
    streaming heads keep block 0 and the last window_blocks blocks of B."""
    Bt = len(scores)
    Hq = len(kinds)
    lists = {}
    for b in range(Bt):
        for h in range(Hq):
            if kinds[h] == STREAMING:
                nb = L // B
                lists[b, h] = sorted({0} | set(range(max(0, nb - window_blocks), nb)))
            else:
                lists[b, h] = select_row(scores[b][h], budget[h])
    kmax = max(len(x) for x in lists.values())
    idx = np.full((Bt, Hq, kmax), -1, np.int32)
    cnt = np.zeros((Bt, Hq), np.int32)
    for (b, h), sel in lists.items():
        idx[b, h, :len(sel)] = sel
        cnt[b, h] = len(sel)
    return idx, cnt
