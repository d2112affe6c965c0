"""Oracle: pooled block scores (Index), top-k block selection (Select) and
block-sparse causal attention (Attention) for prefill, in fp64.

Test infrastructure only (see the package docstring).

Layout: Q [Hq, S, d]; K, V [Hkv, S, d]; query head h reads KV head h // G
(contiguous grouped-query sharing, G = Hq / Hkv).  Blocks are B consecutive
tokens; nb = S / B.
"""
from __future__ import annotations

import math

import numpy as np


def pool_blocks(x: np.ndarray, B: int) -> np.ndarray:
    """Mean of each block of B rows: [H, S, d] -> [H, S/B, d] (fp64).

    The pages select at block granularity (Fluxion, "Accoppiamento
    Granularità-Budget"; Spin's Index step) but do not name the block summary;
    the mean is the reading used here.
    """
    H, S, d = x.shape
    return x.astype(np.float64).reshape(H, S // B, B, d).mean(axis=2)


def block_scores(qbar: np.ndarray, kbar: np.ndarray, group: int) -> np.ndarray:
    """S[h, i, j] = qbar[h, i] . kbar[h // group, j] / sqrt(d) for j <= i.

    Entries above the diagonal (j > i) are -inf: a query block never selects a
    future key block.
    """
    Hq, nb, d = qbar.shape
    out = np.full((Hq, nb, nb), -np.inf)
    lower = np.tril(np.ones((nb, nb), dtype=bool))
    for h in range(Hq):
        s = qbar[h] @ kbar[h // group].T / math.sqrt(d)
        out[h][lower] = s[lower]
    return out


def select_row(scores: np.ndarray, i: int, k: int) -> list[int]:
    """Blocks kept by query-block row i under a budget of k blocks.

    The sink block 0 (Fluxion, "Intuizioni Chiave" 1: the first tokens draw
    large attention) and the diagonal block i are always kept; the remaining
    min(k, i+1) - |{0, i}| blocks are the highest-scoring of 1..i-1, ties to
    the lower block index.  Returned in ascending block order.
    """
    keep = min(k, i + 1)
    mandatory = sorted({0, i})
    rest = keep - len(mandatory)
    chosen = list(mandatory)
    if rest > 0:
        cand = np.arange(1, i)
        order = np.lexsort((cand, -scores[cand]))   # score desc, then index asc
        chosen += [int(j) for j in cand[order[:rest]]]
    return sorted(chosen)


def select_all(scores: np.ndarray, budgets, kmax: int):
    """Selection for every (h, i): idx [Hq, nb, kmax] (-1 padded), cnt [Hq, nb]."""
    Hq, nb, _ = scores.shape
    idx = np.full((Hq, nb, kmax), -1, np.int32)
    cnt = np.zeros((Hq, nb), np.int32)
    for h in range(Hq):
        for i in range(nb):
            sel = select_row(scores[h, i], i, budgets[h])
            idx[h, i, :len(sel)] = sel
            cnt[h, i] = len(sel)
    return idx, cnt


def block_probabilities(scores_row: np.ndarray, i: int) -> np.ndarray:
    """Softmax over the causal blocks j <= i of a row's pooled scores: the
    row's estimate of how its attention mass falls on each block (fp64)."""
    s = scores_row[:i + 1].astype(np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def select_row_topp(scores_row: np.ndarray, i: int, p: float) -> list[int]:
    """Top-p block selection, the adaptive alternative the S-HPLB pages compare
    against (Italian summary, "Sparsità Eterogenea"; Chinese summary, "Top-p
    方法的局限"): the number of blocks a row keeps depends on its data.

    Reading: keep the sink block 0 and the diagonal block i, then blocks of
    1..i-1 by probability (score) descending, ties to the lower index, until
    the kept blocks' cumulative probability reaches p.  Ascending order.
    """
    prob = block_probabilities(scores_row, i)
    chosen = sorted({0, i})
    acc = float(sum(prob[j] for j in chosen))
    rest = np.arange(1, i)
    for j in rest[np.lexsort((rest, -prob[rest]))]:
        if acc >= p:
            break
        chosen.append(int(j))
        acc += float(prob[j])
    return sorted(chosen)


def select_all_topp(scores: np.ndarray, p: float, kmax: int):
    """select_row_topp for every (h, i); same layout as select_all."""
    Hq, nb, _ = scores.shape
    idx = np.full((Hq, nb, kmax), -1, np.int32)
    cnt = np.zeros((Hq, nb), np.int32)
    for h in range(Hq):
        for i in range(nb):
            sel = select_row_topp(scores[h, i], i, p)
            idx[h, i, :len(sel)] = sel
            cnt[h, i] = len(sel)
    return idx, cnt


def group_scores(scores: np.ndarray, group: int) -> np.ndarray:
    """Group-pooled block scores: the mean over the G query heads of a KV group.

    scores [Hq, nb, nb] (fp64, -inf above the diagonal) -> [Hkv, nb, nb].  With
    one list per group, one fetched K/V block serves all G heads (Fluxion,
    group-level access); the mean of the heads' scores is the reading used to
    rank blocks for the whole group.
    """
    Hq, nb, _ = scores.shape
    return scores.reshape(Hq // group, group, nb, nb).mean(axis=1)


def select_all_grouped(scores: np.ndarray, budgets, group: int, kmax: int):
    """Group-shared selection: for every (g, i) the blocks chosen by select_row
    on the group-pooled scores with the group's budget, given to each of the
    group's query heads.  Same output layout as select_all."""
    Hq, nb, _ = scores.shape
    gs = group_scores(scores, group)
    idx = np.full((Hq, nb, kmax), -1, np.int32)
    cnt = np.zeros((Hq, nb), np.int32)
    for g in range(Hq // group):
        for i in range(nb):
            sel = select_row(gs[g, i], i, budgets[g * group])
            for h in range(g * group, (g + 1) * group):
                idx[h, i, :len(sel)] = sel
                cnt[h, i] = len(sel)
    return idx, cnt


def attend_item(q: np.ndarray, k: np.ndarray, v: np.ndarray, i: int,
                blocks, B: int):
    """Causal softmax attention of query block i over the listed key blocks.

    q: the head's queries [S, d]; k, v: its KV head's keys/values [S, d]
    (any float type; promoted to fp64).  Key u is visible to query t when
    u <= t, so only the diagonal block is partly masked.  Two-pass softmax with
    scale 1/sqrt(d) (inputs are taken as already position-encoded).
    Returns (o [B, d], lse [B]) with lse the natural-log sum of exponentials.
    """
    d = q.shape[1]
    t = np.arange(i * B, (i + 1) * B)
    u = np.concatenate([np.arange(j * B, (j + 1) * B) for j in blocks])
    qi = q[t].astype(np.float64)
    ku = k[u].astype(np.float64)
    vu = v[u].astype(np.float64)
    logits = qi @ ku.T / math.sqrt(d)
    logits[u[None, :] > t[:, None]] = -np.inf
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    denom = p.sum(axis=1, keepdims=True)
    o = (p @ vu) / denom
    lse = (m + np.log(denom))[:, 0]
    return o, lse


def attend_all(q: np.ndarray, k: np.ndarray, v: np.ndarray, idx: np.ndarray,
               cnt: np.ndarray, B: int, items=None):
    """Attention for every (h, i) in ``items`` (default: all).

    q [Hq, S, d], k/v [Hkv, S, d]; idx/cnt as from selection.
    Returns dict item -> (o [B, d], lse [B]) with item = h*nb + i.
    """
    Hq, S, _ = q.shape
    group = Hq // k.shape[0]
    nb = S // B
    if items is None:
        items = range(Hq * nb)
    out = {}
    for item in items:
        h, i = divmod(int(item), nb)
        blocks = [int(j) for j in idx[h, i, :cnt[h, i]]]
        out[int(item)] = attend_item(q[h], k[h // group], v[h // group], i, blocks, B)
    return out
