"""Oracle: offline coverage calibration, from a calibration draw to per-head
block demands d_h.

Test infrastructure only (see the package docstring).

S-HPLB profiles each head offline on calibration data and sizes its budget by
the attention-weight recovery ratio, e.g. 90% of the total weight (Italian
summary, "Profilatura Offline"; Chinese summary 2.1 "离线分析").  Because the
ratio of budget to context length is stable across lengths (Chinese summary
2.1, "稀疏性稳定性观察"), the draw may be shorter than the target length; the
head's density is carried over and turned into blocks at the target nb.
"""
from __future__ import annotations

import math

import numpy as np

from .plan import budget_for_density, causal_blocks


def block_mass(q: np.ndarray, k: np.ndarray, B: int, i: int) -> np.ndarray:
    """Attention mass of query block i on each key block j <= i.

    m[j] = (1/B) * sum over queries t in block i of the causal softmax weight
    that t puts on keys u in block j (u <= t).  The masses sum to 1.
    """
    d = q.shape[1]
    t = np.arange(i * B, (i + 1) * B)
    u = np.arange(0, (i + 1) * B)
    logits = q[t].astype(np.float64) @ k[u].astype(np.float64).T / math.sqrt(d)
    logits[u[None, :] > t[:, None]] = -np.inf
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p.reshape(B, i + 1, B).sum(axis=2).sum(axis=0) / B


def coverage_count(mass: np.ndarray, cover: float) -> int:
    """Fewest blocks whose mass reaches ``cover``, taking blocks by mass,
    largest first (ties to the lower block index)."""
    order = np.lexsort((np.arange(len(mass)), -mass))
    acc = 0.0
    for n, j in enumerate(order, start=1):
        acc += mass[j]
        if acc >= cover:
            return n
    return len(mass)


def head_density(q: np.ndarray, k: np.ndarray, B: int, cover: float = 0.9) -> float:
    """rho_h = sum_i c_i / sum_i (i+1): the fraction of causal blocks a head
    needs to recover ``cover`` of its attention mass in every query block."""
    nb = q.shape[0] // B
    need = 0
    for i in range(nb):
        need += coverage_count(block_mass(q, k, B, i), cover)
    return need / causal_blocks(nb)


def demand_for_density(rho: float, nb: int) -> int:
    """d_h: the per-row block budget whose density at nb is nearest rho
    (ties -> smaller budget)."""
    return budget_for_density(rho, nb)


# ---------------------------------------------------------------------------
# Output-aware demand (Fluxion, "Intuizioni Chiave" 1, "Budgeting KV
# Consapevole dell'Output"): budgets follow how far the sparse attention output
# strays from the full output, and the head's relative contribution, rather
# than attention mass -- a sink block can draw most of the mass while its
# values carry little of the output.

def block_output(q: np.ndarray, k: np.ndarray, v: np.ndarray, B: int, i: int):
    """Full causal attention of query block i, split by key block.

    Returns (parts [i+1, B, d], mass [i+1, B]): parts[j, t] = sum over keys u
    of block j (u <= t) of p[t, u] v[u] and mass[j, t] = sum of those p[t, u],
    with p the causal softmax of query t over all its keys.  sum_j parts[j] is
    the full output and sum_j mass[j] = 1 for every query.
    """
    d = q.shape[1]
    t = np.arange(i * B, (i + 1) * B)
    u = np.arange(0, (i + 1) * B)
    logits = q[t].astype(np.float64) @ k[u].astype(np.float64).T / math.sqrt(d)
    logits[u[None, :] > t[:, None]] = -np.inf
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    pb = p.reshape(B, i + 1, B)                           # [t, j, u within block]
    vb = v[u].astype(np.float64).reshape(i + 1, B, -1)    # [j, u, d]
    parts = np.einsum("tju,jud->jtd", pb, vb)
    mass = pb.sum(axis=2).T                               # [j, t]
    return parts, mass


def output_deviation(parts: np.ndarray, mass: np.ndarray, blocks) -> float:
    """Relative deviation of attention restricted to ``blocks`` (and
    renormalised over their keys, as the sparse kernel computes it) from the
    full output: mean_t |o_S[t] - o[t]| / mean_t |o[t]|."""
    full = parts.sum(axis=0)
    sel = list(blocks)
    o_s = parts[sel].sum(axis=0) / mass[sel].sum(axis=0)[:, None]
    num = np.linalg.norm(o_s - full, axis=1).mean()
    den = np.linalg.norm(full, axis=1).mean()
    return float(num / den) if den > 0 else 0.0


def output_count(parts: np.ndarray, mass: np.ndarray, i: int, eps: float) -> int:
    """Fewest blocks whose restricted output deviates by at most ``eps``.

    The sink block 0 and the diagonal block i come first (every selection
    keeps them); then blocks 1..i-1 by the size of their output part,
    mean_t |parts[j, t]|, largest first (ties to the lower block index).
    """
    order = sorted({0, i})
    rest = np.arange(1, i)
    if len(rest):
        size = np.linalg.norm(parts[rest], axis=2).mean(axis=1)
        order += [int(j) for j in rest[np.lexsort((rest, -size))]]
    for n in range(len(sorted({0, i})), len(order) + 1):
        if output_deviation(parts, mass, order[:n]) <= eps:
            return n
    return len(order)


def head_output_norm(q: np.ndarray, k: np.ndarray, v: np.ndarray, B: int) -> float:
    """Mean norm of a head's full attention output: its contribution to the
    layer's representation (the pages' "relative contribution of the head")."""
    nb = q.shape[0] // B
    tot = 0.0
    for i in range(nb):
        parts, _ = block_output(q, k, v, B, i)
        tot += np.linalg.norm(parts.sum(axis=0), axis=1).mean()
    return tot / nb


def head_output_density(q: np.ndarray, k: np.ndarray, v: np.ndarray, B: int,
                        eps: float) -> float:
    """rho_h = sum_i c_i / sum_i (i+1) with c_i = output_count at tolerance eps."""
    nb = q.shape[0] // B
    need = 0
    for i in range(nb):
        parts, mass = block_output(q, k, v, B, i)
        need += output_count(parts, mass, i, eps)
    return need / causal_blocks(nb)


def output_aware_tolerances(norms, eps: float) -> list[float]:
    """Per-head tolerance: eps scaled by the heads' mean output norm over the
    head's own, so heads that contribute more are held to a tighter bound."""
    mean = float(np.mean(norms))
    return [eps * mean / n if n > 0 else float("inf") for n in norms]
