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
