"""Oracle: one decode step over an HBM-resident KV cache with streaming and
retrieval heads, in fp64.

Test infrastructure only (see the package docstring).

Fluxion ("Intuizioni Chiave" 2) splits heads into streaming heads, which keep
only the default-retained KV (the sink block plus a recent window), and
retrieval heads, which pick blocks by top-k at block granularity.  Layout:
q [Bt, Hq, d]; K, V [Bt, Hkv, L, d]; blocks of B tokens, nb = L / B.  The new
token is already in the cache at position L-1, so every key is visible.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import select_row

STREAMING = 1


def pool_cache(k: np.ndarray, B: int) -> np.ndarray:
    """Mean key of each block: [Bt, Hkv, L, d] -> [Bt, Hkv, L/B, d] (fp64)."""
    Bt, Hkv, L, d = k.shape
    return k.astype(np.float64).reshape(Bt, Hkv, L // B, B, d).mean(axis=3)


def decode_scores(q: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """scores[b, h, j] = q[b, h] . kbar[b, h // G, j] / sqrt(d)."""
    Bt, Hq, d = q.shape
    group = Hq // kbar.shape[1]
    out = np.empty((Bt, Hq, kbar.shape[2]))
    for b in range(Bt):
        for h in range(Hq):
            out[b, h] = kbar[b, h // group] @ q[b, h].astype(np.float64) / math.sqrt(d)
    return out


def streaming_blocks(nb: int, window_blocks: int) -> list[int]:
    """Block 0 plus the last ``window_blocks`` blocks."""
    return sorted({0} | set(range(max(0, nb - window_blocks), nb)))


def decode_select(scores: np.ndarray, kinds, budget: int, window_blocks: int):
    """idx [Bt, Hq, kmax] (-1 padded) and cnt [Bt, Hq].

    Retrieval heads keep ``budget`` blocks: block 0, the last block (holding
    the current token) and the top-scoring rest, ties to the lower index --
    the prefill rule for the last query-block row.  Streaming heads keep the
    fixed sink + window list.
    """
    Bt, Hq, nb = scores.shape
    lists = {}
    for b in range(Bt):
        for h in range(Hq):
            if kinds[h] == STREAMING:
                lists[b, h] = streaming_blocks(nb, window_blocks)
            else:
                lists[b, h] = select_row(scores[b, h], nb - 1, budget)
    kmax = max(len(x) for x in lists.values())
    idx = np.full((Bt, Hq, kmax), -1, np.int32)
    cnt = np.zeros((Bt, Hq), np.int32)
    for (b, h), sel in lists.items():
        idx[b, h, :len(sel)] = sel
        cnt[b, h] = len(sel)
    return idx, cnt


def decode_attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, idx: np.ndarray,
                  cnt: np.ndarray, B):
    """Softmax attention of each new query over its selected blocks.

    B is the block size in tokens, one for all heads or one per head (a
    head's block j covers tokens [j*B_h, (j+1)*B_h)).
    Returns (o [Bt, Hq, d], lse [Bt, Hq]) in fp64.
    """
    Bt, Hq, d = q.shape
    group = Hq // k.shape[1]
    sizes = [int(B)] * Hq if np.isscalar(B) else [int(x) for x in B]
    o = np.empty((Bt, Hq, d))
    lse = np.empty((Bt, Hq))
    for b in range(Bt):
        for h in range(Hq):
            blocks = idx[b, h, :cnt[b, h]]
            Bh = sizes[h]
            u = np.concatenate([np.arange(j * Bh, (j + 1) * Bh) for j in blocks])
            ku = k[b, h // group, u].astype(np.float64)
            vu = v[b, h // group, u].astype(np.float64)
            logits = ku @ q[b, h].astype(np.float64) / math.sqrt(d)
            m = logits.max()
            p = np.exp(logits - m)
            o[b, h] = p @ vu / p.sum()
            lse[b, h] = m + math.log(p.sum())
    return o, lse
