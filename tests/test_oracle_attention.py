"""Pins for the oracle's pooling, scoring, selection and attention (no GPU).

Attention is pinned to torch's scaled_dot_product_attention (a library
routine, run on the CPU in fp64) in the special cases where block-sparse
attention reduces to dense masked attention; selection to brute-force ranking;
scores to scalar loops; pooling to a closed form.
"""
import itertools
import math
import random

import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_pool_closed_form():
    H, nb, B, d = 2, 3, 4, 5
    a = _rand((H, nb, 1, d), 0)
    step = _rand((H, nb, 1, d), 1)
    r = np.arange(B).reshape(1, 1, B, 1)
    x = (a + r * step).reshape(H, nb * B, d)
    # mean of an arithmetic sequence a, a+s, ..., a+(B-1)s is a + s(B-1)/2
    np.testing.assert_allclose(A.pool_blocks(x, B), (a + step * (B - 1) / 2)[:, :, 0], rtol=1e-12)


def test_block_scores_scalar_loops():
    Hq, Hkv, nb, d = 4, 2, 5, 3
    qb = _rand((Hq, nb, d), 2)
    kb = _rand((Hkv, nb, d), 3)
    s = A.block_scores(qb, kb, Hq // Hkv)
    for h in range(Hq):
        for i in range(nb):
            for j in range(nb):
                if j > i:
                    assert s[h, i, j] == -math.inf
                else:
                    acc = 0.0
                    for c in range(d):
                        acc += qb[h, i, c] * kb[h // 2, j, c]
                    assert abs(s[h, i, j] - acc / math.sqrt(d)) < 1e-12


def _brute_select(scores, i, k):
    keep = min(k, i + 1)
    chosen = {0, i}
    rest = keep - len(chosen)
    cand = list(range(1, i))
    picked = []
    for j in cand:
        # rank: candidates strictly better (higher score, or equal score at a lower index)
        rank = sum(1 for jj in cand if scores[jj] > scores[j] or (scores[jj] == scores[j] and jj < j))
        if rank < rest:
            picked.append(j)
    return sorted(chosen | set(picked))


@pytest.mark.parametrize("seed", range(60))
def test_select_row_brute_force(seed):
    r = random.Random(seed)
    i = r.randint(0, 12)
    k = r.randint(2, 14)
    # integer scores force many ties
    scores = np.array([float(r.randint(0, 4)) for _ in range(i + 1)])
    got = A.select_row(scores, i, k)
    assert got == _brute_select(scores, i, k)
    assert 0 in got and i in got and len(got) == min(k, i + 1)
    assert got == sorted(set(got))


def _sdpa(q, k, v, mask):
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None])[0, 0].numpy()


@pytest.mark.parametrize("B,nb,d", [(4, 6, 8), (8, 5, 16), (16, 3, 32)])
def test_all_blocks_equals_dense_causal(B, nb, d):
    S = B * nb
    q, k, v = _rand((S, d), 10, 2.0), _rand((S, d), 11), _rand((S, d), 12)
    causal = np.tril(np.ones((S, S), dtype=bool))
    ref = _sdpa(q, k, v, causal)
    for i in range(nb):
        o, lse = A.attend_item(q, k, v, i, list(range(i + 1)), B)
        np.testing.assert_allclose(o, ref[i * B:(i + 1) * B], atol=1e-12, rtol=1e-10)
        logits = torch.from_numpy(q[i * B:(i + 1) * B] @ k[:(i + 1) * B].T / math.sqrt(d))
        logits = logits.masked_fill(~torch.from_numpy(causal[i * B:(i + 1) * B, :(i + 1) * B]), -math.inf)
        np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=1).numpy(), rtol=1e-12)


def test_sink_and_diagonal_equals_masked_dense():
    B, nb, d = 8, 6, 16
    S = B * nb
    q, k, v = _rand((S, d), 20, 3.0), _rand((S, d), 21), _rand((S, d), 22)
    mask = np.zeros((S, S), dtype=bool)
    for t in range(S):
        i = t // B
        for u in range(S):
            if u <= t and (u // B == 0 or u // B == i):
                mask[t, u] = True
    ref = _sdpa(q, k, v, mask)
    for i in range(nb):
        o, _ = A.attend_item(q, k, v, i, sorted({0, i}), B)
        np.testing.assert_allclose(o, ref[i * B:(i + 1) * B], atol=1e-12, rtol=1e-10)


def test_lse_merge_of_disjoint_block_sets():
    B, nb, d = 4, 9, 8
    S = B * nb
    q, k, v = _rand((S, d), 30), _rand((S, d), 31), _rand((S, d), 32)
    i = 8
    blocks = [0, 2, 3, 5, 8]
    o, lse = A.attend_item(q, k, v, i, blocks, B)
    o1, l1 = A.attend_item(q, k, v, i, blocks[:2], B)
    o2, l2 = A.attend_item(q, k, v, i, blocks[2:], B)
    lm = np.logaddexp(l1, l2)
    om = o1 * np.exp(l1 - lm)[:, None] + o2 * np.exp(l2 - lm)[:, None]
    np.testing.assert_allclose(lse, lm, rtol=1e-12)
    np.testing.assert_allclose(o, om, atol=1e-12)


def test_select_all_shapes_and_counts():
    Hq, Hkv, nb, d = 4, 2, 10, 6
    s = A.block_scores(_rand((Hq, nb, d), 40), _rand((Hkv, nb, d), 41), 2)
    budgets = [2, 3, 5, 20]
    idx, cnt = A.select_all(s, budgets, 20)
    for h in range(Hq):
        for i in range(nb):
            assert cnt[h, i] == min(budgets[h], i + 1)
            row = list(idx[h, i, :cnt[h, i]])
            assert row == A.select_row(s[h, i], i, budgets[h])
            assert all(x == -1 for x in idx[h, i, cnt[h, i]:])


def test_select_matches_itertools_best_subset():
    # the kept set maximises the summed score among all valid sets of that size
    r = np.random.default_rng(5)
    for _ in range(20):
        i = int(r.integers(2, 10))
        k = int(r.integers(2, i + 2))
        scores = r.standard_normal(i + 1)
        got = A.select_row(scores, i, k)
        keep = min(k, i + 1)
        best = max(
            (c for c in itertools.combinations(range(1, i), keep - 2)),
            key=lambda c: sum(scores[j] for j in c))
        assert got == sorted({0, i} | set(best))
