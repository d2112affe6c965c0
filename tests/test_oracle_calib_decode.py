"""Pins for the oracle's coverage calibration and decode step (no GPU)."""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import calib, decode
from oracle.attention import select_row


def test_block_mass_sums_to_one_and_uniform_closed_form():
    B, nb, d = 4, 6, 8
    S = B * nb
    q = np.zeros((S, d))          # every logit 0: uniform causal attention
    k = np.random.default_rng(0).standard_normal((S, d))
    for i in range(nb):
        m = calib.block_mass(q, k, B, i)
        assert abs(m.sum() - 1.0) < 1e-12
        # closed form: query t gives 1/(t+1) to each key u <= t
        exp = np.zeros(i + 1)
        for t in range(i * B, (i + 1) * B):
            for j in range(i + 1):
                visible = min(B, max(0, t - j * B + 1))
                exp[j] += visible / (t + 1) / B
        np.testing.assert_allclose(m, exp, rtol=1e-12)


@pytest.mark.parametrize("seed", range(25))
def test_coverage_count_brute_force(seed):
    r = np.random.default_rng(seed)
    n = int(r.integers(1, 9))
    mass = r.random(n)
    mass /= mass.sum()
    cover = 0.9
    got = calib.coverage_count(mass, cover)
    best = min(len(c) for size in range(1, n + 1)
               for c in itertools.combinations(range(n), size)
               if sum(mass[j] for j in c) >= cover - 1e-15)
    assert got == best


@pytest.mark.parametrize("B,nb", [(8, 16), (4, 9), (16, 5)])
def test_uniform_attention_density_closed_form(B, nb):
    # q = 0 gives every visible key the same weight: query t puts 1/(t+1) on
    # each key u <= t.  Block j < i then holds (1/B) sum_t B/(t+1), the
    # diagonal block (1/B) sum_t (t - iB + 1)/(t+1).  The count for row i is
    # the fewest of these, largest first, reaching 0.9; the density is the
    # counts' sum over the causal block total.
    d = 4
    q = np.zeros((B * nb, d))
    k = np.random.default_rng(1).standard_normal((B * nb, d))
    need = 0
    for i in range(nb):
        ts = range(i * B, (i + 1) * B)
        off = sum(B / (t + 1) for t in ts) / B
        diag = sum((t - i * B + 1) / (t + 1) for t in ts) / B
        masses = sorted([off] * i + [diag], reverse=True)
        acc, c = 0.0, 0
        while c < len(masses) and acc < 0.9 - 1e-12:
            acc += masses[c]
            c += 1
        need += c
    assert calib.head_density(q, k, B) == pytest.approx(need / (nb * (nb + 1) / 2), abs=1e-15)


def test_peaked_head_needs_fewer_blocks():
    B, nb, d = 8, 16, 16
    S = B * nb
    rng = np.random.default_rng(2)
    k = rng.standard_normal((S, d))
    q = rng.standard_normal((S, d))
    assert calib.head_density(q * 8.0, k, B) < calib.head_density(q * 0.1, k, B)


def test_decode_streaming_blocks():
    assert decode.streaming_blocks(10, 3) == [0, 7, 8, 9]
    assert decode.streaming_blocks(4, 8) == [0, 1, 2, 3]


def test_decode_against_sdpa():
    Bt, Hq, Hkv, L, B, d = 2, 6, 2, 64, 4, 8
    rng = np.random.default_rng(3)
    q = rng.standard_normal((Bt, Hq, d)) * 2
    k = rng.standard_normal((Bt, Hkv, L, d))
    v = rng.standard_normal((Bt, Hkv, L, d))
    kbar = decode.pool_cache(k, B)
    sc = decode.decode_scores(q, kbar)
    kinds = np.array([1, 0, 0, 1, 0, 0], np.uint8)
    idx, cnt = decode.decode_select(sc, kinds, 5, 3)
    o, lse = decode.decode_attend(q, k, v, idx, cnt, B)
    nb = L // B
    for b in range(Bt):
        for h in range(Hq):
            sel = list(idx[b, h, :cnt[b, h]])
            if kinds[h] == 1:
                assert sel == decode.streaming_blocks(nb, 3)
            else:
                assert sel == select_row(sc[b, h], nb - 1, 5)
            mask = np.zeros(L, dtype=bool)
            for j in sel:
                mask[j * B:(j + 1) * B] = True
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, h])[None, None, None],
                torch.from_numpy(k[b, h // 3])[None, None],
                torch.from_numpy(v[b, h // 3])[None, None],
                attn_mask=torch.from_numpy(mask)[None, None, None])[0, 0, 0].numpy()
            np.testing.assert_allclose(o[b, h], ref, atol=1e-12)
            logits = torch.from_numpy(k[b, h // 3][mask] @ q[b, h] / math.sqrt(d))
            assert abs(lse[b, h] - torch.logsumexp(logits, 0).item()) < 1e-12
            # scores are pooled-key dot products
            for j in range(nb):
                ref_s = k[b, h // 3, j * B:(j + 1) * B].mean(0) @ q[b, h] / math.sqrt(d)
                assert abs(sc[b, h, j] - ref_s) < 1e-12
