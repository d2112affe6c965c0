"""Pins for the oracle's per-head decode granularity (block size and budget of
retrieval heads) and its selector.

Checked against: the exact decode softmax (masses sum to one, merge across
block sizes, reduce to single-token weights), the token-level attention logit
(scores at block size one), brute force over all block subsets (kept mass,
fewest blocks, and the group-level optimum of the selector), the token-set
invariance of attention (a selection at one block size equals the same tokens
at another), and the existing per-head decode selection at the default size.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import decode as D
from oracle import granularity as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _draw(seed, Bt=1, Hq=2, Hkv=1, L=256, d=16, scale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((Bt, Hq, d)) * scale
    k = r.standard_normal((Bt, Hkv, L, d))
    v = r.standard_normal((Bt, Hkv, L, d))
    return q, k, v


def test_block_mass_sums_merges_and_reduces_to_token_weights():
    q, k, _ = _draw(1, scale=2.0)
    m16 = G.decode_block_mass(q[0, 0], k[0, 0], 16)
    m32 = G.decode_block_mass(q[0, 0], k[0, 0], 32)
    assert abs(m16.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(m16.reshape(-1, 2).sum(axis=1), m32, rtol=1e-12, atol=1e-15)
    assert np.allclose(G.decode_block_mass(q[0, 0], k[0, 0], 256), [1.0])
    # block size one: the softmax of the scaled logits
    logits = np.array([k[0, 0, u] @ q[0, 0] for u in range(256)]) / 4.0
    w = np.exp(logits - logits.max())
    np.testing.assert_allclose(G.decode_block_mass(q[0, 0], k[0, 0], 1), w / w.sum(),
                               rtol=1e-12)


def _best_subset(mass, k):
    nb = len(mass)
    mand = sorted({0, nb - 1})
    rest = [j for j in range(nb) if j not in mand]
    take = max(0, k - len(mand))
    if take >= len(rest):
        return mass.sum()
    return max(mass[mand].sum() + mass[list(c)].sum() for c in itertools.combinations(rest, take))


def test_kept_mass_and_fewest_blocks_by_brute_force():
    r = np.random.default_rng(2)
    for _ in range(60):
        nb = int(r.integers(1, 8))
        mass = r.dirichlet(np.full(nb, 0.5))
        for k in range(len({0, nb - 1}), nb + 1):
            assert abs(G.kept_mass(mass, k) - _best_subset(mass, k)) < 1e-14
        target = float(r.uniform(0, 1))
        want = min(k for k in range(len({0, nb - 1}), nb + 1)
                   if _best_subset(mass, k) >= target or k == nb)
        assert G.blocks_for_mass(mass, target) == want


def test_scores_reduce_to_logits_and_average_across_sizes():
    q, k, _ = _draw(3)
    kinds = [0, 0]
    s1 = G.decode_scores(q, k, kinds, [1, 1])
    logits = np.array([k[0, 0, u] @ q[0, 1] for u in range(256)]) / 4.0
    np.testing.assert_allclose(s1[0][1], logits, rtol=1e-12, atol=1e-12)
    s16 = G.decode_scores(q, k, kinds, [16, 16])
    s32 = G.decode_scores(q, k, kinds, [32, 32])
    np.testing.assert_allclose(s16[0][0].reshape(-1, 2).mean(axis=1), s32[0][0],
                               rtol=1e-12, atol=1e-12)
    assert G.decode_scores(q, k, [1, 0], [16, 32])[0][0] is None


def test_selection_at_the_default_size_equals_the_decode_oracle():
    q, k, _ = _draw(4, Bt=2, Hq=4, Hkv=2, L=512)
    kinds = np.array([0, 1, 0, 0], np.uint8)
    B = 32
    s = D.decode_scores(q, D.pool_cache(k, B))
    sg = G.decode_scores(q, k, kinds, [B] * 4)
    want_idx, want_cnt = D.decode_select(s, kinds, 5, 3)
    idx, cnt = G.decode_select(sg, kinds, [5, 0, 5, 5], [B] * 4, 3, 512, B)
    assert np.array_equal(cnt, want_cnt)
    assert np.array_equal(idx, want_idx)


def test_attention_depends_only_on_the_token_set():
    q, k, v = _draw(5, Hq=3)
    # head 0: 16-token blocks pairing up into 32-token blocks {0, 2, 7};
    # head 1: 64-token blocks {0, 3} = 32-token blocks {0, 1, 6, 7}
    idx_g = np.array([[[0, 1, 4, 5, 14, 15], [0, 3, -1, -1, -1, -1],
                       [0, 7, -1, -1, -1, -1]]], np.int32)
    cnt_g = np.array([[6, 2, 2]], np.int32)
    idx_b = np.array([[[0, 2, 7, -1], [0, 1, 6, 7], [0, 7, -1, -1]]], np.int32)
    cnt_b = np.array([[3, 4, 2]], np.int32)
    o_g, l_g = D.decode_attend(q, k, v, idx_g, cnt_g, [16, 64, 32])
    o_b, l_b = D.decode_attend(q, k, v, idx_b, cnt_b, 32)
    np.testing.assert_allclose(o_g, o_b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l_g, l_b, rtol=1e-12)


def _brute_group(masses, heads, g0, k0, cands, L, d):
    """Least bytes over every size per head and every block subset that keeps
    the mandatory blocks and reaches the default's mass."""
    best = None
    opts = {}
    for h in heads:
        target = _best_subset(masses[h][g0], k0)
        for g in cands:
            m = masses[h][g]
            nb = len(m)
            mand = sorted({0, nb - 1})
            rest = [j for j in range(nb) if j not in mand]
            fewest = None
            for n in range(len(rest) + 1):
                if any(m[mand].sum() + m[list(c)].sum() >= target * (1 - 1e-12)
                       for c in itertools.combinations(rest, n)):
                    fewest = len(mand) + n
                    break
            opts[h, g] = fewest * g * d * 4
    for combo in itertools.product(cands, repeat=len(heads)):
        cost = sum(opts[h, g] for h, g in zip(heads, combo))
        cost += sum((L // g) * d * 4 for g in set(combo))
        best = cost if best is None else min(best, cost)
    return best


@pytest.mark.parametrize("seed", range(8))
def test_selector_reaches_the_group_optimum(seed):
    r = np.random.default_rng(100 + seed)
    L, d, Hq, group = 64, 4, 4, 2
    cands = (8, 16, 32)
    g0, k0 = 16, 2
    kinds = [0, int(r.integers(0, 2)), 0, 0]
    q = r.standard_normal((Hq, d)) * r.uniform(0.5, 4.0, (Hq, 1))
    k = r.standard_normal((Hq // group, L, d))
    masses = {h: {g: G.decode_block_mass(q[h], k[h // group], g) for g in cands}
              for h in range(Hq) if kinds[h] != 1}
    res = G.choose_granularity(masses, kinds, group, g0, k0, cands, L, d)
    total = 0
    for grp in range(Hq // group):
        heads = [h for h in range(grp * group, (grp + 1) * group) if kinds[h] != 1]
        total += _brute_group(masses, heads, g0, k0, cands, L, d)
        for h in heads:
            assert res["kept"][h] >= res["target"][h] * (1 - 1e-12)
    assert res["bytes"] == total
    assert res["bytes"] <= res["bytes_default"]
    assert res["budget"][1] == 0 or kinds[1] == 0


RATES0 = {"attn_bps": 1.0, "score_bps": 1.0, "score_pass_s": 0.0, "select_s": [[10 ** 9, 0.0]]}


def _tiny(seed, kinds=None):
    r = np.random.default_rng(300 + seed)
    L, d, Hq, group = 64, 4, 4, 2
    cands = (8, 16, 32)
    kinds = kinds or [0, int(r.integers(0, 2)), 0, 0]
    q = r.standard_normal((Hq, d)) * r.uniform(0.5, 4.0, (Hq, 1))
    k = r.standard_normal((Hq // group, L, d))
    masses = {h: {g: G.decode_block_mass(q[h], k[h // group], g) for g in cands}
              for h in range(Hq) if kinds[h] != 1}
    return L, d, Hq, group, cands, kinds, masses


@pytest.mark.parametrize("seed", range(6))
def test_time_selector_with_free_passes_and_selection_is_the_byte_selector(seed):
    # no fixed costs and one rate for every byte: the modelled time is the
    # byte count, and per-group choices are independent
    L, d, Hq, group, cands, kinds, masses = _tiny(seed)
    rb = G.choose_granularity(masses, kinds, group, 16, 2, cands, L, d)
    rt = G.choose_granularity_time(masses, kinds, group, 16, 2, cands, L, d, 1, RATES0)
    assert rt["time_s"] == pytest.approx(rb["bytes"], rel=1e-12)
    assert rt["time_s_default"] == pytest.approx(rb["bytes_default"], rel=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_time_selector_reaches_the_global_optimum(seed):
    # every assignment of sizes to every retrieval head, across groups
    L, d, Hq, group, cands, kinds, masses = _tiny(seed)
    rates = {"attn_bps": 3.0, "score_bps": 7.0, "score_pass_s": 40.0 + 30.0 * seed,
             "select_s": [[2, 5.0], [4, 90.0], [8, 400.0]]}
    res = G.choose_granularity_time(masses, kinds, group, 16, 2, cands, L, d, 2, rates)
    heads = [h for h in range(Hq) if kinds[h] != 1]
    need = {}
    for h in heads:
        target = G.kept_mass(masses[h][16], 2)
        for g in cands:
            need[h, g] = G.blocks_for_mass(masses[h][g], target * (1 - G.REL_TOL))
    best = min(G.step_time(dict(zip(heads, combo)), need, kinds, group, 16, L, d, 2, rates)
               for combo in itertools.product(cands, repeat=len(heads)))
    assert res["time_s"] == pytest.approx(best, rel=1e-12)
    for h in heads:
        assert res["kept"][h] >= res["target"][h] * (1 - 1e-12)
    assert res["time_s"] <= res["time_s_default"] * (1 + 1e-12)


def test_step_time_hand_example():
    # one group of two retrieval heads, L 64, d 4, batch 3, no streaming head:
    # head 0 at 8 tokens keeps 5 blocks, head 1 at 16 keeps 2.
    #   K/V: 3 * (5*8*4*4 + 2*16*4*4) = 3 * (640 + 512) = 3456 bytes at 2/s
    #   scoring: sizes 8 and 16, one group each: 2 passes of 10 s, plus
    #            3 * ((64/8)*4*4 + (64/16)*4*4) = 3 * (128 + 64) = 576 bytes at 4/s
    #   selection: the longest row has 64/8 = 8 candidates -> the [8, 7] bin
    kinds = [0, 0]
    rates = {"attn_bps": 2.0, "score_bps": 4.0, "score_pass_s": 10.0,
             "select_s": [[4, 1.0], [8, 7.0], [16, 50.0]]}
    t = G.step_time({0: 8, 1: 16}, {(0, 8): 5, (1, 16): 2}, kinds, 2, 16, 64, 4, 3, rates)
    assert t == pytest.approx(3456 / 2 + 20 + 576 / 4 + 7)
    # per-size attention rates: 8-token pieces at 1/s, 16-token ones at 4/s
    rates["attn_bps"] = [[8, 1.0], [16, 4.0]]
    t = G.step_time({0: 8, 1: 16}, {(0, 8): 5, (1, 16): 2}, kinds, 2, 16, 64, 4, 3, rates)
    assert t == pytest.approx(3 * 640 / 1 + 3 * 512 / 4 + 20 + 576 / 4 + 7)


def test_stored_decode_granularity_matches_the_oracle():
    from oracle import make_demands
    with open(os.path.join(ROOT, "workloads", "demands.json")) as f:
        stored = json.load(f)["5"]["granularity"]
    again = make_demands.profile_granularity(5)
    for key in ("gran", "budget", "bytes", "bytes_default", "candidates", "g0", "k0"):
        assert stored[key] == again[key], key
    for key in ("gran", "budget", "rates", "batch"):
        assert stored["time_model"][key] == again["time_model"][key], key
    assert stored["time_model"]["time_us"] == pytest.approx(again["time_model"]["time_us"])
    np.testing.assert_allclose(stored["kept"], again["kept"], rtol=1e-9)
