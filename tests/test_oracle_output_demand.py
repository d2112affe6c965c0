"""Pins for the output-aware demand signal of the calibration oracle.

The per-block split of the full output is checked against the attention
oracle run over all blocks; the deviation of a restricted output against the
attention oracle run over that block set (an independent route through the
renormalisation); the counts against closed forms (constant values), the
attention-sink case the pages describe, and monotonicity in the tolerance.
"""
import numpy as np

from oracle import attention as A
from oracle import calib as C


def _draw(seed, S=384, d=16, scale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((S, d)) * scale
    k = r.standard_normal((S, d))
    v = r.standard_normal((S, d))
    return q, k, v


def test_parts_add_up_to_the_full_attention_output():
    q, k, v = _draw(1)
    B = 32
    for i in (0, 1, 5, 11):
        parts, mass = C.block_output(q, k, v, B, i)
        o, _ = A.attend_item(q, k, v, i, list(range(i + 1)), B)
        np.testing.assert_allclose(parts.sum(axis=0), o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(mass.sum(axis=0), 1.0, rtol=1e-12)


def test_restricted_output_matches_sparse_attention_oracle():
    q, k, v = _draw(2, scale=2.0)
    B = 32
    r = np.random.default_rng(3)
    for i in (3, 7, 11):
        parts, mass = C.block_output(q, k, v, B, i)
        o_full, _ = A.attend_item(q, k, v, i, list(range(i + 1)), B)
        for _ in range(4):
            extra = r.choice(np.arange(1, i), size=int(r.integers(0, i - 1)), replace=False)
            blocks = sorted({0, i} | set(int(j) for j in extra))
            o_s, _ = A.attend_item(q, k, v, i, blocks, B)
            want = (np.linalg.norm(o_s - o_full, axis=1).mean()
                    / np.linalg.norm(o_full, axis=1).mean())
            assert abs(C.output_deviation(parts, mass, blocks) - want) < 1e-12
        assert C.output_deviation(parts, mass, range(i + 1)) < 1e-12


def test_constant_values_need_only_the_mandatory_blocks():
    q, k, _ = _draw(4)
    v = np.tile(np.arange(16.0), (q.shape[0], 1))      # every value row equal
    B = 32
    for i in range(12):
        parts, mass = C.block_output(q, k, v, B, i)
        assert C.output_count(parts, mass, i, 1e-9) == len({0, i})


def test_attention_sink_draws_mass_but_not_output():
    # block 0's keys align with every query (large logits) but its values are
    # zero: attention mass says "block 0 is enough", the output says otherwise
    r = np.random.default_rng(5)
    S, d, B = 512, 16, 32
    u = r.standard_normal(d)
    u /= np.linalg.norm(u)
    q = r.standard_normal((S, d)) * 0.3 + 3.0 * u
    k = r.standard_normal((S, d)) * 0.3
    k[:B] += 9.0 * u
    v = r.standard_normal((S, d))
    v[:B] = 0.0
    i = 15
    mass_count = C.coverage_count(C.block_mass(q, k, B, i), 0.9)
    parts, mass = C.block_output(q, k, v, B, i)
    out_count = C.output_count(parts, mass, i, 0.1)
    assert mass_count <= 2
    assert out_count > mass_count + 3


def test_counts_shrink_as_the_tolerance_grows():
    q, k, v = _draw(6, scale=1.5)
    B = 32
    for i in (4, 9, 11):
        parts, mass = C.block_output(q, k, v, B, i)
        counts = [C.output_count(parts, mass, i, e) for e in (0.0, 0.05, 0.1, 0.3, 1.0, 10.0)]
        assert counts == sorted(counts, reverse=True)
        assert counts[0] == i + 1
        assert counts[-1] == len({0, i})


def test_tolerances_follow_the_heads_relative_contribution():
    assert C.output_aware_tolerances([1.0, 1.0, 1.0], 0.1) == [0.1, 0.1, 0.1]
    tol = C.output_aware_tolerances([2.0, 1.0, 1.0, 0.0], 0.1)
    # mean norm 1.0: the doubled head is held to half the tolerance
    assert abs(tol[0] - 0.05) < 1e-15 and abs(tol[1] - 0.1) < 1e-15
    assert tol[3] == float("inf")
