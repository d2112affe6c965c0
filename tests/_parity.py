"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the oracle.

Tolerances (bf16 inputs, fp32 accumulation on the GPU, fp64 oracle):
  scores      rtol 1e-4, atol 1e-6 (fp32 dot products of 64-128 terms)
  selection   bit-exact, except blocks whose oracle score lies within 1e-3
              relative of the row's k-th (last kept) score
  attention   fp32 output: max |O_gpu - O_ref| <= 1e-2 and
              sum|O_gpu - O_ref| / sum|O_ref| <= 2e-3, the oracle run on the
              GPU's own selected blocks, on the raw difference.
              bf16 output (the fp32 value rounded to nearest even): the mean
              relative error is taken against the oracle rounded the same
              way, with no allowance; the max-abs bound applies to the error
              in excess of the output's own rounding, max(0, |diff| -
              half_ulp) with half_ulp = 2^(e-8) for the larger of |O_gpu|,
              |O_ref| in [2^e, 2^(e+1)) -- without it a value above 2 could
              not meet 1e-2 even if it were exact before rounding
  lse         |lse_gpu - lse_ref| <= 4.5e-3 (natural log units): the
              normaliser sums the bf16-rounded weights, each within 2^-8
              relative of the exact weight, i.e. <= ln(1 + 2^-8) = 3.9e-3 in
              log, plus fp32 and ex2.approx error
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oa
from workloads import generate

MAX_ABS = 1e-2
MEAN_REL = 2e-3
SEL_REL = 1e-3
LSE_ABS = 4.5e-3


def to_dev(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def pooled(bits: np.ndarray, B: int) -> np.ndarray:
    """Oracle pooling one head at a time (keeps fp64 memory small)."""
    out = np.empty((bits.shape[0], bits.shape[1] // B, bits.shape[2]))
    for h in range(bits.shape[0]):
        out[h] = oa.pool_blocks(generate.bf16_to_f32(bits[h])[None], B)[0]
    return out


def check_scores(gpu: np.ndarray, ref: np.ndarray, rows=None):
    """gpu/ref [H, nb, nb]; only j <= i is defined."""
    H, nb, _ = ref.shape
    lower = np.tril(np.ones((nb, nb), dtype=bool))
    for h in range(H):
        g, r = gpu[h][lower], ref[h][lower]
        np.testing.assert_allclose(g, r, rtol=1e-4, atol=1e-6)


def check_selection_row(gpu_sel, ref_sel, scores_row, i):
    """Threshold rule; returns the number of tolerated mismatches."""
    g, r = set(int(x) for x in gpu_sel), set(int(x) for x in ref_sel)
    assert len(gpu_sel) == len(ref_sel), (i, gpu_sel, ref_sel)
    assert list(gpu_sel) == sorted(g), gpu_sel
    assert 0 in g and i in g and all(0 <= j <= i for j in g)
    diff = g ^ r
    if not diff:
        return 0
    kept = [j for j in r if j not in (0, i)]
    thr = min(scores_row[j] for j in kept)
    for j in diff:
        assert abs(scores_row[j] - thr) <= SEL_REL * abs(thr), (i, j, scores_row[j], thr)
    return len(diff)


def check_selection(idx, cnt, scores_ref, budgets, rows=None):
    """idx [H, nb, kmax], cnt [H, nb] from the GPU against oracle selection on
    the oracle's fp64 scores."""
    H, nb = cnt.shape
    tolerated = 0
    rows = rows if rows is not None else [(h, i) for h in range(H) for i in range(nb)]
    for h, i in rows:
        assert cnt[h, i] == min(budgets[h], i + 1), (h, i, cnt[h, i])
        ref = oa.select_row(scores_ref[h, i], i, budgets[h])
        gsel = idx[h, i, :cnt[h, i]]
        assert all(x == -1 for x in idx[h, i, cnt[h, i]:])
        tolerated += check_selection_row(gsel, ref, scores_ref[h, i], i)
    return tolerated


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (ties to even) of each element, as float64."""
    return generate.bf16_to_f64(generate.bf16_bits(np.asarray(x, dtype=np.float32)))


def output_errors(got: np.ndarray, ref: np.ndarray, bf16_out: bool):
    """Element errors for the two attention bounds: (for max-abs, for mean-rel)."""
    d = np.abs(got - ref)
    if not bf16_out:
        return d, d
    d_max = np.maximum(d - half_ulp_bf16(np.maximum(np.abs(ref), np.abs(got))), 0.0)
    return d_max, np.abs(got - bf16_round(ref))


def check_attention(out_gpu: np.ndarray, lse_gpu, x: dict, idx, cnt, B: int, items, group: int,
                    bf16_out: bool = False):
    """out_gpu [Hq, S, d] float; x holds the bf16 bits; items: ids h*nb+i."""
    nb = cnt.shape[1]
    by_head = {}
    for it in items:
        by_head.setdefault(int(it) // nb, []).append(int(it) % nb)
    num = den = 0.0
    worst = 0.0
    kv_cache = {}
    for h, rows in sorted(by_head.items()):
        g = h // group
        if g not in kv_cache:
            kv_cache.clear()
            kv_cache[g] = (generate.bf16_to_f32(x["k"][g]), generate.bf16_to_f32(x["v"][g]))
        k, v = kv_cache[g]
        q = generate.bf16_to_f32(x["q"][h])
        for i in rows:
            blocks = [int(j) for j in idx[h, i, :cnt[h, i]]]
            o, lse = oa.attend_item(q, k, v, i, blocks, B)
            got = out_gpu[h, i * B:(i + 1) * B]
            d_max, d_rel = output_errors(got, o, bf16_out)
            worst = max(worst, float(d_max.max()))
            num += float(d_rel.sum())
            den += float(np.abs(o).sum())
            if lse_gpu is not None:
                lg = lse_gpu[h, i * B:(i + 1) * B]
                assert np.abs(lg - lse).max() <= LSE_ABS, (h, i, np.abs(lg - lse).max())
    assert worst <= MAX_ABS, f"max abs error {worst} (beyond output rounding)"
    assert num / den <= MEAN_REL, f"mean relative error {num / den}"
    return worst, num / den


def sample_items(budgets, nb, per_head: int, seed: int):
    """First, last, heaviest (smallest i reaching the head's budget) and
    random items of every head."""
    r = np.random.default_rng(seed)
    items = []
    for h, k in enumerate(budgets):
        pick = {0, nb - 1, min(nb - 1, k - 1)}
        while len(pick) < min(per_head, nb):
            pick.add(int(r.integers(0, nb)))
        items += [h * nb + i for i in sorted(pick)]
    return items
