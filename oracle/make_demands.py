"""Write ``workloads/demands.json``: the offline profile of every prefill workload.

Test infrastructure: this script calls only the oracle and the seeded input
generator.  It performs the offline profiling step of S-HPLB (Italian summary,
"Profilatura Offline"; Chinese summary 2.1 "离线分析"): per head, the fraction
of causal blocks needed to recover 90% of the attention mass on a calibration
draw, turned into a per-row block demand d_h at the workload's length.  It
also records the uniform budget k_u for the workload's target density.

Workloads 1-3 calibrate on a draw with their own heads (scales s_h) and a
separate seed at min(S, 8192) tokens.  Workload 4 draws its head densities
from a lognormal (its recipe), clamped to [density(2), 1].

With --output-aware it adds, for the calibrated workloads, the output-aware
demand signal (Fluxion, "Intuizioni Chiave" 1): per head, the fraction of
causal blocks needed to keep the sparse output within a tolerance of the full
output, the tolerance scaled by the head's relative output norm.  The result
goes under "output_aware" beside the mass-based profile, which is left as is.

With --granularity it writes, for the decode workload, each retrieval head's
selection block size and budget (Fluxion, "Intuizioni Chiave" 2 and its
granularity-budget selector): on a calibration draw, every head keeps at least
the attention mass of the default selection, and each KV group takes the sizes
that move the fewest bytes per decode step (``oracle.granularity``).

Usage:  python -m oracle.make_demands [--out workloads/demands.json]
        python -m oracle.make_demands --output-aware [--workloads 1,2,3]
        python -m oracle.make_demands --granularity [--workloads 5]
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import calib, granularity, plan  # noqa: E402
from workloads import WORKLOADS, generate  # noqa: E402

K_MIN = 2
COVER = 0.9
EPS = 0.1          # output-aware: relative output deviation allowed for a mean head


def _head_density(args):
    number, h = args
    w = WORKLOADS[number]
    x = generate.prefill_inputs(w, tensors="qk", heads=[h], kv_heads=[h // w.group],
                                seed=w.calib_seed, seq_len=w.calib_len)
    q = generate.bf16_to_f64(x["q"][0])
    k = generate.bf16_to_f64(x["k"][0])
    return calib.head_density(q, k, w.block, COVER)


def _calib_qkv(number, h):
    w = WORKLOADS[number]
    x = generate.prefill_inputs(w, tensors="qkv", heads=[h], kv_heads=[h // w.group],
                                seed=w.calib_seed, seq_len=w.calib_len)
    return (generate.bf16_to_f64(x["q"][0]), generate.bf16_to_f64(x["k"][0]),
            generate.bf16_to_f64(x["v"][0]))


def _head_norm(args):
    number, h = args
    q, k, v = _calib_qkv(number, h)
    return calib.head_output_norm(q, k, v, WORKLOADS[number].block)


def _head_output_density(args):
    number, h, eps = args
    q, k, v = _calib_qkv(number, h)
    return calib.head_output_density(q, k, v, WORKLOADS[number].block, eps)


def profile_output_aware(number: int, pool) -> dict:
    w = WORKLOADS[number]
    nb = w.nb
    k_u = plan.budget_for_density(w.target_density, nb)
    heads = range(w.num_q_heads)
    norms = list(pool.map(_head_norm, [(number, h) for h in heads]))
    tol = calib.output_aware_tolerances(norms, EPS)
    rho = list(pool.map(_head_output_density, [(number, h, tol[h]) for h in heads]))
    demand = [calib.demand_for_density(r, nb) for r in rho]
    budgets = plan.maxmin_shift(k_u, demand, K_MIN, nb)
    return {
        "source": (f"output deviation <= {EPS} x (mean head output norm / head's) on the "
                   f"calibration draw (seed {w.calib_seed}, {w.calib_len} tokens)"),
        "eps": EPS, "output_norm": [round(float(x), 12) for x in norms],
        "tolerance": [round(float(x), 12) for x in tol],
        "density": [round(float(r), 12) for r in rho], "demand": demand,
        "budgets_maxmin": budgets,
        "mean_density_after_shift": sum(plan.kept_blocks(k, nb) for k in budgets)
        / (w.num_q_heads * plan.causal_blocks(nb)),
    }


GRANULARITIES = (16, 32, 64, 128)   # candidate block sizes of a retrieval head

# Rates of the decode kernels on a GB300 at the 16 x 64K shape, from the
# bench's decode block.  Attention: 320 MB of K/V at 32-token blocks in
# 60 us (5.3 TB/s); 248-257 MB at 16-token blocks in 51-53 us (4.85 TB/s,
# the selected pieces being half as long).  One scoring pass: 67 MB of
# pooled keys in 18 us and 134 MB in 31.4 us, i.e. 4.6 us plus 5.0 TB/s.
# Selection: 12.3 us when rows have up to 2048 candidates, 16.4 us up to 4096.
DECODE_RATES = {"attn_bps": [[16, 4.85e12], [32, 5.3e12]], "score_bps": 5.0e12,
                "score_pass_s": 4.6e-6, "select_s": [[2048, 12.3e-6], [4096, 16.4e-6]]}


def profile_granularity(number: int) -> dict:
    w = WORKLOADS[number]
    kinds = generate.head_kinds(w)
    x = generate.decode_inputs(w, tensors="qk", batches=[0], seed=w.calib_seed)
    q = generate.bf16_to_f64(x["q"][0])
    k = generate.bf16_to_f64(x["k"][0])
    g0, k0 = w.block, w.budget_tokens // w.block
    sizes = sorted(set(GRANULARITIES) | {g0})
    masses = {h: {g: granularity.decode_block_mass(q[h], k[h // w.group], g) for g in sizes}
              for h in range(w.num_q_heads) if kinds[h] != granularity.STREAMING}
    res = granularity.choose_granularity(masses, kinds, w.group, g0, k0, GRANULARITIES,
                                         w.seq_len, w.head_dim)
    rt = granularity.choose_granularity_time(masses, kinds, w.group, g0, k0, GRANULARITIES,
                                             w.seq_len, w.head_dim, w.batch, DECODE_RATES)
    return {
        "workload": w.name,
        "source": (f"decode query of a calibration draw (seed {w.calib_seed}, one sequence, "
                   f"{w.seq_len} tokens): each retrieval head keeps at least the attention "
                   f"mass of the default selection ({k0} blocks of {g0}); per KV group the "
                   f"block sizes that move the fewest bytes per step"),
        "candidates": list(GRANULARITIES), "g0": g0, "k0": k0,
        "gran": res["gran"], "budget": res["budget"],
        "target": [round(float(t), 12) for t in res["target"]],
        "kept": [round(float(t), 12) for t in res["kept"]],
        "bytes": res["bytes"], "bytes_default": res["bytes_default"],
        "time_model": {
            "rates": DECODE_RATES, "batch": w.batch,
            "gran": rt["gran"], "budget": rt["budget"],
            "time_us": round(rt["time_s"] * 1e6, 6),
            "time_us_default": round(rt["time_s_default"] * 1e6, 6),
            "time_us_of_byte_choice": round(granularity.step_time(
                {h: res["gran"][h] for h in range(w.num_q_heads) if kinds[h] != granularity.STREAMING},
                {(h, g): res["budget"][h] for h in range(w.num_q_heads)
                 for g in [res["gran"][h]] if kinds[h] != granularity.STREAMING},
                kinds, w.group, g0, w.seq_len, w.head_dim, w.batch, DECODE_RATES) * 1e6, 6),
        },
    }


def profile(number: int, pool=None) -> dict:
    w = WORKLOADS[number]
    nb = w.nb
    k_u = plan.budget_for_density(w.target_density, nb)
    if w.demand_source == "coverage":
        jobs = [(number, h) for h in range(w.num_q_heads)]
        rho = list(pool.map(_head_density, jobs)) if pool else [_head_density(j) for j in jobs]
        source = (f"90% attention-mass coverage on a calibration draw "
                  f"(seed {w.calib_seed}, {w.calib_len} tokens)")
    elif w.demand_source == "lognormal":
        raw = generate.lognormal_densities(w)
        lo = plan.density(2, nb)
        rho = [float(min(1.0, max(lo, r))) for r in raw]
        source = (f"lognormal densities (sigma {w.lognormal_sigma}, mean "
                  f"{w.target_density}) clamped to [density(2), 1]")
    else:
        raise ValueError(w.demand_source)
    demand = [calib.demand_for_density(r, nb) for r in rho]
    budgets = plan.maxmin_shift(k_u, demand, K_MIN, nb)
    return {
        "workload": w.name, "nb": nb, "target_density": w.target_density,
        "k_uniform": k_u, "k_min": K_MIN, "cover": COVER, "source": source,
        "density": [round(float(r), 12) for r in rho], "demand": demand,
        "budgets_maxmin": budgets,
        "mean_density_after_shift": sum(plan.kept_blocks(k, nb) for k in budgets)
        / (w.num_q_heads * plan.causal_blocks(nb)),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(ROOT, "workloads", "demands.json"))
    ap.add_argument("--workloads", default="1,2,3,4")
    ap.add_argument("--output-aware", action="store_true")
    ap.add_argument("--granularity", action="store_true")
    args = ap.parse_args()
    out = {}
    if os.path.exists(args.out):
        with open(args.out) as f:
            out = json.load(f)
    if args.granularity:
        nums = [int(x) for x in args.workloads.split(",")] if args.workloads != "1,2,3,4" else [5]
        for n in nums:
            if WORKLOADS[n].demand_source != "decode":
                continue
            t = time.time()
            out.setdefault(str(n), {})["granularity"] = profile_granularity(n)
            gr = out[str(n)]["granularity"]
            print(f"workload {n} granularity: {time.time() - t:.1f}s sizes {gr['gran']} "
                  f"bytes {gr['bytes']} vs {gr['bytes_default']}", flush=True)
        with open(args.out, "w") as f:
            json.dump(out, f, indent=1)
            f.write("\n")
        return
    ctx = mp.get_context("spawn")
    with ctx.Pool(max(1, os.cpu_count() or 1)) as pool:
        for n in [int(x) for x in args.workloads.split(",")]:
            t = time.time()
            if args.output_aware:
                if WORKLOADS[n].demand_source != "coverage":
                    continue
                out[str(n)]["output_aware"] = profile_output_aware(n, pool)
                oa = out[str(n)]["output_aware"]
                print(f"workload {n} output-aware: {time.time() - t:.1f}s demand "
                      f"{min(oa['demand'])}..{max(oa['demand'])}", flush=True)
                continue
            prev = out.get(str(n), {}).get("output_aware")
            out[str(n)] = profile(n, pool)
            if prev is not None:
                out[str(n)]["output_aware"] = prev
            print(f"workload {n}: {time.time() - t:.1f}s k_u={out[str(n)]['k_uniform']} "
                  f"demand range {min(out[str(n)]['demand'])}..{max(out[str(n)]['demand'])}",
                  flush=True)
    with open(args.out, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
