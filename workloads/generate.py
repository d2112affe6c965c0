"""Seeded synthetic inputs shared by the CUDA path, the oracle and the bench.

Every array is produced from a counter-free PCG64 stream keyed by
``SeedSequence([seed, tensor_code, *index])`` so any single head (or sequence)
can be regenerated on its own.  Floating-point tensors are drawn in fp32 and
rounded to bfloat16 with round-to-nearest-even; they are returned as the raw
``uint16`` bit patterns so that every consumer reads identical bits.

Nothing here computes a step of the sparse-attention method: pooling,
scoring, selection, budgets, schedules and attention all live elsewhere.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import Workload

# stream codes
_Q, _K, _V, _SCALE, _HEAVY, _KIND, _LOGNORMAL = 1, 2, 3, 10, 11, 12, 13

STREAMING = 1
RETRIEVAL = 0


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


def q_scales(w: Workload, seed: int | None = None) -> np.ndarray:
    """Per-query-head scale s_h, log-uniform in [q_scale_lo, q_scale_hi]."""
    seed = w.seed if seed is None else seed
    u = _rng(seed, _SCALE).random(w.num_q_heads)
    lo, hi = math.log(w.q_scale_lo), math.log(w.q_scale_hi)
    return np.exp(lo + (hi - lo) * u).astype(np.float32)


def heavy_keys(w: Workload, seed: int | None = None):
    """Planted heavy keys: per KV head, ``heavy_keys`` positions and a unit vector."""
    seed = w.seed if seed is None else seed
    pos = np.zeros((w.num_kv_heads, w.heavy_keys), np.int64)
    unit = np.zeros((w.num_kv_heads, w.head_dim), np.float32)
    for g in range(w.num_kv_heads):
        r = _rng(seed, _HEAVY, g)
        pos[g] = np.sort(r.choice(w.seq_len, size=w.heavy_keys, replace=False))
        v = r.standard_normal(w.head_dim)
        unit[g] = (v / np.linalg.norm(v)).astype(np.float32)
    return pos, unit


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def prefill_inputs(w: Workload, tensors: str = "qkv", heads=None, kv_heads=None,
                   seed: int | None = None, seq_len: int | None = None) -> dict:
    """Q [Hq,S,d], K and V [Hkv,S,d] as bfloat16 bit patterns.

    ``heads`` / ``kv_heads`` restrict generation to a subset (the arrays then
    hold only those heads, in the given order).  ``seed`` and ``seq_len``
    override the workload's for the random values only (the calibration draw
    uses ``w.calib_seed`` at a capped length); the heads themselves -- their
    scales s_h and planted heavy keys -- always come from ``w.seed``, so a
    calibration draw profiles the same heads on different data.
    """
    seed = w.seed if seed is None else seed
    S = w.seq_len if seq_len is None else seq_len
    d = w.head_dim
    heads = list(range(w.num_q_heads)) if heads is None else list(heads)
    kv_heads = list(range(w.num_kv_heads)) if kv_heads is None else list(kv_heads)
    scale = q_scales(w)
    if w.heavy_keys:
        hpos, hunit = heavy_keys(w)
        hpos = [p[p < S] for p in hpos]
    out = {}
    jobs = []
    if "q" in tensors:
        out["q"] = np.empty((len(heads), S, d), np.uint16)
        jobs += [("q", n, h) for n, h in enumerate(heads)]
    if "k" in tensors:
        out["k"] = np.empty((len(kv_heads), S, d), np.uint16)
        jobs += [("k", n, g) for n, g in enumerate(kv_heads)]
    if "v" in tensors:
        out["v"] = np.empty((len(kv_heads), S, d), np.uint16)
        jobs += [("v", n, g) for n, g in enumerate(kv_heads)]
    G = w.group

    def run(job):
        t, n, h = job
        code = {"q": _Q, "k": _K, "v": _V}[t]
        z = np.empty((S, d), np.float32)
        _rng(seed, code, h).standard_normal(dtype=np.float32, out=z)
        if t == "q":
            if w.heavy_keys:
                z += hunit[h // G][None, :]
            z *= scale[h]
        elif t == "k" and w.heavy_keys:
            z[hpos[h]] += np.float32(4.0 * math.sqrt(d)) * hunit[h][None, :]
        out[t][n] = bf16_bits(z)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(run, jobs))
    return out


def head_kinds(w: Workload, seed: int | None = None) -> np.ndarray:
    """Decode head kinds: a seeded permutation; the first floor(f*Hq) stream."""
    seed = w.seed if seed is None else seed
    perm = _rng(seed, _KIND).permutation(w.num_q_heads)
    n_stream = int(math.floor(w.streaming_fraction * w.num_q_heads))
    kinds = np.full(w.num_q_heads, RETRIEVAL, np.uint8)
    kinds[perm[:n_stream]] = STREAMING
    return kinds


def decode_inputs(w: Workload, tensors: str = "qkv", batches=None,
                  seed: int | None = None) -> dict:
    """q [Bt,Hq,d]; K and V [Bt,Hkv,L,d] (bfloat16 bits).

    The cache already holds the new token at position L-1.
    """
    seed = w.seed if seed is None else seed
    L, d = w.seq_len, w.head_dim
    batches = list(range(w.batch)) if batches is None else list(batches)
    scale = q_scales(w)
    out = {}
    jobs = []
    if "q" in tensors:
        out["q"] = np.empty((len(batches), w.num_q_heads, d), np.uint16)
        jobs += [("q", n, b, 0) for n, b in enumerate(batches)]
    for t in "kv":
        if t in tensors:
            out[t] = np.empty((len(batches), w.num_kv_heads, L, d), np.uint16)
            jobs += [(t, n, b, g) for n, b in enumerate(batches)
                     for g in range(w.num_kv_heads)]

    def run(job):
        t, n, b, g = job
        if t == "q":
            z = _rng(seed, _Q, b).standard_normal((w.num_q_heads, d), dtype=np.float32)
            z *= scale[:, None]
            out["q"][n] = bf16_bits(z)
        else:
            z = np.empty((L, d), np.float32)
            _rng(seed, _K if t == "k" else _V, b, g).standard_normal(dtype=np.float32, out=z)
            out[t][n, g] = bf16_bits(z)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(run, jobs))
    return out


def lognormal_densities(w: Workload, seed: int | None = None) -> np.ndarray:
    """Per-head target densities rho_h ~ LogNormal(ln(mean) - sigma^2/2, sigma)."""
    seed = w.seed if seed is None else seed
    s = w.lognormal_sigma
    mu = math.log(w.target_density) - 0.5 * s * s
    return _rng(seed, _LOGNORMAL).lognormal(mu, s, w.num_q_heads)
