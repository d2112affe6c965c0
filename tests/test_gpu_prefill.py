"""GPU parity of the prefill path (score -> select -> forward) against the
oracle, through the C ABI.  Small cases are checked element by element; the
full-size workloads run in the bench's launch configuration (one CTA per SM,
LPT schedule) and are checked in full for plan, scores and selection and on
sampled items for attention."""
import json
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import head_heterogeneous_block_gb300 as sa
    return sa, torch


def _run(sa, torch, w, x, budgets_args, schedule="lpt", workers=None, with_lse=True,
         out_dtype="float32"):
    from head_heterogeneous_block_gb300.layer import PrefillLayer
    from tests._parity import to_dev
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    layer = PrefillLayer(shape, schedule=schedule, num_workers=workers, with_lse=with_lse,
                         out_dtype=getattr(torch, out_dtype), **budgets_args)
    t = {n: to_dev(x[n]) for n in "qkv"}
    out = layer(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    H, nb, S = w.num_q_heads, w.nb, w.seq_len
    res = {
        "status": int(layer.dev_status.item()),
        "scores": layer.scores.view(H, nb, nb).cpu().numpy(),
        "idx": layer.idx.view(H, nb, layer.kmax).cpu().numpy(),
        "cnt": layer.cnt.view(H, nb).cpu().numpy(),
        "out": out.float().cpu().numpy(),
        "lse": layer.lse.view(H, S).cpu().numpy() if with_lse else None,
        "budgets": layer.plan.get()["budgets"].tolist(),
        "layer": layer, "tensors": t,
    }
    return res


def _oracle_scores(w, x):
    from oracle import attention as oa
    from tests._parity import pooled
    return oa.block_scores(pooled(x["q"], w.block), pooled(x["k"], w.block), w.group)


SMALL = [
    # (workload number, seq_len, Hq, Hkv, budget mode)
    (1, 4096, 8, 2, "calibrated"),
    (1, 1024, 8, 8, "uniform"),        # G = 1
    (1, 64, 4, 1, "uniform"),          # nb = 1
    (1, 2368, 8, 2, "uniform"),        # nb = 37: ragged score tiles
    (2, 4096, 8, 2, "shifted"),
    (2, 8192, 16, 4, "shifted"),
]


@pytest.mark.parametrize("out_dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("number,S,Hq,Hkv,mode", SMALL)
def test_prefill_small_full_parity(env, number, S, Hq, Hkv, mode, out_dtype):
    sa, torch = env
    from oracle import plan as op
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(number), S, Hq, Hkv)
    x = generate.prefill_inputs(w)
    nb = w.nb
    if mode == "calibrated":
        prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))[str(number)]
        args = {"k_uniform": prof["k_uniform"], "demand": prof["demand"]}
    elif mode == "uniform":
        args = {"k_uniform": max(2, min(nb, op.budget_for_density(w.target_density, nb)))}
    else:
        k_u = op.budget_for_density(w.target_density, nb)
        rng = np.random.default_rng(S)
        args = {"k_uniform": k_u, "demand": rng.integers(1, nb, Hq).tolist()}
    r = _run(sa, torch, w, x, args, workers=16, out_dtype=out_dtype)
    assert r["status"] == 0
    ref_scores = _oracle_scores(w, x)
    P.check_scores(r["scores"], ref_scores)
    P.check_selection(r["idx"], r["cnt"], ref_scores, r["budgets"])
    P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block,
                      range(Hq * nb), w.group, bf16_out=out_dtype == "bfloat16")


@pytest.mark.parametrize("budget", ["dense", "sink_diag"])
def test_prefill_special_cases(env, budget):
    """k >= nb is dense causal attention; k = 2 keeps only sink + diagonal."""
    sa, torch = env
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 4096, 4, 2)
    x = generate.prefill_inputs(w)
    k = w.nb if budget == "dense" else 2
    r = _run(sa, torch, w, x, {"k_uniform": k}, workers=7)
    assert r["status"] == 0
    for h in range(w.num_q_heads):
        for i in range(w.nb):
            exp = list(range(i + 1)) if budget == "dense" else sorted({0, i})
            assert r["idx"][h, i, :r["cnt"][h, i]].tolist() == exp
    P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block,
                      range(w.num_q_heads * w.nb), w.group)
    if budget == "dense":
        # against the library's dense causal attention as well
        t = r["tensors"]
        ref = torch.nn.functional.scaled_dot_product_attention(
            t["q"].float()[None], t["k"].float().repeat_interleave(w.group, 0)[None],
            t["v"].float().repeat_interleave(w.group, 0)[None], is_causal=True)[0]
        assert float((ref - torch.from_numpy(r["out"]).cuda()).abs().max()) < 1e-2


def test_schedules_give_identical_outputs(env):
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 8192, 8, 2)
    x = generate.prefill_inputs(w)
    rng = np.random.default_rng(5)
    args = {"k_uniform": 13, "demand": rng.integers(1, w.nb, 8).tolist()}
    outs = {}
    for sched, W in [("lpt", 152), ("lpt_grouped", 152), ("head_order", 152), ("lpt", 1),
                     ("head_order", 300)]:
        r = _run(sa, torch, w, x, args, schedule=sched, workers=W)
        assert r["status"] == 0
        outs[(sched, W)] = r["out"]
    ref = outs[("lpt", 152)]
    for key, o in outs.items():
        assert np.array_equal(o, ref), key


def test_corrupt_indices_are_flagged_not_dereferenced(env):
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(1), 2048, 4, 2)
    x = generate.prefill_inputs(w)
    r = _run(sa, torch, w, x, {"k_uniform": 6}, workers=4)
    layer, t = r["layer"], r["tensors"]
    assert r["status"] == 0
    idx = layer.idx.view(w.num_q_heads, w.nb, layer.kmax)
    cnt = layer.cnt.view(w.num_q_heads, w.nb)
    idx[1, 20, 2] = 1 << 28          # far out of range
    idx[2, 5, 1] = -7
    cnt[3, 9] = layer.kmax + 50      # count beyond the row stride
    layer.dev_status.zero_()
    layer.attend(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    st = int(layer.dev_status.item())
    assert st & sa.SA_DEV_BAD_INDEX and st & sa.SA_DEV_BAD_COUNT
    assert not st & sa.SA_DEV_TIMEOUT
    assert torch.isfinite(layer.out.float()).all()


@pytest.mark.parametrize("factor,exact", [(3.0, False), (5.0, False), (30.0, True)])
def test_later_blocks_scoring_far_above_the_first(env, factor, exact):
    """The forward takes each row's reference maximum from the item's first
    block and keeps it; a later block that scores higher only makes the
    weights exceed 1.  A key planted along one query (k = factor * q) makes
    its block score about factor * |q|^2 / sqrt(d) above the rest: 2^69 with
    factor 3 and 2^116 with factor 5, both on the tensor-core pass (the sum
    stays below 2^126); with factor 30 the weights overflow and every
    affected item is recomputed exactly.  All must match the oracle at the
    plain tolerance, output and log-sum-exp."""
    sa, torch = env
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 4096, 8, 2)
    x = generate.prefill_inputs(w)
    h, i, r, j, u = 1, 20, 5, 10, 7          # query row (h, 128 i + r); key 128 j + u
    q_row = generate.bf16_to_f32(x["q"][h, i * w.block + r])
    k = x["k"].copy()
    k[h // w.group, j * w.block + u] = generate.bf16_bits(q_row * factor)
    x = dict(x, k=k)
    rr = _run(sa, torch, w, x, {"k_uniform": w.nb}, workers=16)
    assert rr["status"] == 0
    assert rr["idx"][h, i, j] == j
    P.check_attention(rr["out"], rr["lse"], x, rr["idx"], rr["cnt"], w.block,
                      range(w.num_q_heads * w.nb), w.group)
    s_jump = float(q_row @ generate.bf16_to_f32(k[h // w.group, j * w.block + u]))
    assert (s_jump / np.sqrt(w.head_dim) / np.log(2) > 140) == exact


@pytest.mark.parametrize("pairs", [False, True])
def test_wait_timeout_is_reported_and_the_context_stays_usable(env, pairs):
    """The forward's watchdog: with every wait limited to 100 ns (far below
    the latency of the first copy from memory), waits run out on every CTA.
    The launch must report SA_DEV_TIMEOUT and return; each CTA drains its own
    copies and tensor-core operations and frees its tensor memory, so a normal
    launch right after, on every SM, gives the same output as before."""
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(1), 4096)
    x = generate.prefill_inputs(w)
    W = torch.cuda.get_device_properties(0).multi_processor_count
    r = _run(sa, torch, w, x, {"k_uniform": 9, "group_shared": pairs, "share_kv": pairs},
             workers=W)
    layer, t = r["layer"], r["tensors"]
    assert r["status"] == 0
    want = layer.out.clone()
    try:
        sa.sparse_attn_set_wait_limit(100)
        layer.dev_status.zero_()
        layer.out.fill_(float("nan"))
        layer.attend(t["q"], t["k"], t["v"])
        torch.cuda.synchronize()
        st = int(layer.dev_status.item())
    finally:
        sa.sparse_attn_set_wait_limit(0)
    assert st & sa.SA_DEV_TIMEOUT, st
    assert not st & (sa.SA_DEV_BAD_INDEX | sa.SA_DEV_BAD_COUNT | sa.SA_DEV_BAD_ITEM)
    for _ in range(2):
        layer.dev_status.zero_()
        layer.out.fill_(float("nan"))
        layer.attend(t["q"], t["k"], t["v"])
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        assert torch.equal(layer.out, want)


FULL = [2, 3, 4]


@pytest.mark.parametrize("number", FULL)
def test_prefill_full_size(env, number):
    """Full-size workloads in the bench's launch configuration: fp32 output at
    the plain tolerance on the main sample, then bf16 output (the bench's) on
    a smaller one."""
    sa, torch = env
    from oracle import attention as oa
    from tests import _parity as P
    from workloads import generate, workload
    w = workload(number)
    prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))[str(number)]
    x = generate.prefill_inputs(w)
    W = torch.cuda.get_device_properties(0).multi_processor_count
    for out_dtype, per_head in (("float32", 16 if number == 4 else 64),
                                ("bfloat16", 4 if number == 4 else 8)):
        r = _run(sa, torch, w, x, {"k_uniform": prof["k_uniform"], "demand": prof["demand"]},
                 schedule="lpt_grouped", workers=W, out_dtype=out_dtype)
        assert r["status"] == 0
        assert r["budgets"] == prof["budgets_maxmin"]
        if out_dtype == "float32":
            ref_scores = oa.block_scores(P.pooled(x["q"], w.block), P.pooled(x["k"], w.block),
                                         w.group)
            # scores: all rows of a sample of heads; selection: every row
            heads = sorted({0, w.num_q_heads - 1, 5 % w.num_q_heads})
            P.check_scores(r["scores"][heads], ref_scores[heads])
            P.check_selection(r["idx"], r["cnt"], ref_scores, r["budgets"])
            del ref_scores
        items = P.sample_items(r["budgets"], w.nb, per_head, seed=number)
        P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block, items, w.group,
                          bf16_out=out_dtype == "bfloat16")
        del r
        torch.cuda.empty_cache()


def _check_group_shared(r, x, w, k_uniform, demand):
    """Group-shared selection: one list per (KV group, row), equal across the
    group's heads, matching the oracle's selection on the group-pooled scores;
    attention checked on the GPU's own lists."""
    from oracle import attention as oa
    from oracle import plan as op
    from tests import _parity as P
    G, nb = w.group, w.nb
    assert r["budgets"] == op.group_budgets(k_uniform, demand, G, 2, nb)
    idx, cnt = r["idx"], r["cnt"]
    for g in range(w.num_kv_heads):
        for hh in range(1, G):
            assert np.array_equal(idx[g * G], idx[g * G + hh])
            assert np.array_equal(cnt[g * G], cnt[g * G + hh])
    ref_scores = _oracle_scores(w, x)
    P.check_scores(r["scores"], ref_scores)
    per_head = np.repeat(oa.group_scores(ref_scores, G), G, axis=0)
    P.check_selection(idx, cnt, per_head, r["budgets"])
    return ref_scores


@pytest.mark.parametrize("number,S,Hq,Hkv", [(1, 4096, 8, 2), (2, 4096, 8, 2), (2, 2432, 8, 8),
                                             (2, 8192, 16, 4), (2, 4096, 8, 4), (1, 2368, 16, 2)])
def test_prefill_group_shared_parity(env, number, S, Hq, Hkv):
    """Group-shared lists, one query head per item; with an even G also head
    pairs, one K/V block load feeding both heads' tiles."""
    sa, torch = env
    from oracle import plan as op
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(number), S, Hq, Hkv)
    x = generate.prefill_inputs(w)
    nb = w.nb
    k_u = max(2, op.budget_for_density(w.target_density, nb))
    rng = np.random.default_rng(S + 7)
    demand = rng.integers(1, nb, Hq).tolist()
    for share in ([False, True] if w.group % 2 == 0 else [False]):
        r = _run(sa, torch, w, x, {"k_uniform": k_u, "demand": demand, "group_shared": True,
                                   "share_kv": share}, workers=16)
        assert r["status"] == 0
        _check_group_shared(r, x, w, k_u, demand)
        P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block, range(Hq * nb),
                          w.group)


def test_prefill_group_shared_dense_pairs_equal_causal_attention(env):
    # every block kept: the pair kernel's output is dense causal attention for
    # every head, against the library's SDPA as well as the oracle
    sa, torch = env
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 4096, 8, 2)
    x = generate.prefill_inputs(w)
    r = _run(sa, torch, w, x, {"k_uniform": w.nb, "group_shared": True, "share_kv": True},
             workers=11)
    assert r["status"] == 0
    assert r["layer"].plan.info()["num_items"] == w.num_q_heads // 2 * w.nb
    P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block,
                      range(w.num_q_heads * w.nb), w.group)
    t = r["tensors"]
    ref = torch.nn.functional.scaled_dot_product_attention(
        t["q"].float()[None], t["k"].float().repeat_interleave(w.group, 0)[None],
        t["v"].float().repeat_interleave(w.group, 0)[None], is_causal=True)[0]
    assert float((ref - torch.from_numpy(r["out"]).cuda()).abs().max()) < 1e-2


def test_prefill_group_shared_full_size(env):
    """The 128K Llama-3.1-8B workload with one list per KV group, in the
    bench's launch configuration; selection checked on every row, attention on
    sampled items (fp32 output at the plain tolerance, then bf16 output, then
    fp32 output from head pairs on one K/V load)."""
    sa, torch = env
    from tests import _parity as P
    from workloads import generate, workload
    w = workload(3)
    prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))["3"]
    x = generate.prefill_inputs(w)
    W = torch.cuda.get_device_properties(0).multi_processor_count
    for out_dtype, per_head, pairs in (("float32", 32, False), ("bfloat16", 8, False),
                                       ("float32", 8, True)):
        r = _run(sa, torch, w, x, {"k_uniform": prof["k_uniform"], "demand": prof["demand"],
                                   "group_shared": True, "share_kv": pairs},
                 schedule="lpt_grouped", workers=W, out_dtype=out_dtype)
        assert r["status"] == 0
        if out_dtype == "float32" and not pairs:
            _check_group_shared(r, x, w, prof["k_uniform"], prof["demand"])
        items = P.sample_items(r["budgets"], w.nb, per_head, seed=33)
        P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block, items, w.group,
                          bf16_out=out_dtype == "bfloat16")
        del r
        torch.cuda.empty_cache()


def test_prefill_largest_rows(env):
    """d 64 / B 64 at 131072 tokens: rows of nb = 2048 blocks, the largest the
    select kernel takes; selection checked on every row, attention sampled."""
    sa, torch = env
    from oracle import plan as op
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(1), 131072, 4, 1)
    assert w.nb == 2048
    x = generate.prefill_inputs(w)
    k_u = op.budget_for_density(0.02, w.nb)
    rng = np.random.default_rng(2048)
    args = {"k_uniform": k_u, "demand": rng.integers(2, 4 * k_u, w.num_q_heads).tolist()}
    r = _run(sa, torch, w, x, args, workers=152, out_dtype="float32")
    assert r["status"] == 0
    ref_scores = _oracle_scores(w, x)
    P.check_scores(r["scores"], ref_scores)
    P.check_selection(r["idx"], r["cnt"], ref_scores, r["budgets"])
    items = P.sample_items(r["budgets"], w.nb, 24, seed=2048)
    P.check_attention(r["out"], r["lse"], x, r["idx"], r["cnt"], w.block, items, w.group)


def test_host_pipeline_matches_the_layer_step_by_step(env):
    # overlapped host copies change only when data moves, never the result:
    # each step's output equals the layer run on that step's inputs alone
    sa, torch = env
    from head_heterogeneous_block_gb300.layer import HostPipeline, PrefillLayer
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 4096, 8, 2)
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    layer = PrefillLayer(shape, 9)
    steps, want = [], []
    for seed in (11, 12, 13, 14, 15):
        x = generate.prefill_inputs(w, seed=seed)
        host = {n: torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).pin_memory()
                for n in "qkv"}
        o = torch.empty(w.num_q_heads, w.seq_len, w.head_dim, dtype=torch.bfloat16,
                        pin_memory=True)
        steps.append((host["q"], host["k"], host["v"], o))
        ref = layer(*(host[n].cuda() for n in "qkv")).cpu()
        torch.cuda.synchronize()
        want.append(ref)
    HostPipeline(layer).run(steps)
    for (_, _, _, o), ref in zip(steps, want):
        assert torch.equal(o, ref)
    assert int(layer.dev_status.item()) == 0
