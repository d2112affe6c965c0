"""The C-ABI library on the CPU: it loads, exports every declared symbol, its
host-only planning matches the oracle bit for bit, and its argument checks
return the documented status codes before anything touches a GPU."""
import ctypes
import json
import os
import random
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sa():
    import __graft_entry__
    __graft_entry__.build()
    import head_heterogeneous_block_gb300 as sa
    return sa


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(sa):
    declared = _declared_functions()
    assert {"sparse_attn_plan", "sparse_attn_score", "sparse_attn_select",
            "sparse_attn_forward"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", sa.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared - exported
    assert not missing, missing
    lib = ctypes.CDLL(sa.library_path())
    for name in declared:
        assert getattr(lib, name)


def _oracle_plan(budgets_from, k_u, demand, k_min, nb, W, policy, G):
    from oracle import plan as op
    k = op.maxmin_shift(k_u, list(demand), k_min, nb) if demand is not None else [k_u] * budgets_from
    wptr, items, loads = op.schedule(k, nb, W, policy, G)
    return k, wptr, items, loads


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("policy", ["lpt", "lpt_grouped", "head_order"])
def test_plan_matches_oracle_random(sa, seed, policy):
    r = random.Random(seed)
    Hkv = r.choice([1, 2, 4])
    Hq = Hkv * r.choice([1, 2, 4])
    B = 64
    nb = r.randint(1, 40)
    W = r.randint(1, 20)
    k_min = 2
    k_u = r.randint(k_min, max(k_min, nb)) if nb >= 2 else None
    if k_u is None:
        return
    demand = [r.randint(0, nb + 3) for _ in range(Hq)] if seed % 3 else None
    shape = sa.Shape.prefill(nb * B, B, Hq, Hkv, 64)
    plan = sa.sparse_attn_plan(shape, k_u, demand=demand, k_min=k_min, num_workers=W,
                               schedule=policy)
    got = plan.get()
    k, wptr, items, loads = _oracle_plan(Hq, k_u, demand, k_min, nb, W, policy, Hq // Hkv)
    assert got["budgets"].tolist() == k
    assert got["wptr"].tolist() == wptr
    assert got["items"].tolist() == items
    assert got["loads"].tolist() == loads
    assert got["makespan"] == max(loads)
    assert got["total_blocks"] == sum(loads)
    assert got["kmax"] == max(min(x, nb) for x in k)


@pytest.mark.parametrize("number", [1, 2, 3, 4])
@pytest.mark.parametrize("policy", ["lpt", "lpt_grouped", "head_order"])
def test_plan_matches_oracle_workloads(sa, number, policy):
    from workloads import workload
    w = workload(number)
    prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))[str(number)]
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    W = 152
    plan = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=prof["demand"],
                               k_min=prof["k_min"], num_workers=W, schedule=policy)
    got = plan.get()
    k, wptr, items, loads = _oracle_plan(w.num_q_heads, prof["k_uniform"], prof["demand"],
                                         prof["k_min"], w.nb, W, policy, w.group)
    assert got["budgets"].tolist() == k == prof["budgets_maxmin"]
    assert got["wptr"].tolist() == wptr
    assert np.array_equal(got["items"], np.array(items, np.int32))
    assert got["loads"].tolist() == loads


def test_plan_lpt_balances(sa):
    from workloads import workload
    w = workload(4)
    prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))["4"]
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    ms = {}
    for pol in ["lpt", "lpt_grouped", "head_order"]:
        ms[pol] = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=prof["demand"],
                                      num_workers=152, schedule=pol).info()
    lower = -(-ms["lpt"]["total_blocks"] // 152)
    assert ms["lpt"]["makespan"] <= lower + 315
    assert ms["lpt_grouped"]["makespan"] <= lower + 8 * 315
    assert ms["head_order"]["makespan"] > 1.5 * ms["lpt"]["makespan"]


def test_decode_plan(sa):
    shape = sa.Shape.decode(65536, 32, 28, 4, 128, 16)
    kinds = np.zeros(28, np.uint8)
    kinds[[1, 5, 9]] = sa.SA_HEAD_STREAMING
    plan = sa.sparse_attn_plan(shape, 64, head_kind=kinds, window_blocks=64, num_workers=1)
    got = plan.get()
    exp = np.where(kinds == 1, 65, 64)
    assert got["budgets"].tolist() == exp.tolist()
    assert got["kmax"] == 65 and got["num_items"] == 16 * 28 and got["num_workers"] == 0
    assert got["total_blocks"] == 16 * int(exp.sum())


def _raw_plan(sa, shape, params):
    out = ctypes.c_void_p()
    st = sa._lib.sparse_attn_plan(ctypes.byref(shape) if shape is not None else None,
                                  ctypes.byref(params) if params is not None else None,
                                  ctypes.byref(out))
    if st == 0:
        sa._lib.sparse_attn_plan_destroy(out)
    return st


def _params(sa, **kw):
    p = sa._PlanParams()
    p.k_uniform, p.k_min, p.num_workers, p.schedule = 4, 2, 8, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_plan_argument_errors(sa):
    good = sa.Shape.prefill(1024, 64, 8, 2, 64)
    assert _raw_plan(sa, good, _params(sa)) == 0
    assert _raw_plan(sa, None, _params(sa)) == 1
    assert _raw_plan(sa, good, None) == 1
    assert _raw_plan(sa, good, _params(sa, k_min=1)) == 1
    assert _raw_plan(sa, good, _params(sa, k_uniform=1)) == 1
    assert _raw_plan(sa, good, _params(sa, k_uniform=17)) == 1          # > nb = 16
    assert _raw_plan(sa, good, _params(sa, num_workers=0)) == 1
    assert _raw_plan(sa, good, _params(sa, schedule=7)) == 1
    assert _raw_plan(sa, sa.Shape.prefill(1000, 64, 8, 2, 64), _params(sa)) == 2   # S % B
    assert _raw_plan(sa, sa.Shape.prefill(1024, 64, 6, 4, 64), _params(sa)) == 2   # Hq % Hkv
    bad = sa.Shape.prefill(1024, 64, 8, 2, 64)
    bad.batch = 2
    assert _raw_plan(sa, bad, _params(sa)) == 2
    neg = (ctypes.c_int32 * 8)(1, 2, 3, -1, 5, 6, 7, 8)
    assert _raw_plan(sa, good, _params(sa, demand=ctypes.cast(neg, ctypes.POINTER(ctypes.c_int32)))) == 1
    kinds = (ctypes.c_uint8 * 8)(*([0] * 8))
    kp = ctypes.cast(kinds, ctypes.POINTER(ctypes.c_uint8))
    assert _raw_plan(sa, good, _params(sa, head_kind=kp)) == 1            # kinds on prefill
    dec = sa.Shape.decode(2048, 32, 8, 2, 128, 2)
    kinds[3] = 1
    assert _raw_plan(sa, dec, _params(sa, head_kind=kp, window_blocks=0)) == 1
    assert _raw_plan(sa, dec, _params(sa, head_kind=kp, window_blocks=4)) == 0
    kinds[2] = 5
    assert _raw_plan(sa, dec, _params(sa, head_kind=kp, window_blocks=4)) == 1
    assert sa.sa_status_string(3) == "unsupported shape or mode"


def test_device_calls_reject_bad_arguments_before_launch(sa):
    shape = sa.Shape.prefill(4096, 64, 8, 2, 64)
    plan = sa.sparse_attn_plan(shape, 9, num_workers=4)
    lib, P = sa._lib, 8192   # P: any non-null, 16-byte aligned fake address
    s = ctypes.byref(shape)
    # null inputs
    assert lib.sparse_attn_score(s, None, P, P, P, 1 << 30, None) == 1
    # workspace too small
    assert lib.sparse_attn_score(s, P, P, P, P, 16, None) == 1
    # unsupported head dim / block
    s96 = sa.Shape.prefill(4096, 64, 8, 2, 96)
    assert lib.sparse_attn_score(ctypes.byref(s96), P, P, P, P, 1 << 30, None) == 3
    s32 = sa.Shape.prefill(4096, 32, 8, 2, 64)
    assert lib.sparse_attn_score(ctypes.byref(s32), P, P, P, P, 1 << 30, None) == 3
    # misaligned pointer
    assert lib.sparse_attn_score(s, P + 2, P, P, P, 1 << 30, None) == 1
    # select: plan not uploaded, kmax too small, shape mismatch
    assert lib.sparse_attn_select(s, plan.handle, P, P, P, 9, None) == 8
    assert lib.sparse_attn_select(s, plan.handle, P, P, P, 8, None) == 2
    other = sa.Shape.prefill(8192, 64, 8, 2, 64)
    assert lib.sparse_attn_select(ctypes.byref(other), plan.handle, P, P, P, 9, None) == 2
    # forward: not uploaded, null status word
    assert lib.sparse_attn_forward(s, plan.handle, P, P, P, P, P, 9, P, 0, None, P, None) == 8
    assert lib.sparse_attn_forward(s, plan.handle, P, P, P, P, P, 9, P, 0, None, None, None) == 1
    assert lib.sparse_attn_forward(s, plan.handle, P, P, P, P, P, 9, P, 3, None, P, None) == 1
    assert lib.sparse_attn_forward(s, None, P, P, P, P, P, 9, P, 1, None, P, None) == 1
    # pool_kcache is decode only
    assert lib.sparse_attn_pool_kcache(s, P, P, None) == 1
    # the per-kind decode calls: prefill plans, unknown kinds, not uploaded
    assert lib.sparse_attn_select_kind(s, plan.handle, P, P, P, 9, 1, None) == 1
    assert lib.sparse_attn_forward_kind(s, plan.handle, P, P, P, P, P, 9, P, 0, None, P, 1,
                                        None) == 1
    dshape = sa.Shape.decode(2048, 32, 8, 2, 128, 2)
    dplan = sa.sparse_attn_plan(dshape, 8, head_kind=[1, 0] * 4, window_blocks=4,
                                num_workers=1)
    ds = ctypes.byref(dshape)
    assert lib.sparse_attn_select_kind(ds, dplan.handle, P, P, P, 16, 2, None) == 1
    assert lib.sparse_attn_select_kind(ds, dplan.handle, None, P, P, 16, 1, None) == 8
    assert lib.sparse_attn_forward_kind(ds, dplan.handle, P, P, P, P, P, 16, P, 0, None, P, 7,
                                        None) == 1
    assert lib.sparse_attn_forward_kind(ds, None, P, P, P, P, P, 16, P, 0, None, P, 0,
                                        None) == 1
    assert lib.sparse_attn_forward_kind(ds, dplan.handle, P, P, P, P, P, 16, P, 0, None, P, 0,
                                        None) == 8
    # fused decode scoring and selection: prefill plans, null or misaligned
    # pointers, kmax below the plan's, unsupported plans, not uploaded
    ss = lib.sparse_attn_score_select
    assert ss(s, plan.handle, P, P, P, P, P, 9, None) == 1
    assert ss(ds, None, P, P, P, P, P, 16, None) == 1
    assert ss(ds, dplan.handle, None, P, P, P, P, 16, None) == 1
    assert ss(ds, dplan.handle, P, P, P, None, P, 16, None) == 1
    assert ss(ds, dplan.handle, P, P + 4, P, P, P, 16, None) == 1
    assert ss(ds, dplan.handle, P, P, P + 8, P, P, 16, None) == 1
    assert ss(ds, dplan.handle, P, P, P, P, P, 3, None) == 2
    assert ss(ctypes.byref(sa.Shape.decode(4096, 32, 8, 2, 128, 2)), dplan.handle, P, P, P, P, P,
              16, None) == 2
    assert ss(ds, dplan.handle, P, P, None, P, P, 16, None) == 8   # scores may be NULL
    d64 = sa.Shape.decode(2048, 32, 8, 2, 64, 2)
    p64 = sa.sparse_attn_plan(d64, 8, head_kind=[0] * 8, num_workers=1)
    assert ss(ctypes.byref(d64), p64.handle, P, P, P, P, P, 16, None) == 3
    sized = sa.sparse_attn_plan(dshape, 8, head_kind=[1, 0] * 4, window_blocks=4, num_workers=1,
                                granularity=[32, 16] * 4, head_budget=[8] * 8)
    assert ss(ds, sized.handle, P, P, P, P, P, sized.info()["kmax"], None) == 3
    # the one-launch decode step: the fused call's checks, plus the attention's
    # (k, v, o and the status word, the output type, block size 32)
    st = lib.sparse_attn_decode_step
    ok = (P, P, P, P, P, P, P, 16, P, 0, None, P, None)

    def step(shape, plan_, *args):
        return st(shape, plan_, *args)

    assert step(ds, dplan.handle, *ok) == 8                                   # not uploaded
    assert step(s, plan.handle, *ok) == 1                                     # prefill plan
    assert step(ds, None, *ok) == 1
    for i in (0, 1, 2, 3, 5, 6, 8, 11):                                      # q kbar k v idx cnt o st
        bad = list(ok)
        bad[i] = None
        assert step(ds, dplan.handle, *bad) == 1, i
    for i in (0, 1, 2, 3, 4, 8):                                             # q kbar k v scores o
        bad = list(ok)
        bad[i] = P + 4
        assert step(ds, dplan.handle, *bad) == 1, i
    bad = list(ok)
    bad[9] = 3                                                               # output type
    assert step(ds, dplan.handle, *bad) == 1
    bad = list(ok)
    bad[7] = 3                                                               # kmax below the plan's
    assert step(ds, dplan.handle, *bad) == 2
    assert step(ctypes.byref(sa.Shape.decode(4096, 32, 8, 2, 128, 2)), dplan.handle, *ok) == 2
    ok64 = list(ok)
    assert step(ctypes.byref(d64), p64.handle, *ok64) == 3                   # d = 64
    assert step(ds, sized.handle, *ok[:7], sized.info()["kmax"], *ok[8:]) == 3
    b64 = sa.Shape.decode(2048, 64, 8, 2, 128, 2)
    p_b64 = sa.sparse_attn_plan(b64, 8, head_kind=[1, 0] * 4, window_blocks=4, num_workers=1)
    assert step(ctypes.byref(b64), p_b64.handle, *ok) == 3                  # block size 64
    n = ctypes.c_size_t()
    assert lib.sparse_attn_score_workspace_size(s, ctypes.byref(n)) == 0
    assert n.value == (8 + 2) * 64 * 64 * 4


@pytest.mark.parametrize("seed", range(12))
def test_group_shared_plan_matches_oracle(sa, seed):
    # one list per KV group: Max-Min shifting between the groups, each with
    # its most demanding head's demand, and the schedule on those budgets
    r = random.Random(100 + seed)
    Hkv = r.choice([1, 2, 4])
    G = r.choice([1, 2, 4, 7])
    Hq = Hkv * G
    B, nb = 64, r.randint(2, 40)
    W = r.randint(1, 20)
    policy = r.choice(["lpt", "lpt_grouped", "head_order"])
    k_u = r.randint(2, nb)
    demand = [r.randint(0, nb + 3) for _ in range(Hq)]
    from oracle import plan as op
    shape = sa.Shape.prefill(nb * B, B, Hq, Hkv, 64)
    share = G % 2 == 0 and r.random() < 0.5   # head pairs on one K/V load
    got = sa.sparse_attn_plan(shape, k_u, demand=demand, num_workers=W, schedule=policy,
                              group_shared=True, share_kv=share).get()
    k = op.group_budgets(k_u, demand, G, 2, nb)
    if share:
        wptr, items, loads = op.pair_schedule(k, nb, W, policy, G)
    else:
        wptr, items, loads = op.schedule(k, nb, W, policy, G)
    assert got["budgets"].tolist() == k
    assert got["wptr"].tolist() == wptr
    assert got["items"].tolist() == items
    assert got["loads"].tolist() == loads


def test_group_shared_is_prefill_only(sa):
    shape = sa.Shape.decode(4096, 32, 8, 2, 128, 2)
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_plan(shape, 8, num_workers=1, group_shared=True)


def test_shared_kv_loads_need_group_shared_lists_and_an_even_group(sa):
    # pairs of heads can share a K/V load only when they share the list
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_plan(sa.Shape.prefill(4096, 64, 8, 2, 64), 8, num_workers=4,
                            share_kv=True)
    with pytest.raises(sa.SparseAttnError):      # G = 3
        sa.sparse_attn_plan(sa.Shape.prefill(4096, 64, 6, 2, 64), 8, num_workers=4,
                            group_shared=True, share_kv=True)
    with pytest.raises(sa.SparseAttnError):
        sa.sparse_attn_plan(sa.Shape.decode(4096, 32, 8, 2, 128, 2), 8, num_workers=1,
                            share_kv=True)
    p = sa.sparse_attn_plan(sa.Shape.prefill(4096, 64, 8, 2, 64), 8, num_workers=4,
                            group_shared=True, share_kv=True)
    assert p.info()["num_items"] == 4 * 64


@pytest.mark.parametrize("number", [1, 2, 3])
def test_output_aware_profile_plans_match_oracle(sa, number):
    # the stored output-aware demands shift to the stored budgets under the
    # oracle's Max-Min, and the library's plan gives the same budgets
    from oracle import plan as op
    from workloads import workload
    prof = json.load(open(os.path.join(ROOT, "workloads", "demands.json")))[str(number)]
    if "output_aware" not in prof:
        pytest.skip("no output-aware profile stored")
    oa = prof["output_aware"]
    w = workload(number)
    k = op.maxmin_shift(prof["k_uniform"], oa["demand"], prof["k_min"], w.nb)
    assert k == oa["budgets_maxmin"]
    assert sum(k) == prof["k_uniform"] * w.num_q_heads
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    got = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=oa["demand"],
                              k_min=prof["k_min"], num_workers=152).get()
    assert got["budgets"].tolist() == k


def test_topp_and_rebuild_reject_bad_arguments_before_launch(sa):
    shape = sa.Shape.prefill(4096, 64, 8, 2, 64)
    plan = sa.sparse_attn_plan(shape, 9, num_workers=4)
    lib, P = sa._lib, 8192
    s = ctypes.byref(shape)
    nb = shape.nb
    # not uploaded; kmax below nb; NaN threshold; null output
    assert lib.sparse_attn_select_topp(s, plan.handle, P, 0.9, P, P, nb, None) == 8
    assert lib.sparse_attn_select_topp(s, plan.handle, P, 0.9, P, P, nb - 1, None) == 2
    assert lib.sparse_attn_select_topp(s, plan.handle, P, float("nan"), P, P, nb, None) == 1
    assert lib.sparse_attn_select_topp(s, plan.handle, P, 0.9, None, P, nb, None) == 1
    # decode shapes have no top-p rows
    dshape = sa.Shape.decode(4096, 32, 8, 2, 128, 2)
    dplan = sa.sparse_attn_plan(dshape, 8, num_workers=1)
    assert lib.sparse_attn_select_topp(ctypes.byref(dshape), dplan.handle, P, 0.9, P, P, 128,
                                       None) == 1
    # rebuild: not uploaded, decode plan, null counts
    assert lib.sparse_attn_plan_rebuild(plan.handle, P, None) == 8
    assert lib.sparse_attn_plan_rebuild(dplan.handle, P, None) == 1
    assert lib.sparse_attn_plan_rebuild(plan.handle, None, None) == 1
    assert lib.sparse_attn_plan_device_schedule(plan.handle, P, P, None) == 8


def test_decode_plan_per_head_block_sizes(sa):
    shape = sa.Shape.decode(65536, 32, 8, 2, 128, 4)
    kinds = np.array([0, 1, 0, 0, 0, 0, 1, 0], np.uint8)
    gran = [16, 8, 64, 128, 16, 32, 999, 64]          # streaming entries are ignored
    budget = [70, 0, 40, 9000, 2, 64, 0, 31]
    plan = sa.sparse_attn_plan(shape, 64, head_kind=kinds, window_blocks=16, num_workers=1,
                               granularity=gran, head_budget=budget)
    got = plan.get()
    nbh = [65536 // g for g in (16, 32, 64, 128, 16, 32, 32, 64)]
    want = [17 if kinds[h] else min(budget[h], nbh[h]) for h in range(8)]
    assert got["budgets"].tolist() == want
    assert got["kmax"] == max(want)
    assert got["total_blocks"] == 4 * sum(want)
    lay = plan.decode_layout()
    assert lay["sizes"] == [16, 32, 64, 128]
    assert lay["score_stride"] == 65536 // 16
    assert lay["kcache_floats"] == sum(4 * 2 * (65536 // g) * 128 for g in (16, 32, 64, 128))
    # without sizes: B for every head, scores of nb per row
    plain = sa.sparse_attn_plan(shape, 64, head_kind=kinds, window_blocks=16, num_workers=1)
    assert plain.decode_layout() == {"sizes": [32], "kcache_floats": 4 * 2 * 2048 * 128,
                                     "score_stride": 2048}


def test_decode_block_size_argument_errors(sa):
    dshape = sa.Shape.decode(65536, 32, 4, 2, 128, 2)
    kinds = np.zeros(4, np.uint8)

    def plan_status(shape, gran=None, budget=None, kinds_=kinds):
        keep = []
        p = _params(sa)
        p.k_uniform, p.num_workers = 8, 1
        for name, arr, ct in (("granularity", gran, ctypes.c_int32),
                              ("head_budget", budget, ctypes.c_int32),
                              ("head_kind", kinds_, ctypes.c_uint8)):
            if arr is not None:
                a = np.ascontiguousarray(arr, dtype=np.int32 if ct is ctypes.c_int32 else np.uint8)
                keep.append(a)
                setattr(p, name, a.ctypes.data_as(ctypes.POINTER(ct)))
        return _raw_plan(sa, shape, p)

    assert plan_status(dshape, [16, 32, 64, 128]) == 0
    assert plan_status(dshape, [8, 32, 32, 32]) == 1          # below 16
    assert plan_status(dshape, [24, 32, 32, 32]) == 1         # not a multiple of 16
    assert plan_status(dshape, [48, 32, 32, 32]) == 1         # does not divide L
    big = sa.Shape.decode(131072, 32, 4, 2, 128, 2)
    assert plan_status(big, [16, 32, 32, 32]) == 1            # 8192 blocks > 4096
    assert plan_status(big, [32, 32, 32, 32]) == 0
    assert plan_status(dshape, None, [8, 1, 8, 8]) == 1       # budget below k_min
    many = sa.Shape.decode(40320, 32, 16, 2, 128, 1)        # 16 * m divides L for m <= 9
    sizes = [16 * m for m in (1, 2, 3, 4, 5, 6, 7, 8, 9)] + [16] * 7
    assert plan_status(many, sizes, None, np.zeros(16, np.uint8)) == 1   # 9 distinct sizes
    assert plan_status(many, sizes[:8] + [16] * 8, None, np.zeros(16, np.uint8)) == 0
    pshape = sa.Shape.prefill(4096, 64, 8, 2, 64)
    p = _params(sa)
    g = np.full(8, 64, np.int32)
    p.granularity = g.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert _raw_plan(sa, pshape, p) == 1                      # prefill plans take none
    pplan = sa.sparse_attn_plan(pshape, 9, num_workers=4)
    with pytest.raises(sa.SparseAttnError):
        pplan.decode_layout()


def test_decode_block_size_calls_reject_bad_arguments_before_launch(sa):
    lib, P = sa._lib, 8192
    dshape = sa.Shape.decode(4096, 32, 4, 2, 128, 2)
    s = ctypes.byref(dshape)
    plan = sa.sparse_attn_plan(dshape, 8, num_workers=1, granularity=[16, 32, 64, 128])
    other = sa.Shape.decode(8192, 32, 4, 2, 128, 2)
    pshape = sa.Shape.prefill(4096, 64, 8, 2, 64)
    pplan = sa.sparse_attn_plan(pshape, 9, num_workers=4)
    assert lib.sparse_attn_pool_kcache_plan(s, None, P, P, None) == 1
    assert lib.sparse_attn_pool_kcache_plan(s, plan.handle, None, P, None) == 1
    assert lib.sparse_attn_pool_kcache_plan(s, plan.handle, P + 4, P, None) == 1
    assert lib.sparse_attn_pool_kcache_plan(ctypes.byref(other), plan.handle, P, P, None) == 2
    assert lib.sparse_attn_pool_kcache_plan(ctypes.byref(pshape), pplan.handle, P, P, None) == 1
    assert lib.sparse_attn_score_plan(s, plan.handle, P, P, P, None) == 8   # not uploaded
    assert lib.sparse_attn_score_plan(s, plan.handle, P, None, P, None) == 1
    assert lib.sparse_attn_score_plan(ctypes.byref(other), plan.handle, P, P, P, None) == 2
    # a forward with sizes needs the plan on the device
    assert lib.sparse_attn_forward(s, plan.handle, P, P, P, P, P, 8, P, 1, None, P, None) == 8


@pytest.mark.parametrize("policy", ["lpt", "lpt_grouped"])
@pytest.mark.parametrize("Hq,Hkv,nb,W,k_u,demand", [
    (2, 1, 3, 50, 2, None),              # more workers than items
    (4, 2, 37, 1, 9, [1, 30, 5, 37]),    # one worker takes everything, in walk order
    (2, 2, 1, 3, 2, None),               # one block per sequence: every cost is 1
    (8, 2, 64, 256, 20, [2, 64, 3, 60, 5, 40, 2, 64]),   # many workers, very unequal budgets
    (16, 4, 200, 152, 31, None),         # long runs of equal cost
])
def test_plan_lpt_edge_cases_match_oracle(sa, policy, Hq, Hkv, nb, W, k_u, demand):
    shape = sa.Shape.prefill(nb * 64, 64, Hq, Hkv, 64)
    plan = sa.sparse_attn_plan(shape, k_u, demand=demand, k_min=2, num_workers=W,
                               schedule=policy)
    got = plan.get()
    k, wptr, items, loads = _oracle_plan(Hq, k_u, demand, 2, nb, W, policy, Hq // Hkv)
    assert got["budgets"].tolist() == k
    assert got["wptr"].tolist() == wptr
    assert got["items"].tolist() == items
    assert got["loads"].tolist() == loads
