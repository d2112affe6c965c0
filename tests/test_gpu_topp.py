"""GPU parity of top-p selection and of the LPT schedule rebuilt on the device
from its block counts, through the C ABI, against the oracle."""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MASS_TOL = 1e-4        # fp32 softmax + 2^-32 fixed point vs fp64, at the p boundary
TIE_REL = 1e-3         # near-equal scores may swap across the last kept block


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import head_heterogeneous_block_gb300 as sa
    return sa, torch


def check_topp_row(gsel, scores_row, i, p):
    from oracle import attention as oa
    prob = oa.block_probabilities(scores_row, i)
    mand = sorted({0, i})
    g = [int(x) for x in gsel]
    assert g == sorted(set(g)) and all(0 <= j <= i for j in g)
    assert set(mand) <= set(g), (i, g)
    rest = [j for j in g if j not in mand]
    cand = np.arange(1, i)
    order = [int(j) for j in cand[np.lexsort((cand, -prob[cand]))]] if i >= 2 else []
    n = len(rest)
    if n:
        thr = prob[order[n - 1]]
        for j in set(rest) ^ set(order[:n]):
            assert abs(prob[j] - thr) <= TIE_REL * thr, (i, j, prob[j], thr)
    base = prob[mand].sum()
    mass_n = base + prob[order[:n]].sum()
    assert mass_n >= p - MASS_TOL or n == len(order), (i, n, mass_n, p)
    if n > 0:
        mass_prev = base + prob[order[:n - 1]].sum()
        assert mass_prev < p + MASS_TOL, (i, n, mass_prev, p)


def _setup(sa, torch, w, x, W, schedule="lpt"):
    from head_heterogeneous_block_gb300.layer import PrefillLayer
    from tests._parity import to_dev
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    layer = PrefillLayer(shape, max(2, min(w.nb, 4)), num_workers=W, schedule=schedule,
                         with_lse=True, out_dtype=torch.float32)
    t = {n: to_dev(x[n]) for n in "qkv"}
    layer.score(t["q"], t["k"])
    nb = w.nb
    idx = torch.empty(w.num_q_heads * nb * nb, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.num_q_heads * nb, dtype=torch.int32, device="cuda")
    return shape, layer, t, idx, cnt


def _device_schedule(torch, layer, W, N):
    wptr = torch.empty(W + 1, dtype=torch.int32, device="cuda")
    items = torch.empty(N, dtype=torch.int32, device="cuda")
    layer.plan.device_schedule(wptr, items)
    torch.cuda.synchronize()
    return wptr.cpu().tolist(), items.cpu().tolist()


@pytest.mark.parametrize("number,S,Hq,Hkv,p", [(2, 4096, 8, 2, 0.3), (2, 4096, 8, 2, 0.9),
                                               (1, 4096, 8, 2, 0.6), (2, 8192, 16, 4, 0.06)])
def test_topp_selection_and_device_rebuild(env, number, S, Hq, Hkv, p):
    sa, torch = env
    from oracle import attention as oa
    from oracle import plan as op
    from tests import _parity as P
    from workloads import generate, scaled, workload
    w = scaled(workload(number), S, Hq, Hkv)
    x = generate.prefill_inputs(w)
    nb = w.nb
    W = 16
    shape, layer, t, idx, cnt = _setup(sa, torch, w, x, W)
    sa.sparse_attn_select_topp(shape, layer.plan, layer.scores, p, idx, cnt, nb)
    layer.plan.rebuild(cnt)
    out = torch.empty(Hq, S, w.head_dim, dtype=torch.float32, device="cuda")
    lse = torch.empty(Hq * S, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.sparse_attn_forward(shape, layer.plan, t["q"], t["k"], t["v"], idx, cnt, nb, out, lse,
                           status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g_idx = idx.view(Hq, nb, nb).cpu().numpy()
    g_cnt = cnt.view(Hq, nb).cpu().numpy()
    ref_scores = oa.block_scores(P.pooled(x["q"], w.block), P.pooled(x["k"], w.block), w.group)
    for h in range(Hq):
        for i in range(nb):
            assert np.all(g_idx[h, i, g_cnt[h, i]:] == -1)
            check_topp_row(g_idx[h, i, :g_cnt[h, i]], ref_scores[h, i], i, p)
    # the device schedule is exactly the oracle's LPT on the GPU's own counts,
    # each worker's list in item order
    wptr, items = _device_schedule(torch, layer, W, Hq * nb)
    want_wptr, want_items, _ = op.schedule_from_costs(g_cnt.reshape(-1).tolist(), W,
                                                      within="item")
    assert wptr == want_wptr and items == want_items
    P.check_attention(out.cpu().numpy(), lse.view(Hq, S).cpu().numpy(), x, g_idx, g_cnt,
                      w.block, range(Hq * nb), w.group)


@pytest.mark.parametrize("W", [1, 7, 152, 256])
def test_device_rebuild_matches_oracle_lpt(env, W):
    # arbitrary counts (not from a selection) exercise ties and ragged workers
    sa, torch = env
    from oracle import plan as op
    shape = sa.Shape.prefill(8192, 128, 8, 2, 128)
    plan = sa.sparse_attn_plan(shape, 4, num_workers=W)
    plan.upload()
    nb = shape.nb
    rng = np.random.default_rng(W)
    costs = np.minimum(rng.integers(1, 9, 8 * nb), np.tile(np.arange(1, nb + 1), 8))
    cnt = torch.from_numpy(costs.astype(np.int32)).cuda()
    plan.rebuild(cnt)
    wptr = torch.empty(W + 1, dtype=torch.int32, device="cuda")
    items = torch.empty(8 * nb, dtype=torch.int32, device="cuda")
    plan.device_schedule(wptr, items)
    torch.cuda.synchronize()
    want_wptr, want_items, _ = op.schedule_from_costs(costs.tolist(), W, within="item")
    assert wptr.cpu().tolist() == want_wptr
    assert items.cpu().tolist() == want_items


@pytest.mark.parametrize("W,kind", [(152, "mixed"), (256, "equal"), (37, "wide")])
def test_device_rebuild_full_size_and_clamped_counts(env, W, kind):
    # 32 heads x 1024 query blocks: long runs of equal cost, zero-cost items,
    # and counts outside [0, 2048], which the rebuild clamps to that range
    sa, torch = env
    from oracle import plan as op
    shape = sa.Shape.prefill(131072, 128, 32, 8, 128)
    plan = sa.sparse_attn_plan(shape, 4, num_workers=W)
    plan.upload()
    n = 32 * shape.nb
    rng = np.random.default_rng(W)
    if kind == "mixed":
        costs = rng.integers(1, 64, n)
        costs[rng.random(n) < 0.05] = 0
        costs[rng.random(n) < 0.01] = -3
        costs[rng.random(n) < 0.01] = 5000
    elif kind == "equal":
        costs = np.ones(n, dtype=np.int64)
    else:
        costs = rng.integers(1, 2049, n)
    cnt = torch.from_numpy(costs.astype(np.int32)).cuda()
    plan.rebuild(cnt)
    wptr = torch.empty(W + 1, dtype=torch.int32, device="cuda")
    items = torch.empty(n, dtype=torch.int32, device="cuda")
    plan.device_schedule(wptr, items)
    torch.cuda.synchronize()
    want_wptr, want_items, _ = op.schedule_from_costs(np.clip(costs, 0, 2048).tolist(), W,
                                                      within="item")
    assert wptr.cpu().tolist() == want_wptr
    assert items.cpu().tolist() == want_items


def test_topp_rebuilt_schedule_gives_the_same_output_as_a_static_one(env):
    # the schedule changes only where items run, never their result
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(2), 8192, 8, 2)
    x = generate.prefill_inputs(w)
    nb = w.nb
    outs = []
    for rebuild in (False, True):
        shape, layer, t, idx, cnt = _setup(sa, torch, w, x, 16, schedule="head_order")
        sa.sparse_attn_select_topp(shape, layer.plan, layer.scores, 0.5, idx, cnt, nb)
        if rebuild:
            layer.plan.rebuild(cnt)
        out = torch.empty(8, w.seq_len, w.head_dim, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sa.sparse_attn_forward(shape, layer.plan, t["q"], t["k"], t["v"], idx, cnt, nb, out,
                               None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
