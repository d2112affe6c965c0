"""GPU parity of the decode step (pooled key cache -> scores -> select ->
attention) against the oracle, through the C ABI."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import head_heterogeneous_block_gb300 as sa
    return sa, torch


def _decode(sa, torch, w, x, kinds, budget, window, out_dtype="float32", one_launch=False):
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    step = DecodeStep(shape, budget, kinds, window, with_lse=True,
                      out_dtype=getattr(torch, out_dtype), one_launch=one_launch)
    t = {n: to_dev(x[n]) for n in "qkv"}
    step.build_cache(t["k"])
    out = step(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    Bt, H, nb = w.batch, w.num_q_heads, w.nb
    return {
        "status": int(step.dev_status.item()),
        "kbar": step.kbar.view(Bt, w.num_kv_heads, nb, w.head_dim).cpu().numpy(),
        "scores": step.scores.view(Bt, H, nb).cpu().numpy(),
        "idx": step.idx.view(Bt, H, step.kmax).cpu().numpy(),
        "cnt": step.cnt.view(Bt, H).cpu().numpy(),
        "out": out.float().cpu().numpy(),
        "lse": step.lse.view(Bt, H).cpu().numpy(),
    }


def _check(w, x, r, kinds, budget, window, bf16_out=False):
    from oracle import decode as od
    from tests import _parity as P
    from workloads import generate
    assert r["status"] == 0
    nb = w.nb
    for b in range(w.batch):
        kb = od.pool_cache(generate.bf16_to_f32(x["k"][b:b + 1]), w.block)
        np.testing.assert_allclose(r["kbar"][b], kb[0], rtol=1e-5, atol=1e-6)
        sc = od.decode_scores(generate.bf16_to_f64(x["q"][b:b + 1]), kb)[0]
        # the retrieval heads' scores (the fused step writes no others)
        ret = kinds != 1
        np.testing.assert_allclose(r["scores"][b][ret], sc[ret], rtol=1e-4, atol=1e-6)
        for h in range(w.num_q_heads):
            sel = r["idx"][b, h, :r["cnt"][b, h]]
            assert all(v == -1 for v in r["idx"][b, h, r["cnt"][b, h]:])
            if kinds[h] == 1:
                assert sel.tolist() == od.streaming_blocks(nb, window)
            else:
                from oracle.attention import select_row
                ref = select_row(sc[h], nb - 1, budget)
                P.check_selection_row(sel, ref, sc[h], nb - 1)
        o, lse = od.decode_attend(generate.bf16_to_f64(x["q"][b:b + 1]),
                                  generate.bf16_to_f32(x["k"][b:b + 1]),
                                  generate.bf16_to_f32(x["v"][b:b + 1]),
                                  r["idx"][b:b + 1], r["cnt"][b:b + 1], w.block)
        d_max, d_rel = P.output_errors(r["out"][b], o[0], bf16_out)
        assert d_max.max() <= P.MAX_ABS, d_max.max()
        assert d_rel.sum() / np.abs(o[0]).sum() <= P.MEAN_REL
        assert np.abs(r["lse"][b] - lse[0]).max() <= P.LSE_ABS


@pytest.mark.parametrize("L,Bt,budget,window", [(4096, 2, 16, 8), (2048, 3, 64, 64),
                                                (1024, 1, 32, 32)])
def test_decode_small(env, L, Bt, budget, window):
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(5), L, batch=Bt)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    for out_dtype in ("float32", "bfloat16"):
        for one_launch in (False, True):
            r = _decode(sa, torch, w, x, kinds, budget, window, out_dtype, one_launch)
            _check(w, x, r, kinds, budget, window, bf16_out=out_dtype == "bfloat16")


def test_decode_full_size(env):
    sa, torch = env
    from workloads import generate, workload
    w = workload(5)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    budget = w.budget_tokens // w.block
    window = w.window_tokens // w.block
    # fp32 output at the plain tolerance, then bf16 output as well; the
    # separate launches, then the one-launch step
    for out_dtype in ("float32", "bfloat16"):
        for one_launch in (False, True):
            r = _decode(sa, torch, w, x, kinds, budget, window, out_dtype, one_launch)
            _check(w, x, r, kinds, budget, window, bf16_out=out_dtype == "bfloat16")


def _decode_sized(sa, torch, w, x, kinds, gran, budget, window, out_dtype="float32"):
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    step = DecodeStep(shape, 2, kinds, window, with_lse=True,
                      out_dtype=getattr(torch, out_dtype), granularity=gran, head_budget=budget)
    t = {n: to_dev(x[n]) for n in "qkv"}
    step.build_cache(t["k"])
    out = step(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    Bt, H = w.batch, w.num_q_heads
    return {
        "status": int(step.dev_status.item()),
        "layout": step.plan.decode_layout(),
        "kbar": step.kbar.cpu().numpy(),
        "scores": step.scores.view(Bt, H, step.score_stride).cpu().numpy(),
        "idx": step.idx.view(Bt, H, step.kmax).cpu().numpy(),
        "cnt": step.cnt.view(Bt, H).cpu().numpy(),
        "out": out.float().cpu().numpy(),
        "lse": step.lse.view(Bt, H).cpu().numpy(),
    }


def _check_sized(w, x, r, kinds, gran, budget, window, bf16_out=False):
    from oracle import decode as od
    from oracle import granularity as og
    from tests import _parity as P
    from workloads import generate
    assert r["status"] == 0
    L, d, Bt, Hkv = w.seq_len, w.head_dim, w.batch, w.num_kv_heads
    sizes = sorted({gran[h] for h in range(w.num_q_heads) if kinds[h] != 1})
    assert r["layout"]["sizes"] == sizes
    assert r["layout"]["score_stride"] == L // sizes[0]
    block_of = [gran[h] if kinds[h] != 1 else w.block for h in range(w.num_q_heads)]
    for b in range(Bt):
        q = generate.bf16_to_f64(x["q"][b:b + 1])
        k = generate.bf16_to_f32(x["k"][b:b + 1])
        v = generate.bf16_to_f32(x["v"][b:b + 1])
        off = 0
        for g in sizes:
            n = Bt * Hkv * (L // g) * d
            cache = r["kbar"][off:off + n].reshape(Bt, Hkv, L // g, d)
            np.testing.assert_allclose(cache[b], og.pool_cache(k, g)[0], rtol=1e-5, atol=1e-6)
            off += n
        sc = og.decode_scores(q, k, kinds, gran)[0]
        for h in range(w.num_q_heads):
            n = r["cnt"][b, h]
            sel = r["idx"][b, h, :n]
            assert all(t == -1 for t in r["idx"][b, h, n:])
            if kinds[h] == 1:
                assert sel.tolist() == od.streaming_blocks(w.nb, window)
                continue
            nbh = L // gran[h]
            np.testing.assert_allclose(r["scores"][b, h, :nbh], sc[h], rtol=1e-4, atol=1e-6)
            assert n == min(budget[h], nbh)
            P.check_selection_row(sel, og.select_row(sc[h], min(budget[h], nbh)), sc[h],
                                  nbh - 1)
        o, lse = od.decode_attend(q, k, v, r["idx"][b:b + 1], r["cnt"][b:b + 1], block_of)
        d_max, d_rel = P.output_errors(r["out"][b], o[0], bf16_out)
        assert d_max.max() <= P.MAX_ABS, d_max.max()
        assert d_rel.sum() / np.abs(o[0]).sum() <= P.MEAN_REL
        assert np.abs(r["lse"][b] - lse[0]).max() <= P.LSE_ABS


@pytest.mark.parametrize("L,Bt,window,sizes", [(4096, 2, 8, (16, 32, 64, 128)),
                                               (1024, 3, 4, (128, 16)),
                                               (2048, 1, 16, (64,))])
def test_decode_per_head_block_sizes(env, L, Bt, window, sizes):
    # every size a multiple of 16, odd unit counts (a masked half step),
    # budgets above a head's block count (capped), groups mixing sizes
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(5), L, batch=Bt)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    H = w.num_q_heads
    gran = [sizes[h % len(sizes)] for h in range(H)]
    budget = [3 + (5 * h) % 11 for h in range(H)]
    for out_dtype in ("float32", "bfloat16"):
        r = _decode_sized(sa, torch, w, x, kinds, gran, budget, window, out_dtype)
        _check_sized(w, x, r, kinds, gran, budget, window, bf16_out=out_dtype == "bfloat16")


@pytest.mark.parametrize("choice", ["bytes", "time_model"])
def test_decode_per_head_block_sizes_full_size(env, choice):
    # the 64K decode workload with the block sizes and budgets chosen offline,
    # by the byte model (two sizes) or the time model (one size, every
    # retrieval head at 16 tokens); rows of up to 4096 blocks
    import json
    import os
    sa, torch = env
    from workloads import generate, workload
    w = workload(5)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "workloads", "demands.json")) as f:
        prof = json.load(f)["5"]["granularity"]
    if choice == "time_model":
        prof = prof["time_model"]
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    window = w.window_tokens // w.block
    for out_dtype in ("float32", "bfloat16"):
        r = _decode_sized(sa, torch, w, x, kinds, prof["gran"], prof["budget"], window,
                          out_dtype)
        _check_sized(w, x, r, kinds, prof["gran"], prof["budget"], window,
                     bf16_out=out_dtype == "bfloat16")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (16, 2), (32, 2)])
def test_decode_group_sizes(env, Hq, Hkv):
    # groups of 1, 8 and 16 query heads: one or two 8-head tensor-core tiles
    # in the scores, with the default and with per-head block sizes
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(5), 2048, num_q_heads=Hq, num_kv_heads=Hkv, batch=2)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    r = _decode(sa, torch, w, x, kinds, 9, 4, "float32")
    _check(w, x, r, kinds, 9, 4)
    gran = [(16, 32, 64)[h % 3] for h in range(Hq)]
    budget = [4 + h % 7 for h in range(Hq)]
    if all(k == 1 for k in kinds):
        return
    r = _decode_sized(sa, torch, w, x, kinds, gran, budget, 4, "float32")
    _check_sized(w, x, r, kinds, gran, budget, 4)


def test_decode_all_streaming_with_block_sizes(env):
    # no retrieval head: no pooled cache, no score pass; streaming lists only
    sa, torch = env
    from workloads import generate, scaled, workload
    w = scaled(workload(5), 1024, num_q_heads=8, num_kv_heads=2, batch=2)
    x = generate.decode_inputs(w)
    kinds = np.ones(8, np.uint8)
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from oracle import decode as od
    from tests import _parity as P
    from tests._parity import to_dev
    shape = sa.Shape.decode(w.seq_len, w.block, 8, 2, w.head_dim, 2)
    step = DecodeStep(shape, 2, kinds, 4, with_lse=True, out_dtype=torch.float32,
                      granularity=[16] * 8, head_budget=[4] * 8)
    assert step.plan.decode_layout()["sizes"] == []
    t = {n: to_dev(x[n]) for n in "qkv"}
    step.build_cache(t["k"])
    out = step(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.idx.view(2, 8, step.kmax).cpu().numpy()
    cnt = step.cnt.view(2, 8).cpu().numpy()
    for b in range(2):
        for h in range(8):
            assert idx[b, h, :cnt[b, h]].tolist() == od.streaming_blocks(w.nb, 4)
    from workloads import generate as gen
    o, _ = od.decode_attend(gen.bf16_to_f64(x["q"]), gen.bf16_to_f32(x["k"]),
                            gen.bf16_to_f32(x["v"]), idx, cnt, w.block)
    assert np.abs(out.cpu().numpy() - o).max() <= P.MAX_ABS


@pytest.mark.parametrize("case", ["small", "full", "block_sizes"])
def test_decode_overlapped_step_equals_the_serial_step(env, case):
    """Streaming heads selected and attended on a side stream beside the
    retrieval heads' scoring, and the retrieval heads' scoring and selection
    fused into one launch: every output, log-sum-exp, index and count equals
    the serial step's with separate calls."""
    import json
    import os
    sa, torch = env
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    from workloads import generate, scaled, workload
    w = workload(5) if case != "small" else scaled(workload(5), 4096, batch=3)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    kw = {}
    if case == "block_sizes":
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        with open(os.path.join(root, "workloads", "demands.json")) as f:
            prof = json.load(f)["5"]["granularity"]
        kw = {"granularity": prof["gran"], "head_budget": prof["budget"]}
    t = {n: to_dev(x[n]) for n in "qkv"}
    res = []
    for overlap, fused, one in ((False, False, False), (False, True, False), (True, False, False),
                                (True, True, False), (True, True, True)):
        step = DecodeStep(shape, w.budget_tokens // w.block, kinds, w.window_tokens // w.block,
                          with_lse=True, out_dtype=torch.float32, overlap=overlap, fused=fused,
                          one_launch=one, **kw)
        step.build_cache(t["k"])
        for _ in range(2):   # a second call on the same buffers changes nothing
            step.idx.fill_(-5)
            step.out.fill_(float("nan"))
            out = step(t["q"], t["k"], t["v"])
            torch.cuda.synchronize()
            assert int(step.dev_status.item()) == 0
        res.append((out.clone(), step.lse.clone(), step.idx.clone(), step.cnt.clone()))
        del step
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)


@pytest.mark.parametrize("one_launch", [False, True])
def test_decode_overlapped_step_replays_from_a_cuda_graph(env, one_launch):
    """The overlapped step (two streams, five launches), and the one-launch
    step, captured in a CUDA graph: replays give the eager step's output and
    lists exactly, and the calls allocate nothing while captured."""
    sa, torch = env
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    from workloads import generate, scaled, workload
    w = scaled(workload(5), 8192, batch=4)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    t = {n: to_dev(x[n]) for n in "qkv"}
    step = DecodeStep(shape, w.budget_tokens // w.block, kinds, w.window_tokens // w.block,
                      with_lse=True, out_dtype=torch.float32, overlap=True,
                      one_launch=one_launch)
    step.build_cache(t["k"])
    want = step(t["q"], t["k"], t["v"]).clone()
    want_idx = step.idx.clone()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        step(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step(t["q"], t["k"], t["v"])
    for _ in range(2):
        step.out.fill_(float("nan"))
        step.idx.fill_(-3)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(step.out, want) and torch.equal(step.idx, want_idx)
    assert int(step.dev_status.item()) == 0


def test_decode_wait_timeout_is_reported_and_the_context_stays_usable(env):
    """The decode forward's waits for its copies, limited to 1 ns (far below
    a copy's latency from memory, with L2 flushed first), run out: the launch reports
    SA_DEV_TIMEOUT and returns, each warp having waited (with the full limit)
    for the copies it issued, so a normal launch right after gives the
    previous output exactly."""
    sa, torch = env
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    from workloads import generate, scaled, workload
    w = workload(5)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    t = {n: to_dev(x[n]) for n in "qkv"}
    step = DecodeStep(shape, w.budget_tokens // w.block, kinds, w.window_tokens // w.block,
                      out_dtype=torch.float32, overlap=False, one_launch=False)
    flush = torch.zeros(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    step.build_cache(t["k"])
    want = step(t["q"], t["k"], t["v"]).clone()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0

    def forward():
        sa.sparse_attn_forward(shape, step.plan, t["q"], t["k"], t["v"], step.idx, step.cnt,
                               step.kmax, step.out, None, step.dev_status)
        torch.cuda.synchronize()
        return int(step.dev_status.item())

    try:
        sa.sparse_attn_set_wait_limit(1)
        step.dev_status.zero_()
        step.out.fill_(float("nan"))
        flush.max()                    # the copies come from memory, not L2
        st = forward()
    finally:
        sa.sparse_attn_set_wait_limit(0)
    assert st & sa.SA_DEV_TIMEOUT, st
    assert not st & (sa.SA_DEV_BAD_INDEX | sa.SA_DEV_BAD_COUNT)
    for _ in range(2):
        step.dev_status.zero_()
        step.out.fill_(float("nan"))
        assert forward() == 0
        assert torch.equal(step.out, want)


@pytest.mark.parametrize("L,Hq,Hkv,Bt,budget,zero_q", [
    (65536, 28, 4, 16, 64, False),    # the 64K workload: 2048 blocks, clusters of four CTAs
    (8192, 28, 4, 1, 64, False),      # one sequence: clusters of eight CTAs
    (131072, 16, 1, 1, 100, False),   # 4096 blocks, one KV group of 16 heads
    (4096, 4, 4, 2, 9, False),        # groups of one head
    (256, 8, 2, 2, 3, False),         # 8 blocks: the first CTA of a cluster holds them all
    (2048, 8, 2, 2, 64, False),       # the budget keeps every block
    (4096, 8, 2, 2, 20, True),        # zero queries: every score ties, lowest indices win
    (4096, 8, 2, 3, 16, "group0"),    # KV group 0 all streaming: its clusters return at once
    (65536, 32, 4, 4, 64, False),     # groups of 8 heads (score rows kept per retrieval head)
])
def test_score_select_equals_separate_calls(env, L, Hq, Hkv, Bt, budget, zero_q):
    """The fused Index + Select launch gives the separate score and select
    calls' scores, lists and counts bit for bit on the retrieval heads' rows,
    and leaves the streaming heads' rows as they were."""
    sa, torch = env
    from tests._parity import to_dev
    from workloads import generate, scaled, workload
    w = scaled(workload(5), L, num_q_heads=Hq, num_kv_heads=Hkv, batch=Bt)
    x = generate.decode_inputs(w, tensors="qk")
    kinds = generate.head_kinds(w)
    if zero_q == "group0":
        G = Hq // Hkv
        kinds[:G] = 1                       # every head of KV group 0 streams
        kinds[G:] = [0, 1] * (G // 2)
        zero_q = False
    if not (kinds == 1).any():
        kinds[0] = 1                        # keep one streaming row to check it is untouched
    nb = w.nb
    shape = sa.Shape.decode(L, w.block, Hq, Hkv, w.head_dim, Bt)
    plan = sa.sparse_attn_plan(shape, min(budget, nb), head_kind=kinds, window_blocks=2,
                               num_workers=1)
    plan.upload()
    kmax = plan.info()["kmax"]
    q, k = to_dev(x["q"]), to_dev(x["k"])
    if zero_q:
        q.zero_()
    kbar = torch.empty(Bt * Hkv * nb * w.head_dim, dtype=torch.float32, device="cuda")
    sa.sparse_attn_pool_kcache(shape, k, kbar)
    rows = Bt * Hq

    def buffers():
        return (torch.full((rows * nb,), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((rows * kmax,), -7, dtype=torch.int32, device="cuda"),
                torch.full((rows,), -7, dtype=torch.int32, device="cuda"))

    sc_a, idx_a, cnt_a = buffers()
    sa.sparse_attn_score(shape, q, kbar, sc_a, None, 0)
    sa.sparse_attn_select_kind(shape, plan, sc_a, idx_a, cnt_a, kmax, sa.SA_HEAD_RETRIEVAL)
    sc_b, idx_b, cnt_b = buffers()
    sa.sparse_attn_score_select(shape, plan, q, kbar, sc_b, idx_b, cnt_b, kmax)
    _, idx_c, cnt_c = buffers()
    sa.sparse_attn_score_select(shape, plan, q, kbar, None, idx_c, cnt_c, kmax)
    torch.cuda.synchronize()
    ret = torch.tensor(np.tile(kinds != 1, Bt), device="cuda")
    sc_a, sc_b = sc_a.view(rows, nb), sc_b.view(rows, nb)
    idx_a, idx_b, idx_c = (t.view(rows, kmax) for t in (idx_a, idx_b, idx_c))
    assert torch.equal(sc_a[ret], sc_b[ret])
    assert torch.isnan(sc_b[~ret]).all()
    for idx, cnt in ((idx_b, cnt_b), (idx_c, cnt_c)):
        assert torch.equal(idx[ret], idx_a[ret])
        assert torch.equal(cnt[ret], cnt_a[ret])
        assert (idx[~ret] == -7).all() and (cnt[~ret] == -7).all()
    keep = min(budget, nb)
    assert (cnt_a[ret] == keep).all()
    if zero_q:
        want = list(range(keep - 1)) + [nb - 1]
        assert all(r.tolist()[:keep] == want for r in idx_a[ret].cpu())


def test_score_select_with_no_retrieval_head_launches_nothing(env):
    """A plan whose heads all stream: the fused call returns at once and
    leaves every output as it was."""
    sa, torch = env
    shape = sa.Shape.decode(2048, 32, 8, 2, 128, 2)
    plan = sa.sparse_attn_plan(shape, 8, head_kind=[1] * 8, window_blocks=4, num_workers=1)
    plan.upload()
    kmax = plan.info()["kmax"]
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    kbar = torch.zeros(2 * 2 * 64 * 128, dtype=torch.float32, device="cuda")
    sc = torch.full((2 * 8 * 64,), float("nan"), device="cuda")
    idx = torch.full((2 * 8 * kmax,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((16,), -7, dtype=torch.int32, device="cuda")
    sa.sparse_attn_score_select(shape, plan, q, kbar, sc, idx, cnt, kmax)
    torch.cuda.synchronize()
    assert torch.isnan(sc).all() and (idx == -7).all() and (cnt == -7).all()


@pytest.mark.parametrize("L,Hq,Hkv,Bt,budget,window,case", [
    (4096, 4, 4, 2, 9, 4, ""),            # groups of one head
    (8192, 28, 4, 1, 64, 8, ""),          # one sequence: clusters of eight CTAs
    (256, 8, 2, 2, 3, 2, ""),             # 8 blocks: most CTAs score nothing but attend
    (2048, 8, 2, 2, 64, 2, ""),           # the budget keeps every block
    (2048, 8, 2, 2, 16, 63, ""),          # the window reaches block 1: all blocks
    (4096, 8, 2, 2, 20, 3, "zero_q"),     # zero queries: every score ties
    (4096, 8, 2, 3, 16, 4, "group0"),     # KV group 0 all streaming: no scoring, attention only
    (2048, 8, 2, 2, 16, 4, "all_streaming"),
    (65536, 32, 4, 4, 64, 32, ""),        # groups of 8 heads
    (131072, 16, 1, 1, 100, 16, ""),      # 4096 blocks; 16 heads, two per warpgroup
    (65536, 28, 4, 16, 64, 64, ""),       # the 64K workload: clusters of four CTAs
])
def test_decode_step_one_launch_equals_separate_calls(env, L, Hq, Hkv, Bt, budget, window, case):
    """The one-launch decode step gives the separate calls' (score, select,
    forward) lists, counts, outputs and log-sum-exps bit for bit on every
    row, and their scores on the retrieval rows, in fp32 and bf16 output."""
    sa, torch = env
    from tests._parity import to_dev
    from workloads import generate, scaled, workload
    w = scaled(workload(5), L, num_q_heads=Hq, num_kv_heads=Hkv, batch=Bt)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    G = Hq // Hkv
    if case == "group0":
        kinds[:G] = 1
        kinds[G:] = [0, 1] * ((Hq - G) // 2)
    elif case == "all_streaming":
        kinds[:] = 1
    nb = w.nb
    shape = sa.Shape.decode(L, w.block, Hq, Hkv, w.head_dim, Bt)
    plan = sa.sparse_attn_plan(shape, min(budget, nb), head_kind=kinds, window_blocks=window,
                               num_workers=1)
    plan.upload()
    kmax = plan.info()["kmax"]
    q, k, v = (to_dev(x[n]) for n in "qkv")
    if case == "zero_q":
        q.zero_()
    kbar = torch.empty(Bt * Hkv * nb * w.head_dim, dtype=torch.float32, device="cuda")
    sa.sparse_attn_pool_kcache(shape, k, kbar)
    rows = Bt * Hq
    ret = torch.tensor(np.tile(kinds != 1, Bt), device="cuda")
    for dt in (torch.float32, torch.bfloat16):
        def buffers():
            return (torch.full((rows, nb), float("nan"), device="cuda"),
                    torch.full((rows, kmax), -7, dtype=torch.int32, device="cuda"),
                    torch.full((rows,), -7, dtype=torch.int32, device="cuda"),
                    torch.full((rows, w.head_dim), float("nan"), dtype=dt, device="cuda"),
                    torch.full((rows,), float("nan"), device="cuda"),
                    torch.zeros(1, dtype=torch.int32, device="cuda"))
        sc_a, idx_a, cnt_a, o_a, lse_a, st_a = buffers()
        sa.sparse_attn_score(shape, q, kbar, sc_a, None, 0)
        sa.sparse_attn_select(shape, plan, sc_a, idx_a, cnt_a, kmax)
        sa.sparse_attn_forward(shape, plan, q, k, v, idx_a, cnt_a, kmax, o_a, lse_a, st_a)
        sc_b, idx_b, cnt_b, o_b, lse_b, st_b = buffers()
        sa.sparse_attn_decode_step(shape, plan, q, kbar, k, v, sc_b, idx_b, cnt_b, kmax, o_b,
                                   lse_b, st_b)
        _, idx_c, cnt_c, o_c, _, st_c = buffers()
        sa.sparse_attn_decode_step(shape, plan, q, kbar, k, v, None, idx_c, cnt_c, kmax, o_c,
                                   None, st_c)
        torch.cuda.synchronize()
        assert int(st_a.item()) == 0 and int(st_b.item()) == 0 and int(st_c.item()) == 0
        assert torch.equal(sc_b[ret], sc_a[ret])
        assert torch.isnan(sc_b[~ret]).all()
        for idx, cnt, o in ((idx_b, cnt_b, o_b), (idx_c, cnt_c, o_c)):
            assert torch.equal(idx, idx_a)
            assert torch.equal(cnt, cnt_a)
            assert torch.equal(o, o_a)
        assert torch.equal(lse_b, lse_a)


def test_decode_step_one_launch_wait_timeout_is_reported(env):
    """The one-launch step's waits for its attention copies, limited to 1 ns,
    run out: the launch reports SA_DEV_TIMEOUT and returns (each warp waits
    with the full limit for the copies it issued, and the cluster barriers
    are still met), and normal launches right after give the step's output
    exactly."""
    sa, torch = env
    from tests._parity import to_dev
    from workloads import generate, workload
    w = workload(5)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    plan = sa.sparse_attn_plan(shape, w.budget_tokens // w.block, head_kind=kinds,
                               window_blocks=w.window_tokens // w.block, num_workers=1)
    plan.upload()
    kmax = plan.info()["kmax"]
    q, k, v = (to_dev(x[n]) for n in "qkv")
    rows, nb = w.batch * w.num_q_heads, w.nb
    kbar = torch.empty(w.batch * w.num_kv_heads * nb * w.head_dim, dtype=torch.float32,
                       device="cuda")
    sa.sparse_attn_pool_kcache(shape, k, kbar)
    idx = torch.empty(rows, kmax, dtype=torch.int32, device="cuda")
    cnt = torch.empty(rows, dtype=torch.int32, device="cuda")
    out = torch.empty(rows, w.head_dim, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.zeros(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def step():
        st.zero_()
        out.fill_(float("nan"))
        sa.sparse_attn_decode_step(shape, plan, q, kbar, k, v, None, idx, cnt, kmax, out, None, st)
        torch.cuda.synchronize()
        return int(st.item())

    assert step() == 0
    want = out.clone()
    try:
        sa.sparse_attn_set_wait_limit(1)
        flush.max()                    # the copies come from memory, not L2
        got = step()
    finally:
        sa.sparse_attn_set_wait_limit(0)
    assert got & sa.SA_DEV_TIMEOUT, got
    assert not got & (sa.SA_DEV_BAD_INDEX | sa.SA_DEV_BAD_COUNT)
    for _ in range(2):
        assert step() == 0
        assert torch.equal(out, want)
