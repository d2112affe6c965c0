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


def _decode(sa, torch, w, x, kinds, budget, window, out_dtype="float32"):
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from tests._parity import to_dev
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    step = DecodeStep(shape, budget, kinds, window, with_lse=True,
                      out_dtype=getattr(torch, out_dtype))
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
        np.testing.assert_allclose(r["scores"][b], sc, rtol=1e-4, atol=1e-6)
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
        d = np.abs(r["out"][b] - o[0])
        if bf16_out:
            d = np.maximum(d - P.half_ulp_bf16(np.maximum(np.abs(o[0]), np.abs(r["out"][b]))), 0)
        assert d.max() <= P.MAX_ABS, d.max()
        assert d.sum() / np.abs(o[0]).sum() <= P.MEAN_REL
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
        r = _decode(sa, torch, w, x, kinds, budget, window, out_dtype)
        _check(w, x, r, kinds, budget, window, bf16_out=out_dtype == "bfloat16")


def test_decode_full_size(env):
    sa, torch = env
    from workloads import generate, workload
    w = workload(5)
    x = generate.decode_inputs(w)
    kinds = generate.head_kinds(w)
    budget = w.budget_tokens // w.block
    window = w.window_tokens // w.block
    r = _decode(sa, torch, w, x, kinds, budget, window, "bfloat16")
    _check(w, x, r, kinds, budget, window, bf16_out=True)
