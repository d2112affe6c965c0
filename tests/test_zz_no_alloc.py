"""The allocation-free scoring entry point against the regular one.

sparse_attn_score_noalloc serves callers that cannot allocate device memory
when they score a layer; it keeps the pooled vectors in the library's fixed
scratch area instead of a caller workspace.  It must give the same scores as
sparse_attn_score, also on a second call right after the first (the area keeps
the previous call's contents).  This file is collected last on purpose.
"""
import ctypes

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


def _inputs(torch, w, seed):
    from tests._parity import to_dev
    from workloads import generate
    x = generate.prefill_inputs(w, tensors="qk", seed=seed)
    return to_dev(x["q"]), to_dev(x["k"])


def _noalloc(sa, torch, shape, q, k, out):
    return sa._lib.sparse_attn_score_noalloc(
        ctypes.byref(shape), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare(sa, torch, w, seed):
    """One regular call and one allocation-free call on the same inputs."""
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)
    nb, Hq = w.nb, w.num_q_heads
    lower = torch.tril(torch.ones(nb, nb, dtype=torch.bool, device="cuda"))
    ws = torch.empty(sa.sparse_attn_score_workspace_size(shape) // 4 + 1, dtype=torch.float32,
                     device="cuda")
    q, k = _inputs(torch, w, seed)
    ref = torch.full((Hq, nb, nb), float("nan"), device="cuda")
    got = torch.full((Hq, nb, nb), float("nan"), device="cuda")
    sa.sparse_attn_score(shape, q, k, ref, ws)
    st = _noalloc(sa, torch, shape, q, k, got)
    assert st == 0, sa.sa_status_string(st)
    torch.cuda.synchronize()
    r, g = ref[:, lower], got[:, lower]
    assert torch.isfinite(g).all()
    np.testing.assert_allclose(g.cpu().numpy(), r.cpu().numpy(), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("number,S,Hq,Hkv", [(1, 4096, 8, 2), (2, 16384, 32, 8)])
def test_noalloc_scores_match_workspace_scores(env, number, S, Hq, Hkv):
    sa, torch = env
    from workloads import scaled, workload
    w = scaled(workload(number), S, Hq, Hkv)
    for seed in (w.seed, w.seed + 77):           # two calls in a row, different data
        _compare(sa, torch, w, seed)


def test_noalloc_smaller_call_after_a_larger_one(env):
    # the area keeps the larger call's pooled vectors beyond the smaller
    # call's extent; none of them may leak into the smaller call's scores
    sa, torch = env
    from workloads import scaled, workload
    _compare(sa, torch, scaled(workload(2), 32768, 32, 8), 5)
    _compare(sa, torch, scaled(workload(1), 2048, 8, 2), 6)


def test_noalloc_rejects_shapes_beyond_its_area(env):
    sa, torch = env
    # (64 + 8) heads x 2048 blocks x 64 dims x 4 bytes = 36 MiB > 32 MiB.  The
    # buffers are real (1.07 GB of queries and of scores), so that even a
    # regressed size check would compute on valid memory instead of faulting.
    S, B, Hq, Hkv, d = 131072, 64, 64, 8, 64
    shape = sa.Shape.prefill(S, B, Hq, Hkv, d)
    nb = S // B
    assert (Hq + Hkv) * nb * d * 4 > 32 << 20
    q = torch.zeros(Hq, S, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(Hkv, S, d, dtype=torch.bfloat16, device="cuda")
    out = torch.full((Hq, nb, nb), -1.0, device="cuda")
    st = _noalloc(sa, torch, shape, q, k, out)
    torch.cuda.synchronize()
    assert st == 3, sa.sa_status_string(st)          # SA_ERR_UNSUPPORTED
    assert bool((out == -1.0).all())                 # nothing was written
    del q, k, out
    torch.cuda.empty_cache()
