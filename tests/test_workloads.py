"""The seeded input generator: bfloat16 rounding, determinism and subsetting."""
import numpy as np
import torch

from workloads import generate, scaled, workload


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 5,
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, 65504.0], np.float32),
        # exact ties between two bfloat16 values
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(generate.bf16_bits(x), ref)
    back = generate.bf16_to_f32(ref)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_prefill_inputs_deterministic_and_subsettable():
    w = scaled(workload(1), 512)
    a = generate.prefill_inputs(w)
    b = generate.prefill_inputs(w)
    for t in "qkv":
        np.testing.assert_array_equal(a[t], b[t])
    sub = generate.prefill_inputs(w, tensors="q", heads=[5, 2])
    np.testing.assert_array_equal(sub["q"][0], a["q"][5])
    np.testing.assert_array_equal(sub["q"][1], a["q"][2])
    assert a["q"].shape == (8, 512, 64) and a["k"].shape == (2, 512, 64)
    # different heads are scaled differently (heterogeneous sparsity)
    s = generate.q_scales(w)
    assert s.min() >= 0.5 - 1e-6 and s.max() <= 3.0 + 1e-6 and len(set(s.tolist())) == 8
    std = generate.bf16_to_f32(a["q"]).std(axis=(1, 2))
    np.testing.assert_allclose(std, s, rtol=0.1)


def test_calibration_draw_differs():
    w = scaled(workload(2), 1024, 4, 1)
    a = generate.prefill_inputs(w, tensors="k")
    b = generate.prefill_inputs(w, tensors="k", seed=w.calib_seed)
    assert not np.array_equal(a["k"], b["k"])
    # same heads (scales), different data
    qa = generate.prefill_inputs(w, tensors="q")["q"]
    qb = generate.prefill_inputs(w, tensors="q", seed=w.calib_seed)["q"]
    np.testing.assert_allclose(generate.bf16_to_f32(qa).std(axis=(1, 2)),
                               generate.bf16_to_f32(qb).std(axis=(1, 2)), rtol=0.1)


def test_heavy_keys_planted():
    w = scaled(workload(4), 2048, 8, 1)
    pos, unit = generate.heavy_keys(w)
    x = generate.prefill_inputs(w, tensors="k")
    k = generate.bf16_to_f32(x["k"][0])
    norms = np.linalg.norm(k, axis=1)
    assert set(np.argsort(norms)[-4:].tolist()) == set(pos[0].tolist())
    np.testing.assert_allclose(np.linalg.norm(unit, axis=1), 1.0, rtol=1e-6)


def test_decode_inputs_and_kinds():
    w = scaled(workload(5), 256, batch=2)
    x = generate.decode_inputs(w)
    assert x["q"].shape == (2, 28, 128) and x["k"].shape == (2, 4, 256, 128)
    kinds = generate.head_kinds(w)
    assert int((kinds == generate.STREAMING).sum()) == 11
    y = generate.decode_inputs(w, tensors="k", batches=[1])
    np.testing.assert_array_equal(y["k"][0], x["k"][1])
