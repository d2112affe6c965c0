"""The bench's multi-replica timing on two CPU ranks (gloo).

With N > 1 every rank runs an independent replica of the layer; the job's time
is the slowest rank's, and the reported throughput is all replicas' work over
that time.  This checks that reduction with two processes on the host.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]              # rank 1 is the slow replica
        total = bench.max_over_ranks(local_ms, torch.device("cpu"))
        value = bench.job_value(8.0e12, world, 10, total)
        out.put((rank, total, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_two_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value in res:
        assert total == 150.0                        # every rank sees the slowest time
        # 2 replicas x 10 steps x 8 TFLOP over 0.15 s
        assert value == pytest.approx(2 * 10 * 8.0 / 0.150)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_value(1e12, 1, 4, 2000.0) == pytest.approx(2.0)


def test_reference_arm_prints_the_contract_line():
    # the reference arm times the oracle on the host: one JSON line with the
    # main arm's metric, unit and config, the host baseline and a zero-copy e2e
    import json
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=600, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    import bench
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == "llama31_8b_prefill_128k"
    # the same config the GPU arm prints: the workload and its plan's blocks
    from workloads import workload
    layer_flops, blocks = bench._layer_flops()
    assert line["config"] == bench.workload_config(workload(bench.WORKLOAD), blocks, 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["extrapolation"]["s_per_layer"] == pytest.approx(
        layer_flops / (line["value"] * 1e12), rel=1e-2)
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_cpu_baseline_reports_one_core_and_all_cores():
    # the oracle timed twice on the host, on every core and on one, each
    # figure extrapolated to the whole layer
    import bench
    b = bench.cpu_baseline(None, sample_seconds=4.0)
    assert b["kind"] == "oracle" and b["value"] > 0 and b["one_core"]["value"] > 0
    assert b["one_core"]["cores"] == 1 and b["cores"] >= 1
    ext = b["extrapolation"]
    assert ext["one_core_s_per_layer"] == pytest.approx(
        ext["layer_tflop"] / b["one_core"]["value"], rel=1e-2)
    assert ext["all_cores_s_per_layer"] == pytest.approx(ext["layer_tflop"] / b["value"], rel=1e-2)
