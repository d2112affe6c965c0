"""Benchmark: one block-sparse attention prefill layer (score -> select ->
forward) of the 128K-token Llama-3.1-8B-shaped workload on one GB300, through
the C ABI.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the hot path over the layer: pooled block scoring,
per-head top-k selection and block-sparse attention on the persistent LPT
schedule.  Budgets and the schedule are the offline plan (built once from the
stored calibration profile, as the pages' offline profiling prescribes; its
host time is reported separately and is inside the end-to-end number).
Inputs (Q 1.07 GB, K and V 0.27 GB each) are larger than L2, so no flush is
needed between steps.  With N > 1 (torchrun) every rank runs an independent
replica (the path has no exchange step), timing is the max over ranks and
value is the sum of the replicas' work over that time.

--impl reference times the fp64 oracle on the host cores on a bounded sample
of the same workload (a few heads of scoring and selection plus a sample of
attention items per step), scaled to the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "block-sparse attn ms/layer + TFLOP/s at 128K prefill; % of roofline (1 GB300)"
UNIT = "TFLOP/s"
WORKLOAD = 3
DECODE_WORKLOAD = 5


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _profile(number):
    with open(os.path.join(ROOT, "workloads", "demands.json")) as f:
        return json.load(f)[str(number)]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the job's time is its slowest replica)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_replica_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job TFLOP/s: every replica's work over the slowest replica's time."""
    return flops_per_replica_step * world * steps / (total_ms * 1e-3) / 1e12


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the forward kernel at the 128K Llama-3.1-8B workload, from the ncu capture
# summarised in profiles/prefill_attention_llama8b_128k.md.  It describes only
# the kernel source with this SHA-256; for any other source it is not reported.
FORWARD_TRAFFIC = {"workload": 3,
                   "sha256": {"prefill.cu": "3d2f4f2810b160e3f70b0bc8ccf5f13a3eddbb334167b009cac61bf42a4253ba",
                              "plan.cpp": "c616ba6a80c1066d0afaeaf52cd474c5e421f84c00f0bec29446911e2367f6d2"},
                   "bytes": 1872382208 + 1081516544,
                   "group_shared_bytes": 1739555072 + 1074110464}


def _forward_traffic(workload_number: int):
    # the kernel and the schedule (its order sets what L2 catches) as captured
    import hashlib

    for name, want in FORWARD_TRAFFIC["sha256"].items():
        with open(os.path.join(ROOT, "head_heterogeneous_block_gb300", "csrc", name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != want:
                return None
    return FORWARD_TRAFFIC if FORWARD_TRAFFIC["workload"] == workload_number else None


def _attention_flops(total_blocks: int, B: int, d: int) -> float:
    # QK^T and PV over full B x B tiles of every selected block
    return 4.0 * B * B * d * total_blocks


def _score_flops(w) -> float:
    return 2.0 * w.num_q_heads * (w.nb * (w.nb + 1) / 2) * w.head_dim


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import head_heterogeneous_block_gb300 as sa
    from head_heterogeneous_block_gb300.layer import DecodeStep, PrefillLayer
    from workloads import generate, workload

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = workload(args.workload)
    prof = _profile(args.workload)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    shape = sa.Shape.prefill(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim)

    t0 = time.perf_counter()
    layer = PrefillLayer(shape, prof["k_uniform"], demand=prof["demand"], k_min=prof["k_min"],
                         num_workers=sms, schedule=args.schedule, device=dev)
    setup_ms = (time.perf_counter() - t0) * 1e3
    # the host plan alone (Max-Min budgets and the schedule), best of five
    plan_ms = float("inf")
    for _ in range(5):
        t0 = time.perf_counter()
        p = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=prof["demand"],
                                k_min=prof["k_min"], num_workers=sms, schedule=args.schedule)
        plan_ms = min(plan_ms, (time.perf_counter() - t0) * 1e3)
        p.close()
    x = generate.prefill_inputs(w)
    host = {n: torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).pin_memory()
            for n in "qkv"}
    del x
    t = {n: host[n].to(dev, non_blocking=True) for n in "qkv"}
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    flops = _attention_flops(layer.total_blocks, w.block, w.head_dim) + _score_flops(w)
    attn_flops = _attention_flops(layer.total_blocks, w.block, w.head_dim)

    def step():
        layer(t["q"], t["k"], t["v"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(layer.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.dev_status.item())}")

    # ---- timed region: K steps; the forward kernel is bracketed by its own
    # events on the launching stream to measure its average duration.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        layer.score(t["q"], t["k"], stream=stream)
        ev[k][1].record(stream)
        layer.select(stream=stream)
        ev[k][2].record(stream)
        layer.attend(t["q"], t["k"], t["v"], stream=stream)
        ev[k][3].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(start.elapsed_time(stop), dev)
    fwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    stages = {"score_ms": round(statistics.mean(e[0].elapsed_time(e[1]) for e in ev), 4),
              "select_ms": round(statistics.mean(e[1].elapsed_time(e[2]) for e in ev), 4),
              "forward_ms": round(fwd_ms, 4)}
    ms_step = total_ms / args.steps
    value = job_value(flops, ws, args.steps, total_ms)
    status = int(layer.dev_status.item())

    # ---- schedules: forward alone under each plan (same inputs, same idx)
    sched = {}
    for pol in ("lpt_grouped", "lpt", "head_order"):
        p = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=prof["demand"],
                                k_min=prof["k_min"], num_workers=sms, schedule=pol)
        p.upload()
        for _ in range(2):
            sa.sparse_attn_forward(shape, p, t["q"], t["k"], t["v"], layer.idx, layer.cnt,
                                   layer.kmax, layer.out, None, layer.dev_status, stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record(stream)
        for _ in range(reps):
            sa.sparse_attn_forward(shape, p, t["q"], t["k"], t["v"], layer.idx, layer.cnt,
                                   layer.kmax, layer.out, None, layer.dev_status, stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        inf = p.info()
        sched[pol] = {"forward_ms": round(a.elapsed_time(b) / reps, 4),
                      "makespan_blocks": inf["makespan"],
                      "mean_load_blocks": round(inf["total_blocks"] / sms, 1)}
        p.close()

    # ---- GQA-group-shared selection (one block list per KV group), same inputs
    group_shared = None
    if not args.no_variants:
        lg = PrefillLayer(shape, prof["k_uniform"], demand=prof["demand"], k_min=prof["k_min"],
                          num_workers=sms, schedule=args.schedule, device=dev,
                          group_shared=True)
        for _ in range(2):
            lg(t["q"], t["k"], t["v"], stream=stream)
        evg = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(5)]
        for e in evg:
            e[0].record(stream)
            lg.score(t["q"], t["k"], stream=stream)
            e[1].record(stream)
            lg.select(stream=stream)
            e[2].record(stream)
            lg.attend(t["q"], t["k"], t["v"], stream=stream)
            e[3].record(stream)
        torch.cuda.synchronize(dev)
        g_fwd = statistics.mean(e[2].elapsed_time(e[3]) for e in evg)
        g_flops = _attention_flops(lg.total_blocks, w.block, w.head_dim)
        group_shared = {
            "ms_per_layer": round(statistics.mean(e[0].elapsed_time(e[3]) for e in evg), 4),
            "select_ms": round(statistics.mean(e[1].elapsed_time(e[2]) for e in evg), 4),
            "forward_ms": round(g_fwd, 4), "selected_blocks": lg.total_blocks,
            "forward_tflops": round(g_flops / (g_fwd * 1e-3) / 1e12, 1),
            "budgets": "Max-Min shifted between KV groups, each demanding its most "
                       "demanding head's blocks",
            "device_status": int(lg.dev_status.item())}
        # the same lists with head pairs on one K/V block load each
        lp = PrefillLayer(shape, prof["k_uniform"], demand=prof["demand"], k_min=prof["k_min"],
                          num_workers=sms, schedule=args.schedule, device=dev,
                          group_shared=True, share_kv=True)
        lp.idx.copy_(lg.idx)
        lp.cnt.copy_(lg.cnt)
        for _ in range(2):
            lp.attend(t["q"], t["k"], t["v"], stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            lp.attend(t["q"], t["k"], t["v"], stream=stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        group_shared["share_kv_forward_ms"] = round(a.elapsed_time(b) / 5, 4)
        group_shared["share_kv_device_status"] = int(lp.dev_status.item())
        del lg, lp

    # ---- output-aware demands (calibration signal only; same kernels)
    output_aware = None
    if not args.no_variants and "output_aware" in prof:
        oa = prof["output_aware"]
        lo = PrefillLayer(shape, prof["k_uniform"], demand=oa["demand"], k_min=prof["k_min"],
                          num_workers=sms, schedule=args.schedule, device=dev)
        for _ in range(2):
            lo(t["q"], t["k"], t["v"], stream=stream)
        evo = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(5)]
        for e in evo:
            e[0].record(stream)
            lo(t["q"], t["k"], t["v"], stream=stream)
            e[1].record(stream)
        torch.cuda.synchronize(dev)
        o_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evo)
        output_aware = {
            "ms_per_layer": round(o_ms, 4), "selected_blocks": lo.total_blocks,
            "makespan_blocks": lo.plan.info()["makespan"],
            "demand_range": [min(oa["demand"]), max(oa["demand"])],
            "budget_range": [min(oa["budgets_maxmin"]), max(oa["budgets_maxmin"])],
            "device_status": int(lo.dev_status.item())}
        del lo

    # ---- top-p selection (data-dependent counts) at the plan's mean density:
    # static schedules (head order; LPT over the top-k budgets) against the
    # LPT rebuilt on the GPU from the selected counts
    topp = None
    if not args.no_variants:
        p_thr = layer.total_blocks / (w.num_q_heads * w.nb * (w.nb + 1) / 2)
        tidx = torch.empty(w.num_q_heads * w.nb * w.nb, dtype=torch.int32, device=dev)
        tcnt = torch.empty(w.num_q_heads * w.nb, dtype=torch.int32, device=dev)
        res = {}
        swptr = torch.empty(sms + 1, dtype=torch.int32, device=dev)
        sitems = torch.empty(w.num_q_heads * w.nb, dtype=torch.int32, device=dev)
        for mode in ("head_order_static", "lpt_static", "lpt_rebuilt"):
            pl = sa.sparse_attn_plan(shape, prof["k_uniform"], k_min=prof["k_min"],
                                     demand=prof["demand"], num_workers=sms,
                                     schedule="head_order" if mode == "head_order_static"
                                     else "lpt")
            pl.upload()
            ev_t = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for rep in range(3):
                ev_t[0].record(stream)
                sa.sparse_attn_select_topp(shape, pl, layer.scores, p_thr, tidx, tcnt, w.nb,
                                           stream=stream)
                ev_t[1].record(stream)
                if mode == "lpt_rebuilt":
                    pl.rebuild(tcnt, stream=stream)
                ev_t[2].record(stream)
                sa.sparse_attn_forward(shape, pl, t["q"], t["k"], t["v"], tidx, tcnt, w.nb,
                                       layer.out, None, layer.dev_status, stream)
                ev_t[3].record(stream)
            pl.device_schedule(swptr, sitems, stream=stream)
            torch.cuda.synchronize(dev)
            # makespan in selected blocks of the schedule the forward ran
            cw = np.cumsum(np.concatenate([[0], tcnt.cpu().numpy()[sitems.cpu().numpy()]]))
            wp = swptr.cpu().numpy()
            res[mode] = {"select_ms": round(ev_t[0].elapsed_time(ev_t[1]), 4),
                         "rebuild_ms": round(ev_t[1].elapsed_time(ev_t[2]), 4),
                         "forward_ms": round(ev_t[2].elapsed_time(ev_t[3]), 4),
                         "makespan_blocks": int((cw[wp[1:]] - cw[wp[:-1]]).max())}
            pl.close()
        topp = {"p": round(p_thr, 5), "selected_blocks": int(tcnt.sum().item()),
                "mean_load_blocks": round(float(tcnt.sum().item()) / sms, 1),
                "device_status": int(layer.dev_status.item()), **res}
        del tidx, tcnt, swptr, sitems

    # ---- end to end through the public API with host buffers: every step
    # copies its Q, K and V from pinned host memory and reads its output
    # back; HostPipeline overlaps one step's copies with another's compute.
    # The host plan is rebuilt before every step to charge its cost too.
    from head_heterogeneous_block_gb300.layer import HostPipeline
    out_host = [torch.empty((w.num_q_heads, w.seq_len, w.head_dim), dtype=torch.bfloat16,
                            pin_memory=True) for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in "qkv")
    d2h = out_host[0].numel() * out_host[0].element_size()
    e2e_steps = 16
    pipe = HostPipeline(layer, device=dev)

    def replan(_s):
        p = sa.sparse_attn_plan(shape, prof["k_uniform"], demand=prof["demand"],
                                k_min=prof["k_min"], num_workers=sms, schedule=args.schedule)
        p.close()

    steps_in = [(host["q"], host["k"], host["v"], out_host[s % 2]) for s in range(e2e_steps)]
    pipe.run(steps_in[:2], stream=stream)          # warm-up
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    pipe.run(steps_in, stream=stream, before_step=replan)
    e2e_s = (time.perf_counter() - t1) / e2e_steps
    e2e_value = flops / e2e_s / 1e12

    # the host link alone: one step's copies with no compute, each direction
    # by itself and both at once on the pipeline's two copy streams; the
    # larger of the both-at-once time and the device step bounds e2e
    def link(direction, reps=3, out_buf=0):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            if direction in ("in", "both"):
                with torch.cuda.stream(pipe.copy_in):
                    for n in "qkv":
                        pipe.bufs[0][n].copy_(host[n], non_blocking=True)
            if direction in ("out", "both"):
                with torch.cuda.stream(pipe.copy_out):
                    out_host[out_buf].copy_(pipe.bufs[0]["o"], non_blocking=True)
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / reps

    # where a pipelined step's time goes: six more steps with timing events
    # on the three streams (not timed above); per step the spans of copy-in,
    # compute and copy-out, and the share of copy time that ran while the
    # compute stream was busy
    tl = []
    pipe.run(steps_in[:6], stream=stream, timeline=tl)
    torch.cuda.synchronize(dev)
    t0 = tl[0]["in"][0]

    def span(ev):
        return t0.elapsed_time(ev[0]), t0.elapsed_time(ev[1])

    comp_spans = [span(x["compute"]) for x in tl]

    def hidden(a, b):
        # ms of [a, b) that fall inside some compute span
        return sum(max(0.0, min(b, ce) - max(a, cs)) for cs, ce in comp_spans)

    copy_ms = hid_ms = 0.0
    for x in tl:
        for k in ("in", "out"):
            a, b = span(x[k])
            copy_ms += b - a
            hid_ms += hidden(a, b)
    last = max(span(x["out"])[1] for x in tl)
    pipeline = {"steps": len(tl), "ms_per_step": round(last / len(tl), 3),
                "copy_in_ms": round(statistics.mean(b - a for a, b in (span(x["in"]) for x in tl)), 3),
                "compute_ms": round(statistics.mean(b - a for a, b in comp_spans), 3),
                "copy_out_ms": round(statistics.mean(b - a for a, b in (span(x["out"]) for x in tl)), 3),
                # the two output buffers alternate: their copies apart
                "copy_out_ms_by_buffer": [round(statistics.mean(
                    b - a for a, b in (span(x["out"]) for x in tl[i::2])), 3) for i in (0, 1)],
                "copy_time_under_compute": round(hid_ms / copy_ms, 3) if copy_ms else None}
    del tl

    link("both", 1)
    t_in, t_out, t_both = link("in"), link("out"), link("both")
    t_out1 = link("out", out_buf=1)
    host_link = {"h2d_gbs": round(h2d / t_in / 1e9, 1), "d2h_gbs": round(d2h / t_out / 1e9, 1),
                 "d2h_gbs_second_buffer": round(d2h / t_out1 / 1e9, 1),
                 "copies_ms_per_step": round(t_both * 1e3, 3),
                 "floor_ms_per_step": round(max(t_both * 1e3, ms_step), 3),
                 "bound": "host link" if t_both * 1e3 > ms_step else "device"}
    del pipe

    # ---- decode step (workload 5), reported beside the prefill line
    decode = None
    if not args.no_decode:
        decode = bench_decode(dev, stream)

    peaks = _peaks()
    achieved = attn_flops / (fwd_ms * 1e-3) / 1e12
    # DRAM bytes of one forward launch, from ncu, while the sources are the
    # ones captured (else null)
    traffic = _forward_traffic(args.workload)
    if group_shared is not None:
        group_shared["traffic"] = traffic["group_shared_bytes"] if traffic else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, per-head query scales; calibrated budgets)",
        "config": workload_config(w, layer.total_blocks, ws),
        "launch": {"schedule": args.schedule, "workers": sms},
        "ms_per_layer": round(ms_step, 4),
        "forward_ms": round(fwd_ms, 4),
        "stages": stages,
        "plan_host_ms": round(plan_ms, 3),
        "layer_setup_ms": round(setup_ms, 3),
        "roofline": {"bound": "tensor", "kernel": "prefill_attention_kernel<128,128>",
                     "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "peak_source": peaks["source"] + " bf16 burst",
                     "traffic": traffic["bytes"] if traffic else None,
                     "algorithmic_flops_per_launch": attn_flops},
        "schedules": sched,
        "group_shared": group_shared,
        "output_aware_demands": output_aware,
        "topp": topp,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": round(e2e_s * 1e3, 3),
                "overlap": "double-buffered: copies of one step overlap another's compute",
                "host_link": host_link, "pipeline": pipeline},
        "gpu_launches": 5 * args.steps,
        "clocks": clk,
        "device_status": status,
    }
    if decode is not None:
        line["decode"] = decode
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, sample_seconds=12.0)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_decode(dev, stream):
    import numpy as np
    import torch

    import head_heterogeneous_block_gb300 as sa
    from head_heterogeneous_block_gb300.layer import DecodeStep
    from workloads import generate, workload

    w = workload(DECODE_WORKLOAD)
    x = generate.decode_inputs(w)
    t = {n: torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).to(dev) for n in "qkv"}
    kinds = generate.head_kinds(w)
    shape = sa.Shape.decode(w.seq_len, w.block, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.batch)
    # the serial step (every head's score, select and attention in turn, as
    # separate calls) gives the stage times; the default step (below) fuses
    # the retrieval heads' scoring and selection and overlaps the streaming heads
    step = DecodeStep(shape, w.budget_tokens // w.block, kinds, w.window_tokens // w.block,
                      device=dev, overlap=False, fused=False, one_launch=False)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step.build_cache(t["k"], stream=stream)
    for _ in range(3):
        step(t["q"], t["k"], t["v"], stream=stream)
    # flush L2 between decode steps (the cache is 2 GB but one step touches
    # ~0.5 GB, which would otherwise partly stay in L2) by reading a buffer
    # twice its size: reading leaves clean lines, so the next step's loads do
    # not pay for writing the flush back
    flush = torch.zeros(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    times, fwd, sco = [], [], []
    for _ in range(10):
        flush.max()
        e0, e1, e2, es = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        e0.record(stream)
        sa.sparse_attn_score(shape, t["q"], step.kbar, step.scores, None, 0, stream=stream)
        es.record(stream)
        sa.sparse_attn_select(shape, step.plan, step.scores, step.idx, step.cnt, step.kmax,
                              stream=stream)
        e1.record(stream)
        sa.sparse_attn_forward(shape, step.plan, t["q"], t["k"], t["v"], step.idx, step.cnt,
                               step.kmax, step.out, None, step.dev_status, stream=stream)
        e2.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e2))
        fwd.append(e1.elapsed_time(e2))
        sco.append(e0.elapsed_time(es))
    # the whole step without events between its kernels (an event between two
    # kernels keeps the second from being scheduled behind the first)
    whole = []
    for _ in range(10):
        flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(t["q"], t["k"], t["v"], stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        whole.append(e0.elapsed_time(e1))
    a.record(stream)
    step.build_cache(t["k"], stream=stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    # the fused scoring and selection of the retrieval heads alone
    fz = []
    for _ in range(20):
        flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sa.sparse_attn_score_select(shape, step.plan, t["q"], step.kbar, None, step.idx,
                                    step.cnt, step.kmax, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        fz.append(e0.elapsed_time(e1))

    def overlapped(fused, one_launch=False):
        # the streaming heads on a side stream beside the retrieval heads'
        # scoring and selection (fused into one launch, or apart); or the
        # whole step as one launch
        ov = DecodeStep(shape, w.budget_tokens // w.block, kinds, w.window_tokens // w.block,
                        device=dev, fused=fused, one_launch=one_launch)
        ov.build_cache(t["k"], stream=stream)
        for _ in range(3):
            ov(t["q"], t["k"], t["v"], stream=stream)
        ts = []
        for _ in range(20):
            flush.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ov(t["q"], t["k"], t["v"], stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return ov, ts

    ov, unfused_times = overlapped(False)
    unfused_status = int(ov.dev_status.item())
    del ov
    ov, fused_times = overlapped(True)
    unfused_status = max(unfused_status, int(ov.dev_status.item()))
    del ov
    # the default step: one launch
    ov, ov_times = overlapped(True, one_launch=True)
    ov_status = max(unfused_status, int(ov.dev_status.item()))
    # the default step captured once in a CUDA graph and replayed, as a
    # serving loop runs its decode steps
    graph_ms = None
    try:
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            ov(t["q"], t["k"], t["v"])
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            ov(t["q"], t["k"], t["v"])
        torch.cuda.synchronize(dev)
        for _ in range(3):
            g.replay()
        gr_times = []
        for _ in range(10):
            flush.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            gr_times.append(e0.elapsed_time(e1))
        graph_ms = round(statistics.mean(gr_times), 4)
        del g
    except RuntimeError as exc:   # capture refused: report it, keep the eager numbers
        graph_ms = f"capture failed: {str(exc)[:80]}"
    ov_status = max(ov_status, int(ov.dev_status.item()))
    del ov
    # touched bytes: union of selected blocks per (sequence, kv head), K and V
    idx = step.idx.view(w.batch, w.num_q_heads, step.kmax).cpu().numpy()
    cnt = step.cnt.view(w.batch, w.num_q_heads).cpu().numpy()
    G = w.group
    blocks = 0
    for bb in range(w.batch):
        for g in range(w.num_kv_heads):
            u = set()
            for h in range(g * G, (g + 1) * G):
                u.update(idx[bb, h, :cnt[bb, h]].tolist())
            blocks += len(u)
    kv_bytes = blocks * w.block * w.head_dim * 2 * 2
    kbar_bytes = w.batch * w.num_kv_heads * w.nb * w.head_dim * 4
    q_o = 2 * w.batch * w.num_q_heads * w.head_dim * 2
    fwd_ms = statistics.median(fwd)
    peaks = _peaks()
    # the whole step's compulsory DRAM bytes: pooled keys read by scoring, the
    # selected K/V (union per KV head) and q / o; the score rows (3.7 MB) and
    # index lists pass between kernels through L2 and are not counted
    step_bytes = kbar_bytes + kv_bytes + q_o
    step_ms = statistics.median(whole)
    # means: single launches are timed in steps of ~2 us here
    ov_ms = statistics.mean(ov_times)
    res = {"workload": w.name,
           "ms_per_step": round(ov_ms, 4),
           "step": "DecodeStep default: one launch (sparse_attn_decode_step): per (sequence, "
                   "KV group) a cluster scores and selects the retrieval heads, and each head "
                   "is attended by the warpgroup that selected it; the streaming heads by "
                   "the cluster's other warpgroups",
           "overlapped_ms_per_step": round(statistics.mean(fused_times), 4),
           "unfused_ms_per_step": round(statistics.mean(unfused_times), 4),
           "score_select_ms": round(statistics.mean(fz), 4),
           "graph_ms_per_step": graph_ms,
           "step_frac_hbm": round(step_bytes / (ov_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "device_status": ov_status,
           "serial": {"ms_per_step": round(step_ms, 4),
                      "ms_per_step_with_stage_events": round(statistics.median(times), 4),
                      "step_frac_hbm": round(step_bytes / (step_ms * 1e-3) / 1e9
                                             / peaks["hbm_gbs"], 4)},
           "score_ms": round(statistics.median(sco), 4),
           "select_ms": round(statistics.median(times) - statistics.median(sco) - fwd_ms, 4),
           "forward_ms": round(fwd_ms, 4),
           "forward_gbs": round((kv_bytes + q_o) / (fwd_ms * 1e-3) / 1e9, 1),
           "forward_frac_hbm": round((kv_bytes + q_o) / (fwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "touched_kv_bytes": kv_bytes, "kbar_bytes": kbar_bytes,
           "step_bytes": step_bytes,
           "step_floor_ms": round(step_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3, 4),
           "stages": "score_ms, select_ms and forward_ms time the serial step's kernels "
                     "between events (separate score and select calls); score_select_ms "
                     "times the fused launch alone; ms_per_step (one launch), "
                     "overlapped_ms_per_step (streaming heads on a side stream, the retrieval "
                     "heads' scoring and selection fused) and unfused_ms_per_step (the same "
                     "with separate score and select launches) are means over 20 steps",
           "kcache_pool_ms": round(a.elapsed_time(b), 4),
           "l2": "flushed between steps (a 256 MB read)"}
    del step
    with open(os.path.join(ROOT, "workloads", "demands.json")) as f:
        prof = json.load(f)[str(w.number)]["granularity"]
    res["block_sizes"] = bench_decode_block_sizes(w, t, kinds, shape, dev, stream, flush,
                                                  prof["gran"], prof["budget"])
    res["block_sizes"]["chosen_by"] = "fewest bytes per KV group"
    res["block_sizes"]["modelled_bytes_per_sequence"] = prof["bytes"]
    res["block_sizes"]["modelled_bytes_per_sequence_default"] = prof["bytes_default"]
    tm = prof["time_model"]
    res["block_sizes_time_model"] = bench_decode_block_sizes(w, t, kinds, shape, dev, stream,
                                                             flush, tm["gran"], tm["budget"])
    res["block_sizes_time_model"].update({
        "chosen_by": "least modelled step time (measured kernel rates, one scoring pass per "
                     "size, selection time by the longest row)",
        "modelled_us": tm["time_us"], "modelled_us_default": tm["time_us_default"]})
    return res


def bench_decode_block_sizes(w, t, kinds, shape, dev, stream, flush, gran, budget):
    """The decode step with each retrieval head's block size and budget chosen
    offline (every head keeps at least the default selection's attention
    mass), against the default step timed above."""
    import numpy as np
    import torch

    import head_heterogeneous_block_gb300 as sa
    from head_heterogeneous_block_gb300.layer import DecodeStep

    step = DecodeStep(shape, 2, kinds, w.window_tokens // w.block, device=dev,
                      granularity=gran, head_budget=budget)
    step.build_cache(t["k"], stream=stream)
    for _ in range(3):
        step(t["q"], t["k"], t["v"], stream=stream)
    times, fwd, sco = [], [], []
    for _ in range(10):
        flush.max()
        e0, e1, e2, es = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        e0.record(stream)
        sa.sparse_attn_score_plan(shape, step.plan, t["q"], step.kbar, step.scores, stream=stream)
        es.record(stream)
        sa.sparse_attn_select(shape, step.plan, step.scores, step.idx, step.cnt, step.kmax,
                              stream=stream)
        e1.record(stream)
        sa.sparse_attn_forward(shape, step.plan, t["q"], t["k"], t["v"], step.idx, step.cnt,
                               step.kmax, step.out, None, step.dev_status, stream=stream)
        e2.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e2))
        fwd.append(e1.elapsed_time(e2))
        sco.append(e0.elapsed_time(es))
    # the default (overlapped) step as a whole, as for the default sizes
    whole = []
    for _ in range(10):
        flush.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(t["q"], t["k"], t["v"], stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        whole.append(e0.elapsed_time(e1))
    # touched bytes: union of selected tokens per (sequence, kv head), K and V;
    # pooled keys: each block size a group's retrieval heads use, once
    idx = step.idx.view(w.batch, w.num_q_heads, step.kmax).cpu().numpy()
    cnt = step.cnt.view(w.batch, w.num_q_heads).cpu().numpy()
    size = [gran[h] if kinds[h] != 1 else w.block for h in range(w.num_q_heads)]
    G = w.group
    tokens = 0
    kbar_bytes = 0
    for g in range(w.num_kv_heads):
        used = {size[h] for h in range(g * G, (g + 1) * G) if kinds[h] != 1}
        kbar_bytes += w.batch * sum((w.seq_len // s) * w.head_dim * 4 for s in used)
        for bb in range(w.batch):
            mask = np.zeros(w.seq_len, bool)
            for h in range(g * G, (g + 1) * G):
                for j in idx[bb, h, :cnt[bb, h]].tolist():
                    mask[j * size[h]:(j + 1) * size[h]] = True
            tokens += int(mask.sum())
    status = int(step.dev_status.item())
    return {"ms_per_step": round(statistics.median(whole), 4),
            "serial_ms_per_step_with_stage_events": round(statistics.median(times), 4),
            "score_ms": round(statistics.median(sco), 4),
            "select_ms": round(statistics.median(times) - statistics.median(sco)
                               - statistics.median(fwd), 4),
            "forward_ms": round(statistics.median(fwd), 4),
            "touched_kv_bytes": tokens * w.head_dim * 2 * 2, "kbar_bytes": kbar_bytes,
            "sizes": sorted(set(size[h] for h in range(w.num_q_heads) if kinds[h] != 1)),
            "device_status": status}


def _sample_in_subprocess(steps: int, cores: int):
    """reference_sample in a child process restricted to `cores` host cores
    (CPU affinity and BLAS thread counts), so that numpy's thread pools start
    with that width."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    code = ("import json, os, sys; sys.path.insert(0, %r); "
            "os.sched_setaffinity(0, sorted(os.sched_getaffinity(0))[:%d]) "
            "if hasattr(os, 'sched_setaffinity') else None; "
            "import bench; print(json.dumps(bench.reference_sample(%d)))" % (ROOT, cores, steps))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-400:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def _layer_flops():
    """Algorithmic work of one headline layer (attention over every selected
    block plus block scoring), from the oracle's plan."""
    from oracle import plan as op
    from workloads import workload

    w = workload(WORKLOAD)
    prof = _profile(WORKLOAD)
    budgets = op.maxmin_shift(prof["k_uniform"], prof["demand"], prof["k_min"], w.nb)
    blocks = sum(op.kept_blocks(k, w.nb) for k in budgets)
    return _attention_flops(blocks, w.block, w.head_dim) + _score_flops(w), blocks


def cpu_baseline(args, sample_seconds: float):
    """The oracle, as it stands, on the host cores over a bounded sample: on
    all cores and on one, each extrapolated to the full layer."""
    all_cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    steps = max(1, int(sample_seconds // 4))
    full = _sample_in_subprocess(steps, all_cores)
    one = _sample_in_subprocess(max(1, steps // 2), 1)
    layer_flops, _ = _layer_flops()
    return {"value": full["value"], "unit": UNIT, "cores": full["cores"], "kind": "oracle",
            "sample": full["sample"],
            "one_core": {"value": one["value"], "unit": UNIT, "cores": one["cores"],
                         "sample": one["sample"]},
            "extrapolation": {
                "layer_tflop": round(layer_flops / 1e12, 4),
                "all_cores_s_per_layer": round(layer_flops / (full["value"] * 1e12), 1),
                "one_core_s_per_layer": round(layer_flops / (one["value"] * 1e12), 1),
                "how": "the layer's algorithmic work (selected-block attention plus block "
                       "scoring) over the sample's throughput; attention dominates both"}}


def reference_sample(steps: int):
    """Time the fp64 oracle on a sample of the headline workload and express it
    in the bench's unit (algorithmic TFLOP/s of the work actually done)."""
    import numpy as np

    from oracle import attention as oa
    from oracle import plan as op
    from workloads import generate, workload

    w = workload(WORKLOAD)
    prof = _profile(WORKLOAD)
    budgets = op.maxmin_shift(prof["k_uniform"], prof["demand"], prof["k_min"], w.nb)
    heads = [0]                                  # one head: pool, score, select in full
    x = generate.prefill_inputs(w, heads=heads, kv_heads=[0])
    q = generate.bf16_to_f32(x["q"][0])
    k = generate.bf16_to_f32(x["k"][0])
    v = generate.bf16_to_f32(x["v"][0])
    rng = np.random.default_rng(0)
    items_per_step = 24
    flops = 0.0
    t0 = time.perf_counter()
    for s in range(steps):
        qb = oa.pool_blocks(q[None], w.block)
        kb = oa.pool_blocks(k[None], w.block)
        sc = oa.block_scores(qb, kb, 1)
        rows = rng.integers(0, w.nb, items_per_step)
        for i in rows:
            sel = oa.select_row(sc[0, i], int(i), budgets[0])
            oa.attend_item(q, k, v, int(i), sel, w.block)
            flops += _attention_flops(len(sel), w.block, w.head_dim)
        flops += 2.0 * (w.nb * (w.nb + 1) / 2) * w.head_dim
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(flops / dt / 1e12, 6), "seconds": dt, "cores": cores,
            "sample": f"{steps} x (head 0: pool+score {w.nb}x{w.nb} blocks, "
                      f"{items_per_step} random query blocks selected and attended) of "
                      f"{w.name}; fp64 numpy (BLAS threads)"}


def workload_config(w, total_blocks: int, ws: int) -> dict:
    """The workload as both arms name it in their JSON line."""
    return {"workload": w.name, "seq_len": w.seq_len, "block": w.block,
            "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "mean_density": round(total_blocks / (w.num_q_heads * w.nb * (w.nb + 1) / 2), 5),
            "selected_blocks": total_blocks,
            "budgets": "calibrated per head, Max-Min shifted (workloads/demands.json)",
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{ws}"}


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return
    from workloads import workload
    w = workload(WORKLOAD)
    for _ in range(args.warmup):
        reference_sample(1)
    t0 = time.perf_counter()
    res = [reference_sample(1) for _ in range(args.steps)]
    total = time.perf_counter() - t0
    value = statistics.mean(r["value"] for r in res)
    layer_flops, blocks = _layer_flops()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16, per-head query scales; calibrated budgets)",
        "impl": "reference",
        "config": workload_config(w, blocks, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                         "cores": res[0]["cores"], "sample": res[0]["sample"],
                         "extrapolation": {"layer_tflop": round(layer_flops / 1e12, 4),
                                           "s_per_layer": round(layer_flops / (value * 1e12), 1)}},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--schedule", default="lpt_grouped",
                    choices=["lpt", "lpt_grouped", "head_order"])
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=[1, 2, 3, 4],
                    help="prefill workload (3, the 128K Llama-3.1-8B shape, is the headline; "
                         "the others serve small profiling captures)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the group-shared, output-aware and top-p variants")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
