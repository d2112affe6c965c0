"""Whole-layer drivers over the C ABI: buffers come from PyTorch, every step of
the computation runs in libsparse_attn's kernels.

``PrefillLayer``  Index -> Select -> Attention for one prefill layer
                  (score, select, forward) on a plan built once per
                  configuration (the offline profile gives the demands).
``DecodeStep``    the same three calls for one decode step over an
                  HBM-resident cache, with the pooled key cache built once.
"""
from __future__ import annotations

import torch

from . import (SA_HEAD_RETRIEVAL, SA_HEAD_STREAMING, Shape, sparse_attn_forward,
               sparse_attn_forward_kind, sparse_attn_plan, sparse_attn_pool_kcache,
               sparse_attn_pool_kcache_plan, sparse_attn_score, sparse_attn_score_plan,
               sparse_attn_score_select, sparse_attn_score_workspace_size, sparse_attn_select,
               sparse_attn_decode_step,
               sparse_attn_select_kind)


class PrefillLayer:
    def __init__(self, shape: Shape, k_uniform: int, demand=None, k_min: int = 2,
                 num_workers: int | None = None, schedule="lpt_grouped", device="cuda",
                 with_lse: bool = False, out_dtype=torch.bfloat16, group_shared: bool = False,
                 share_kv: bool = False):
        dev = torch.device(device)
        if num_workers is None:
            num_workers = torch.cuda.get_device_properties(dev).multi_processor_count
        self.shape = shape
        self.plan = sparse_attn_plan(shape, k_uniform, demand=demand, k_min=k_min,
                                     num_workers=num_workers, schedule=schedule,
                                     group_shared=group_shared, share_kv=share_kv)
        self.plan.upload()
        info = self.plan.info()
        self.kmax = info["kmax"]
        self.total_blocks = info["total_blocks"]
        H, nb, S, d = shape.num_q_heads, shape.nb, shape.seq_len, shape.head_dim
        self.scores = torch.empty(H * nb * nb, dtype=torch.float32, device=dev)
        ws = sparse_attn_score_workspace_size(shape)
        self.ws = torch.empty(ws // 4 + 1, dtype=torch.float32, device=dev)
        self.idx = torch.empty(H * nb * self.kmax, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(H * nb, dtype=torch.int32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lse = torch.empty(H * S, dtype=torch.float32, device=dev) if with_lse else None
        self.out = torch.empty(H, S, d, dtype=out_dtype, device=dev)

    def score(self, q, k, stream=None):
        sparse_attn_score(self.shape, q, k, self.scores, self.ws, stream=stream)

    def select(self, stream=None):
        sparse_attn_select(self.shape, self.plan, self.scores, self.idx, self.cnt, self.kmax,
                           stream=stream)

    def attend(self, q, k, v, out=None, stream=None):
        out = self.out if out is None else out
        sparse_attn_forward(self.shape, self.plan, q, k, v, self.idx, self.cnt, self.kmax, out,
                            self.lse, self.dev_status, stream=stream)
        return out

    def __call__(self, q, k, v, out=None, stream=None):
        self.score(q, k, stream)
        self.select(stream)
        return self.attend(q, k, v, out, stream)


class DecodeStep:
    """One decode step: pooled key cache (built once), scores, selection and
    attention.  With ``granularity`` (and ``head_budget``) each retrieval head
    selects ``head_budget[h]`` blocks of ``granularity[h]`` tokens.

    By default (``one_launch``, for plans without per-head block sizes and
    with 32-token blocks) the whole step is one launch
    (``sparse_attn_decode_step``): each head is attended by the warpgroup
    that selected it, as soon as its list is known.  Otherwise, with
    ``overlap`` the streaming heads, whose block lists do not depend on the
    scores, are selected and attended on a side stream while the retrieval
    heads score, select and attend on the caller's stream; the step ends
    when both are done.  ``overlap=False`` runs the calls for every head in
    turn on the caller's stream.  With ``fused`` (plans without per-head
    block sizes) the retrieval heads' scores and selection are one launch
    (``sparse_attn_score_select``); ``fused=False`` runs the score and
    select calls apart.  The results are the same bit for bit; the streaming
    heads' rows of ``scores`` are written only when neither fused nor one
    launch."""

    def __init__(self, shape: Shape, budget_blocks: int, head_kind, window_blocks: int,
                 device="cuda", with_lse: bool = False, out_dtype=torch.bfloat16,
                 granularity=None, head_budget=None, overlap: bool = True, fused: bool = True,
                 one_launch: bool = True):
        dev = torch.device(device)
        self.shape = shape
        self.overlap = overlap
        self.fused = fused and granularity is None
        self.one_launch = one_launch and granularity is None and shape.block == 32
        if overlap:
            self.side = torch.cuda.Stream(device=dev)
        self.plan = sparse_attn_plan(shape, budget_blocks, head_kind=head_kind,
                                     window_blocks=window_blocks, num_workers=1,
                                     granularity=granularity, head_budget=head_budget)
        self.plan.upload()
        self.kmax = self.plan.info()["kmax"]
        self.sized = granularity is not None
        layout = self.plan.decode_layout()
        self.score_stride = layout["score_stride"]
        Bt, H, Hkv, nb, d = (shape.batch, shape.num_q_heads, shape.num_kv_heads, shape.nb,
                             shape.head_dim)
        kfloats = max(1, layout["kcache_floats"]) if self.sized else Bt * Hkv * nb * d
        self.kbar = torch.empty(kfloats, dtype=torch.float32, device=dev)
        self.scores = torch.empty(Bt * H * self.score_stride, dtype=torch.float32, device=dev)
        self.idx = torch.empty(Bt * H * self.kmax, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(Bt * H, dtype=torch.int32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lse = torch.empty(Bt * H, dtype=torch.float32, device=dev) if with_lse else None
        self.out = torch.empty(Bt, H, d, dtype=out_dtype, device=dev)

    def build_cache(self, k, stream=None):
        if self.sized:
            sparse_attn_pool_kcache_plan(self.shape, self.plan, k, self.kbar, stream=stream)
        else:
            sparse_attn_pool_kcache(self.shape, k, self.kbar, stream=stream)

    def __call__(self, q, k, v, out=None, stream=None):
        out = self.out if out is None else out
        if self.one_launch:
            sparse_attn_decode_step(self.shape, self.plan, q, self.kbar, k, v, self.scores,
                                    self.idx, self.cnt, self.kmax, out, self.lse,
                                    self.dev_status, stream=stream)
            return out
        if self.overlap:
            return self._overlapped(q, k, v, out, stream)
        if self.fused:
            self._score_select(q, stream)
            sparse_attn_select_kind(self.shape, self.plan, None, self.idx, self.cnt, self.kmax,
                                    SA_HEAD_STREAMING, stream=stream)
        else:
            self._score(q, stream)
            sparse_attn_select(self.shape, self.plan, self.scores, self.idx, self.cnt, self.kmax,
                               stream=stream)
        sparse_attn_forward(self.shape, self.plan, q, k, v, self.idx, self.cnt, self.kmax, out,
                            self.lse, self.dev_status, stream=stream)
        return out

    def _score_select(self, q, stream):
        sparse_attn_score_select(self.shape, self.plan, q, self.kbar, self.scores, self.idx,
                                 self.cnt, self.kmax, stream=stream)

    def _score(self, q, stream):
        if self.sized:
            sparse_attn_score_plan(self.shape, self.plan, q, self.kbar, self.scores, stream=stream)
        else:
            sparse_attn_score(self.shape, q, self.kbar, self.scores, None, 0, stream=stream)

    def _overlapped(self, q, k, v, out, stream):
        main = torch.cuda.current_stream() if stream is None else stream
        self.side.wait_stream(main)
        # streaming heads: fixed lists, attended beside the scoring
        sparse_attn_select_kind(self.shape, self.plan, None, self.idx, self.cnt, self.kmax,
                                SA_HEAD_STREAMING, stream=self.side)
        sparse_attn_forward_kind(self.shape, self.plan, q, k, v, self.idx, self.cnt, self.kmax,
                                 out, self.lse, self.dev_status, SA_HEAD_STREAMING,
                                 stream=self.side)
        # retrieval heads: scores, top-k, attention
        if self.fused:
            self._score_select(q, main)
        else:
            self._score(q, main)
            sparse_attn_select_kind(self.shape, self.plan, self.scores, self.idx, self.cnt,
                                    self.kmax, SA_HEAD_RETRIEVAL, stream=main)
        sparse_attn_forward_kind(self.shape, self.plan, q, k, v, self.idx, self.cnt, self.kmax,
                                 out, self.lse, self.dev_status, SA_HEAD_RETRIEVAL, stream=main)
        main.wait_stream(self.side)
        return out


class HostPipeline:
    """A PrefillLayer over a sequence of host-resident (pinned) steps, with
    each step's host-to-device copies and the previous step's device-to-host
    read overlapped with compute.

    Two device buffer sets alternate.  Step s copies its Q, K and V into set
    s % 2 on a copy-in stream once the compute of step s - 2 (the last reader
    of that set) is done; the layer runs on the compute stream once the
    copies are in and the read-back of step s - 2's output is done; the
    output is copied to the step's host buffer on a copy-out stream.  Every
    step still moves all of its inputs and its result across the link; only
    the order in time changes.
    """

    def __init__(self, layer: "PrefillLayer", device="cuda"):
        dev = torch.device(device)
        s = layer.shape
        H, Hkv, S, d = s.num_q_heads, s.num_kv_heads, s.seq_len, s.head_dim
        self.layer = layer
        self.bufs = [{"q": torch.empty(H, S, d, dtype=torch.bfloat16, device=dev),
                      "k": torch.empty(Hkv, S, d, dtype=torch.bfloat16, device=dev),
                      "v": torch.empty(Hkv, S, d, dtype=torch.bfloat16, device=dev),
                      "o": torch.empty_like(layer.out)} for _ in range(2)]
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        self.dev = dev

    def run(self, steps, stream=None, before_step=None, timeline=None):
        """steps: iterable of (q, k, v, o) pinned host tensors; o receives the
        step's output.  before_step(s), if given, runs on the host before
        step s is issued.  Returns once every output is on the host.
        timeline: if a list, each step appends its copy-in, compute and
        copy-out spans as (start, end) pairs of timing events recorded on the
        three streams (events between operations; for diagnosis, not for the
        timed steps)."""
        comp = torch.cuda.current_stream(self.dev) if stream is None else stream
        timed = timeline is not None

        def mark(st):
            if not timed:
                return None
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
            return e

        done = [None, None]       # compute of the last step that used each set
        read = [None, None]       # read-back of the last output of each set
        for s, (qh, kh, vh, oh) in enumerate(steps):
            if before_step is not None:
                before_step(s)
            b = s % 2
            buf = self.bufs[b]
            with torch.cuda.stream(self.copy_in):
                if done[b] is not None:
                    self.copy_in.wait_event(done[b])
                in0 = mark(self.copy_in)
                buf["q"].copy_(qh, non_blocking=True)
                buf["k"].copy_(kh, non_blocking=True)
                buf["v"].copy_(vh, non_blocking=True)
                copied = torch.cuda.Event(enable_timing=timed)
                copied.record(self.copy_in)
            comp.wait_event(copied)
            if read[b] is not None:
                comp.wait_event(read[b])
            c0 = mark(comp)
            self.layer(buf["q"], buf["k"], buf["v"], out=buf["o"], stream=comp)
            done[b] = torch.cuda.Event(enable_timing=timed)
            done[b].record(comp)
            with torch.cuda.stream(self.copy_out):
                self.copy_out.wait_event(done[b])
                out0 = mark(self.copy_out)
                oh.copy_(buf["o"], non_blocking=True)
                read[b] = torch.cuda.Event(enable_timing=timed)
                read[b].record(self.copy_out)
            if timed:
                timeline.append({"in": (in0, copied), "compute": (c0, done[b]),
                                 "out": (out0, read[b])})
        self.copy_out.synchronize()
        self.copy_in.synchronize()
        comp.synchronize()
