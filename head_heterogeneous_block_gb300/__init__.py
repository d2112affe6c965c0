"""Per-head-budget block-sparse attention on GB300 (sm_103a).

Thin ctypes binding of ``libsparse_attn.so`` (C ABI in ``include/sparse_attn.h``).
Functions keep the C names; they only marshal arguments (torch tensors or raw
integer device pointers, streams) and raise ``SparseAttnError`` on a non-zero
status.  Every step of the computation runs in the library's CUDA kernels;
there is no Python or CPU fallback -- importing fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from ._build import LIB

__all__ = [
    "Shape", "Plan", "SparseAttnError", "sparse_attn_plan", "sparse_attn_score",
    "sparse_attn_score_workspace_size", "sparse_attn_select", "sparse_attn_forward",
    "sparse_attn_pool_kcache", "sa_status_string", "library_path",
    "sparse_attn_select_topp", "sparse_attn_pool_kcache_plan", "sparse_attn_score_plan",
    "sparse_attn_set_wait_limit", "sparse_attn_select_kind", "sparse_attn_forward_kind",
    "sparse_attn_score_select",
    "sparse_attn_decode_step",
]

SA_OK = 0
SA_MODE_PREFILL, SA_MODE_DECODE = 0, 1
SA_SCHED_LPT, SA_SCHED_LPT_GROUPED, SA_SCHED_HEAD_ORDER = 0, 1, 2
SCHEDULES = {"lpt": SA_SCHED_LPT, "lpt_grouped": SA_SCHED_LPT_GROUPED,
             "head_order": SA_SCHED_HEAD_ORDER}
SA_HEAD_RETRIEVAL, SA_HEAD_STREAMING = 0, 1
SA_DTYPE_BF16, SA_DTYPE_F32 = 0, 1
SA_DEV_BAD_INDEX, SA_DEV_BAD_COUNT, SA_DEV_TIMEOUT, SA_DEV_BAD_ITEM, SA_DEV_BAD_LAUNCH = 1, 2, 4, 8, 16
SA_DEV_RANGE = 32


class Shape(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int64), ("block", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("mode", ctypes.c_int32)]

    @property
    def nb(self) -> int:
        return self.seq_len // self.block

    @staticmethod
    def prefill(seq_len, block, num_q_heads, num_kv_heads, head_dim) -> "Shape":
        return Shape(seq_len, block, num_q_heads, num_kv_heads, head_dim, 1, SA_MODE_PREFILL)

    @staticmethod
    def decode(cache_len, block, num_q_heads, num_kv_heads, head_dim, batch) -> "Shape":
        return Shape(cache_len, block, num_q_heads, num_kv_heads, head_dim, batch, SA_MODE_DECODE)


class _PlanParams(ctypes.Structure):
    _fields_ = [("demand", ctypes.POINTER(ctypes.c_int32)), ("k_uniform", ctypes.c_int32),
                ("k_min", ctypes.c_int32), ("head_kind", ctypes.POINTER(ctypes.c_uint8)),
                ("window_blocks", ctypes.c_int32), ("num_workers", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("group_shared", ctypes.c_int32),
                ("granularity", ctypes.POINTER(ctypes.c_int32)),
                ("head_budget", ctypes.POINTER(ctypes.c_int32)),
                ("share_kv", ctypes.c_int32)]


class SparseAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {sa_status_string(status)} (status {status})")


def library_path() -> str:
    return LIB


def _load():
    if not os.path.exists(LIB):
        raise ImportError(f"{LIB} is missing: build it with __graft_entry__.build() "
                          "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(LIB)
    P = ctypes.c_void_p
    I32, I64, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "sa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "sparse_attn_plan": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(_PlanParams),
                                            ctypes.POINTER(P)]),
        "sparse_attn_plan_info": (ctypes.c_int, [P, ctypes.POINTER(I32), ctypes.POINTER(I32),
                                                 ctypes.POINTER(I32), ctypes.POINTER(I64),
                                                 ctypes.POINTER(I64)]),
        "sparse_attn_plan_get": (ctypes.c_int, [P, P, P, P, P]),
        "sparse_attn_plan_upload": (ctypes.c_int, [P, P]),
        "sparse_attn_plan_destroy": (None, [P]),
        "sparse_attn_score_workspace_size": (ctypes.c_int, [ctypes.POINTER(Shape),
                                                            ctypes.POINTER(SZ)]),
        "sparse_attn_score": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, SZ, P]),
        "sparse_attn_select": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, I32, P]),
        "sparse_attn_forward": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, P, P, I32,
                                               P, I32, P, P, P]),
        "sparse_attn_pool_kcache": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P]),
        "sparse_attn_select_topp": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, ctypes.c_float,
                                                   P, P, I32, P]),
        "sparse_attn_plan_rebuild": (ctypes.c_int, [P, P, P]),
        "sparse_attn_plan_device_schedule": (ctypes.c_int, [P, P, P, P]),
        "sparse_attn_plan_decode_layout": (ctypes.c_int, [P, ctypes.POINTER(I32), P,
                                                          ctypes.POINTER(I64),
                                                          ctypes.POINTER(I32)]),
        "sparse_attn_pool_kcache_plan": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P]),
        "sparse_attn_score_plan": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, P]),
        "sparse_attn_set_wait_limit": (ctypes.c_int, [ctypes.c_uint64]),
        "sparse_attn_select_kind": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, I32, I32,
                                                   P]),
        "sparse_attn_forward_kind": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, P, P,
                                                    I32, P, I32, P, P, I32, P]),
        "sparse_attn_score_select": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, P, P,
                                                    I32, P]),
        "sparse_attn_decode_step": (ctypes.c_int, [ctypes.POINTER(Shape), P, P, P, P, P, P, P,
                                                   P, I32, P, I32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def sa_status_string(status: int) -> str:
    return _lib.sa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != SA_OK:
        raise SparseAttnError(status, where)


def _ptr(x):
    """Device (or host) address of a tensor / array / int; None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if not x.flags.c_contiguous:
            raise ValueError("array must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owner of an ``sa_plan*`` (budgets, head kinds and worker schedule)."""

    def __init__(self, handle: int, shape: Shape):
        self._h = ctypes.c_void_p(handle)
        self.shape = shape

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        w, n, k = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        t, m = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.sparse_attn_plan_info(self._h, ctypes.byref(w), ctypes.byref(n),
                                          ctypes.byref(k), ctypes.byref(t), ctypes.byref(m)),
               "sparse_attn_plan_info")
        return {"num_workers": w.value, "num_items": n.value, "kmax": k.value,
                "total_blocks": t.value, "makespan": m.value}

    def get(self) -> dict:
        inf = self.info()
        budgets = np.zeros(self.shape.num_q_heads, np.int32)
        wptr = np.zeros(inf["num_workers"] + 1, np.int32)
        nitems = inf["num_items"] if inf["num_workers"] else 0
        items = np.zeros(max(nitems, 1), np.int32)
        loads = np.zeros(max(inf["num_workers"], 1), np.int64)
        _check(_lib.sparse_attn_plan_get(self._h, budgets.ctypes.data, wptr.ctypes.data,
                                         items.ctypes.data, loads.ctypes.data),
               "sparse_attn_plan_get")
        return {"budgets": budgets, "wptr": wptr, "items": items[:nitems],
                "loads": loads[:inf["num_workers"]], **inf}

    def upload(self, stream=None):
        _check(_lib.sparse_attn_plan_upload(self._h, _stream(stream)), "sparse_attn_plan_upload")

    def rebuild(self, cnt, stream=None):
        """LPT schedule rebuilt on the GPU from device block counts cnt [Hq*nb]."""
        _check(_lib.sparse_attn_plan_rebuild(self._h, _ptr(cnt), _stream(stream)),
               "sparse_attn_plan_rebuild")

    def device_schedule(self, wptr, items, stream=None):
        """Copy the device schedule (wptr [W+1], items [N]) into the given buffers."""
        _check(_lib.sparse_attn_plan_device_schedule(self._h, _ptr(wptr), _ptr(items),
                                                     _stream(stream)),
               "sparse_attn_plan_device_schedule")

    def decode_layout(self) -> dict:
        """Decode: the retrieval heads' block sizes, the floats of their pooled
        key caches together, and the score row stride."""
        n, floats, stride = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
        sizes = np.zeros(8, np.int32)
        _check(_lib.sparse_attn_plan_decode_layout(self._h, ctypes.byref(n), sizes.ctypes.data,
                                                   ctypes.byref(floats), ctypes.byref(stride)),
               "sparse_attn_plan_decode_layout")
        return {"sizes": [int(x) for x in sizes[:n.value]], "kcache_floats": floats.value,
                "score_stride": stride.value}

    def close(self):
        if self._h is not None and self._h.value:
            _lib.sparse_attn_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sparse_attn_plan(shape: Shape, k_uniform: int, demand=None, k_min: int = 2,
                     head_kind=None, window_blocks: int = 0, num_workers: int = 152,
                     schedule="lpt", group_shared: bool = False, granularity=None,
                     head_budget=None, share_kv: bool = False) -> Plan:
    if isinstance(schedule, str):
        schedule = SCHEDULES[schedule]
    params = _PlanParams()
    keep = []
    if demand is not None:
        d = np.ascontiguousarray(demand, dtype=np.int32)
        keep.append(d)
        params.demand = d.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    if head_kind is not None:
        hk = np.ascontiguousarray(head_kind, dtype=np.uint8)
        keep.append(hk)
        params.head_kind = hk.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))
    for name, arr in (("granularity", granularity), ("head_budget", head_budget)):
        if arr is not None:
            a = np.ascontiguousarray(arr, dtype=np.int32)
            keep.append(a)
            setattr(params, name, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    params.k_uniform = k_uniform
    params.k_min = k_min
    params.window_blocks = window_blocks
    params.num_workers = num_workers
    params.schedule = schedule
    params.group_shared = 1 if group_shared else 0
    params.share_kv = 1 if share_kv else 0
    out = ctypes.c_void_p()
    _check(_lib.sparse_attn_plan(ctypes.byref(shape), ctypes.byref(params), ctypes.byref(out)),
           "sparse_attn_plan")
    return Plan(out.value, shape)


def sparse_attn_score_workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t()
    _check(_lib.sparse_attn_score_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "sparse_attn_score_workspace_size")
    return n.value


def sparse_attn_score(shape: Shape, q, k, scores, ws=None, ws_bytes: int | None = None,
                      stream=None):
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if hasattr(ws, "numel") else 0
    _check(_lib.sparse_attn_score(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(scores), _ptr(ws),
                                  ws_bytes, _stream(stream)), "sparse_attn_score")


def sparse_attn_select(shape: Shape, plan: Plan, scores, idx, cnt, kmax: int, stream=None):
    _check(_lib.sparse_attn_select(ctypes.byref(shape), plan.handle, _ptr(scores), _ptr(idx),
                                   _ptr(cnt), kmax, _stream(stream)), "sparse_attn_select")


def sparse_attn_select_kind(shape: Shape, plan: Plan, scores, idx, cnt, kmax: int, head_kind: int,
                            stream=None):
    """Decode: the selection of the heads of one kind only."""
    _check(_lib.sparse_attn_select_kind(ctypes.byref(shape), plan.handle, _ptr(scores), _ptr(idx),
                                        _ptr(cnt), kmax, int(head_kind), _stream(stream)),
           "sparse_attn_select_kind")


def sparse_attn_score_select(shape: Shape, plan: Plan, q, kbar, scores, idx, cnt, kmax: int,
                             stream=None):
    """Decode: scores and selection of the retrieval heads in one launch
    (``scores`` may be None)."""
    _check(_lib.sparse_attn_score_select(ctypes.byref(shape), plan.handle, _ptr(q), _ptr(kbar),
                                         _ptr(scores), _ptr(idx), _ptr(cnt), kmax,
                                         _stream(stream)),
           "sparse_attn_score_select")


def sparse_attn_select_topp(shape: Shape, plan: Plan, scores, p: float, idx, cnt, kmax: int,
                            stream=None):
    _check(_lib.sparse_attn_select_topp(ctypes.byref(shape), plan.handle, _ptr(scores),
                                        float(p), _ptr(idx), _ptr(cnt), kmax, _stream(stream)),
           "sparse_attn_select_topp")


def _out_dtype(o, o_dtype):
    if o_dtype is not None:
        return o_dtype
    name = str(getattr(o, "dtype", ""))
    if name.endswith("float32"):
        return SA_DTYPE_F32
    if name.endswith("bfloat16"):
        return SA_DTYPE_BF16
    raise TypeError("output must be bfloat16 or float32 (or pass o_dtype)")


def sparse_attn_forward(shape: Shape, plan, q, k, v, idx, cnt, kmax: int, o, lse, dev_status,
                        stream=None, o_dtype=None):
    _check(_lib.sparse_attn_forward(ctypes.byref(shape), plan.handle if plan else None, _ptr(q),
                                    _ptr(k), _ptr(v), _ptr(idx), _ptr(cnt), kmax, _ptr(o),
                                    _out_dtype(o, o_dtype), _ptr(lse), _ptr(dev_status),
                                    _stream(stream)),
           "sparse_attn_forward")


def sparse_attn_decode_step(shape: Shape, plan: Plan, q, kbar, k, v, scores, idx, cnt, kmax: int,
                            o, lse, dev_status, stream=None, o_dtype=None):
    """Decode: the whole step (scores and selection of the retrieval heads,
    the streaming heads' lists, every row's attention) in one launch
    (``scores`` and ``lse`` may be None)."""
    _check(_lib.sparse_attn_decode_step(ctypes.byref(shape), plan.handle, _ptr(q), _ptr(kbar),
                                        _ptr(k), _ptr(v), _ptr(scores), _ptr(idx), _ptr(cnt),
                                        kmax, _ptr(o), _out_dtype(o, o_dtype), _ptr(lse),
                                        _ptr(dev_status), _stream(stream)),
           "sparse_attn_decode_step")


def sparse_attn_forward_kind(shape: Shape, plan: Plan, q, k, v, idx, cnt, kmax: int, o, lse,
                             dev_status, head_kind: int, stream=None, o_dtype=None):
    """Decode: the attention of the heads of one kind only."""
    _check(_lib.sparse_attn_forward_kind(ctypes.byref(shape), plan.handle, _ptr(q), _ptr(k),
                                         _ptr(v), _ptr(idx), _ptr(cnt), kmax, _ptr(o),
                                         _out_dtype(o, o_dtype), _ptr(lse), _ptr(dev_status),
                                         int(head_kind), _stream(stream)),
           "sparse_attn_forward_kind")


def sparse_attn_pool_kcache(shape: Shape, k, kbar, stream=None):
    _check(_lib.sparse_attn_pool_kcache(ctypes.byref(shape), _ptr(k), _ptr(kbar),
                                        _stream(stream)), "sparse_attn_pool_kcache")


def sparse_attn_pool_kcache_plan(shape: Shape, plan: Plan, k, kbar_all, stream=None):
    """Pooled key caches at every block size of the plan's retrieval heads."""
    _check(_lib.sparse_attn_pool_kcache_plan(ctypes.byref(shape), plan.handle, _ptr(k),
                                             _ptr(kbar_all), _stream(stream)),
           "sparse_attn_pool_kcache_plan")


def sparse_attn_score_plan(shape: Shape, plan: Plan, q, kbar_all, scores, stream=None):
    """Decode scores of each retrieval head at its own block size."""
    _check(_lib.sparse_attn_score_plan(ctypes.byref(shape), plan.handle, _ptr(q),
                                       _ptr(kbar_all), _ptr(scores), _stream(stream)),
           "sparse_attn_score_plan")


def sparse_attn_set_wait_limit(ns: int):
    """Limit, in ns, of every wait inside the prefill forward kernel for later
    launches (0: the 4 s default).  A wait that runs out sets SA_DEV_TIMEOUT in
    the launch's status word; the kernel cleans up and returns."""
    _check(_lib.sparse_attn_set_wait_limit(int(ns)), "sparse_attn_set_wait_limit")


_noalloc = None


def sparse_attn_score_noalloc(shape: Shape, q, k, scores, stream=None):
    """Pooled block scores without a workspace (the library's fixed 32 MiB
    scratch area); see the C declaration for the limit and the rules on
    overlapping calls."""
    global _noalloc
    if _noalloc is None:
        fn = _lib.sparse_attn_score_noalloc
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.POINTER(Shape), ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_void_p]
        _noalloc = fn
    _check(_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(scores), _stream(stream)),
           "sparse_attn_score_noalloc")
