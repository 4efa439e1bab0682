"""Python binding of libmarble: exact mask-aware blockwise attention over packed
multimodal sequences with the online-softmax state carried in fp32 across KV shards.

This module only marshals arguments to the C ABI declared in ``include/marble.h``; every
step of the computation runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  There is no CPU fallback: importing works without a GPU, but every
call needs the built library (``__graft_entry__.build()``) and a CUDA device.

Sources (page title and section): "MARBLE: exact sequence parallelism for packed
multimodal masks" s01 (tracks and mask), s03 (block classification, PTRR, exact ring
accumulation), s04 (sparse all-to-all, layout transforms).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

# The library queues work on up to five streams of its own (four side streams and a teardown
# stream) beside the caller's.  With CUDA's default of 8 hardware work queues, streams share
# queues, and work on one waits behind unrelated work on another: in a training loop the
# input and output copies then wait for the attention kernels.  More queues are asked for
# here, before the CUDA context exists, unless the caller chose a value; it has no effect if
# the process created its CUDA context before importing this module.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmarble.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT = range(6)
BLOCK = 128
WINDOW_INF = 2147483647
TILE_FULL, TILE_PARTIAL = 1, 2
KV_NEEDED = -1
STEP_FIRST = 1
STEP_BF16_MERGE = 2  # standard ring merge in bf16 (the comparison baseline)
STEP_FP32_MERGE = 4  # merge of fp32 partials by their LSE
_MERGE = {None: 0, "carried": 0, "bf16": STEP_BF16_MERGE, "fp32": STEP_FP32_MERGE}
ORDERS = {"contiguous": 0, "ptrr_block": 1, "ptrr_chunk": 2, "chunk_search": 3}
FIELDS = {
    "perm": (0, "int32"), "block_perm": (1, "int32"), "tracks_perm": (2, "int32"),
    "tile_rowptr": (3, "int64"), "tile_col": (4, "int32"), "tile_tag": (5, "uint8"),
    "step_ptr": (6, "int64"), "step_col": (7, "int32"), "step_tag": (8, "uint8"),
    "colT_ptr": (9, "int64"), "colT_row": (10, "int32"), "colT_tag": (11, "uint8"),
    "needed_ptr": (12, "int64"), "needed": (13, "int32"),
    "key_intervals": (14, "int32"), "interval_blocks": (15, "uint8"),
}


class MarbleError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"marble error {status}: {msg}")
        self.status = status


class _PlanDesc(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("sample_id", ctypes.c_void_p),
                ("seg_id", ctypes.c_void_p), ("noise_id", ctypes.c_void_p),
                ("window", ctypes.c_int32), ("num_shards", ctypes.c_int32),
                ("order", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32),
                ("range_cost", ctypes.c_int64), ("no_key_intervals", ctypes.c_int32),
                ("pos_id", ctypes.c_void_p)]


class _PlanStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "n_tokens", "n_blocks", "num_shards", "nnz", "n_full", "n_partial", "legal_pairs",
        "shard_cost_max", "shard_cost_sum", "step_cost", "needed_total", "needed_remote",
        "chunks_per_rank", "layout_cost", "layout_step_cost", "step_cost_pairs")]


class _QKV(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class _State(ctypes.Structure):
    _fields_ = [("o_acc", ctypes.c_void_p), ("m", ctypes.c_void_p), ("l", ctypes.c_void_p)]


_lib = None

# every symbol the header declares, with its ctypes signature
_SIGS = {
    "marble_plan": ([ctypes.POINTER(_PlanDesc), ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "marble_plan_destroy": ([ctypes.c_void_p]),
    "marble_plan_stats": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_PlanStats)]),
    "marble_layout_vision_groups": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_void_p]),
    "marble_chunk_layout_search": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "marble_plan_field_bytes": ([ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "marble_plan_export": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                            ctypes.c_void_p]),
    "marble_permute": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                        ctypes.c_int32, ctypes.c_void_p]),
    "marble_permute_cast_bf16": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]),
    "marble_release_memory": ([]),
    "marble_attn_step": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.c_int32, ctypes.c_int32,
                          ctypes.POINTER(_State), ctypes.c_uint32, ctypes.c_void_p]),
    "marble_attn_finalize": ([ctypes.c_void_p, ctypes.POINTER(_State), ctypes.c_int32,
                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "marble_attn_bwd_prep": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "marble_attn_bwd": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.c_void_p, ctypes.c_void_p,
                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]),
    "marble_attn_steps": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.c_int32,
                           ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                           ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(_State),
                           ctypes.c_void_p]),
    "marble_attn_bwd_steps": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                               ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p]),
    "marble_attn_fwd_fused": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.POINTER(_State),
                               ctypes.c_void_p]),
    "marble_attn_bwd_fused": ([ctypes.c_void_p, ctypes.POINTER(_QKV), ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "marble_cast_bf16": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    "marble_check": ([ctypes.c_void_p, ctypes.c_void_p]),
    "marble_set_wait_limit_ns": ([ctypes.c_uint64]),
    "marble_set_side_streams": ([ctypes.c_int32]),
    "marble_debug_wait_timeout": ([ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]),
    "marble_timing_enable": ([ctypes.c_int]),
    "marble_timing_read": ([ctypes.c_void_p]),
    "marble_tile_map_static": ([ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                ctypes.c_void_p]),
    "marble_last_error": ([]),
    "marble_version": ([]),
}


def lib():
    """Load libmarble.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name in ("marble_last_error", "marble_version") \
                else ctypes.c_int
        _lib = L
    return _lib


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != OK:
        raise MarbleError(st, lib().marble_last_error().decode())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class Plan:
    """A plan: tile map, token order, per-step lists and needed-KV index of one pack.

    sample/seg/noise: int32 CUDA tensors [N] in original token order (see marble.h)."""

    def __init__(self, sample, seg, noise, window: int, num_shards: int,
                 order: str = "contiguous", chunk_tokens: int = 0, stream=None,
                 range_cost: int = 0, key_intervals: bool = True, pos=None):
        import torch
        for t, nm in ((sample, "sample"), (seg, "seg"), (noise, "noise")):
            _need(t, torch.int32, nm, (sample.shape[0],))
        if pos is not None:
            _need(pos, torch.int32, "pos", (sample.shape[0],))
        self.n = int(sample.shape[0])
        self.num_shards = int(num_shards)
        self.window = int(window)
        self.order = order
        d = _PlanDesc(self.n, sample.data_ptr(), seg.data_ptr(), noise.data_ptr(),
                      int(window), int(num_shards), ORDERS[order], int(chunk_tokens),
                      int(range_cost), 0 if key_intervals else 1,
                      pos.data_ptr() if pos is not None else None)
        h = ctypes.c_void_p()
        _call("marble_plan", ctypes.byref(d), _stream(stream), ctypes.byref(h))
        self._h = h
        self.n_blocks = self.n // BLOCK
        self.blocks_per_shard = self.n_blocks // self.num_shards

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().marble_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self, stream=None) -> Dict[str, int]:
        s = _PlanStats()
        _call("marble_plan_stats", self._h, _stream(stream), ctypes.byref(s))
        return {name: int(getattr(s, name)) for name, _ in _PlanStats._fields_}

    def export(self, field: str, stream=None):
        """Copy a plan field into a new CUDA tensor."""
        import torch
        fid, dt = FIELDS[field]
        nbytes = ctypes.c_size_t()
        _call("marble_plan_field_bytes", self._h, fid, ctypes.byref(nbytes))
        dtype = getattr(torch, dt)
        elem = torch.tensor([], dtype=dtype).element_size()
        out = torch.empty(nbytes.value // elem, dtype=dtype, device="cuda")
        _call("marble_plan_export", self._h, fid, ctypes.c_void_p(out.data_ptr() if out.numel() else 0),
              nbytes.value, _stream(stream))
        return out

    def permute(self, src, inverse: bool = False, out=None, stream=None):
        """Gather rows into plan order (inverse=False) or scatter back (inverse=True)."""
        import torch
        if not src.is_cuda or not src.is_contiguous() or src.shape[0] != self.n:
            raise ValueError("src must be a contiguous CUDA tensor with N rows")
        out = torch.empty_like(src) if out is None else out
        row_bytes = src.numel() // self.n * src.element_size()
        _call("marble_permute", self._h, _ptr(src), _ptr(out), row_bytes, 1 if inverse else 0,
              _stream(stream))
        return out

    def permute_cast_bf16(self, src, inverse: bool = True, out=None, stream=None):
        """permute() of an fp32 tensor, written as bf16 (round to nearest even)."""
        import torch
        _need(src, torch.float32, "src")
        if src.shape[0] != self.n:
            raise ValueError("src must have N rows")
        out = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device) if out is None else out
        _need(out, torch.bfloat16, "out", src.shape)
        _call("marble_permute_cast_bf16", self._h, _ptr(src), _ptr(out), src.numel() // self.n,
              1 if inverse else 0, _stream(stream))
        return out

    def check(self, stream=None):
        _call("marble_check", self._h, _stream(stream))


class State:
    """fp32 online-softmax state (O_acc [N, hq, d], m [hq, N], l [hq, N]), plan order."""

    def __init__(self, n, hq, d, device="cuda"):
        import torch
        self.o_acc = torch.empty((n, hq, d), dtype=torch.float32, device=device)
        self.m = torch.empty((hq, n), dtype=torch.float32, device=device)
        self.l = torch.empty((hq, n), dtype=torch.float32, device=device)

    def _c(self):
        return _State(self.o_acc.data_ptr(), self.m.data_ptr(), self.l.data_ptr())


def _qkv(plan, q, k, v, scale):
    import torch
    n = plan.n
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q, k, v must be [N, heads, d]")
    hq, d = q.shape[1], q.shape[2]
    hkv = k.shape[1]
    _need(q, torch.bfloat16, "q", (n, hq, d))
    _need(k, torch.bfloat16, "k", (n, hkv, d))
    _need(v, torch.bfloat16, "v", (n, hkv, d))
    return _QKV(q.data_ptr(), k.data_ptr(), v.data_ptr(), hq, hkv, d, float(scale))


def _flags(first: bool, merge) -> int:
    if merge not in _MERGE:
        raise ValueError(f"merge must be one of {sorted(k for k in _MERGE if k)}")
    return (STEP_FIRST if first else 0) | _MERGE[merge]


def attn_step(plan: Plan, q, k, v, q_shard: int, kv_shard: int, state: State,
              first: bool = False, scale: float = 0.0, stream=None, merge: str = "carried"):
    """One forward ring step (marble_attn_step).  ``merge``: "carried" (the fp32 state
    carried across steps), "bf16" (the standard per-step merge of bf16 partials) or "fp32"
    (the same merge of fp32 partials)."""
    c = _qkv(plan, q, k, v, scale)
    st = state._c()
    _call("marble_attn_step", plan.handle, ctypes.byref(c), int(q_shard), int(kv_shard),
          ctypes.byref(st), _flags(first, merge), _stream(stream))


def attn_finalize(plan: Plan, state: State, o, lse, stream=None):
    import torch
    n, hq, d = state.o_acc.shape
    _need(o, torch.bfloat16, "o", (n, hq, d))
    _need(lse, torch.float32, "lse", (hq, n))
    st = state._c()
    _call("marble_attn_finalize", plan.handle, ctypes.byref(st), hq, d, _ptr(o), _ptr(lse),
          _stream(stream))


def attn_bwd_prep(plan: Plan, o, do, delta, stream=None):
    import torch
    n, hq, d = o.shape
    _need(o, torch.bfloat16, "o")
    _need(do, torch.bfloat16, "do", o.shape)
    _need(delta, torch.float32, "delta", (hq, n))
    _call("marble_attn_bwd_prep", plan.handle, _ptr(o), _ptr(do), hq, d, _ptr(delta),
          _stream(stream))


def attn_bwd(plan: Plan, q, k, v, do, lse, delta, q_shard: int, kv_shard: int, dq_acc, dk_acc,
             dv_acc, scale: float = 0.0, stream=None):
    """One backward ring step (marble_attn_bwd); accumulators are fp32 and caller-zeroed."""
    import torch
    c = _qkv(plan, q, k, v, scale)
    _need(do, torch.bfloat16, "do", q.shape)
    _need(lse, torch.float32, "lse", (q.shape[1], plan.n))
    _need(delta, torch.float32, "delta", (q.shape[1], plan.n))
    _need(dq_acc, torch.float32, "dq_acc", q.shape)
    _need(dk_acc, torch.float32, "dk_acc", k.shape)
    _need(dv_acc, torch.float32, "dv_acc", k.shape)
    _call("marble_attn_bwd", plan.handle, ctypes.byref(c), _ptr(do), _ptr(lse), _ptr(delta),
          int(q_shard), int(kv_shard), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), 0,
          _stream(stream))


def cast_bf16(src, dst, stream=None):
    import torch
    _need(src, torch.float32, "src")
    _need(dst, torch.bfloat16, "dst", src.shape)
    _call("marble_cast_bf16", _ptr(src), _ptr(dst), src.numel(), _stream(stream))


def set_wait_limit_ns(ns: int):
    _call("marble_set_wait_limit_ns", int(ns))


def release_memory():
    """Give the memory the library keeps for reuse (cached dS scratch of destroyed plans, the
    pool's unused blocks) back to the current device."""
    _call("marble_release_memory")


def set_side_streams(n: int):
    """Cap the side streams the step-list calls use (0: all launches on the caller's
    stream, in list order)."""
    _call("marble_set_side_streams", int(n))


def timing_enable(on: bool = True):
    """Per-kernel device timing of later attention calls (CUDA events on each kernel's stream)."""
    _call("marble_timing_enable", 1 if on else 0)


def timing_read() -> dict:
    """Summed device ms and launch counts per kernel since the previous read."""
    buf = (ctypes.c_double * 6)()
    _call("marble_timing_read", ctypes.cast(buf, ctypes.c_void_p))
    return {"fwd_ms": buf[0], "fwd_launches": int(buf[1]), "dq_ms": buf[2],
            "dq_launches": int(buf[3]), "dkdv_ms": buf[4], "dkdv_launches": int(buf[5])}


def debug_wait_timeout(plan: Plan, limit_ns: int, stream=None):
    _call("marble_debug_wait_timeout", plan.handle, int(limit_ns), _stream(stream))


TILE_MAP_STATIC_MAX_TOKENS = 2097152


def tile_map_static(sample, seg, noise, window: int, row_ptr, col, tag, stream=None):
    """Global tile map into caller-provided CUDA tensors without any allocation by the
    library (marble_tile_map_static): row_ptr int64[nb+1], col int32[cap], tag uint8[cap]."""
    import torch
    n = int(sample.shape[0])
    for t, nm in ((sample, "sample"), (seg, "seg"), (noise, "noise")):
        _need(t, torch.int32, nm, (n,))
    _need(row_ptr, torch.int64, "row_ptr", (n // BLOCK + 1,))
    _need(col, torch.int32, "col")
    _need(tag, torch.uint8, "tag", (col.numel(),))
    _call("marble_tile_map_static", n, _ptr(sample), _ptr(seg), _ptr(noise), int(window),
          _ptr(row_ptr), _ptr(col), _ptr(tag), col.numel(), _stream(stream))


def ring_schedule(num_shards: int, needed: bool = False):
    """The (q_shard, kv_shard, first) calls of one pass: r-major, kv shard (r - s) mod P at
    step s (MARBLE s03 ring pairing); with ``needed`` one call per q shard."""
    P = num_shards
    if needed:
        return [(r, KV_NEEDED, True) for r in range(P)]
    return [(r, (r - s) % P, s == 0) for r in range(P) for s in range(P)]


def attn_steps(plan: Plan, q, k, v, schedule, state: State, scale: float = 0.0, stream=None,
               merge: str = "carried"):
    """A list of forward ring steps [(q_shard, kv_shard, first), ...] in one C call."""
    c = _qkv(plan, q, k, v, scale)
    st = state._c()
    n = len(schedule)
    qs = (ctypes.c_int32 * n)(*[int(r) for r, _, _ in schedule])
    ks = (ctypes.c_int32 * n)(*[int(j) for _, j, _ in schedule])
    fl = (ctypes.c_uint32 * n)(*[_flags(f, merge) for _, _, f in schedule])
    _call("marble_attn_steps", plan.handle, ctypes.byref(c), n, qs, ks, fl, ctypes.byref(st),
          _stream(stream))


def attn_bwd_steps(plan: Plan, q, k, v, do, lse, delta, schedule, dq_acc, dk_acc, dv_acc,
                   scale: float = 0.0, stream=None):
    """A list of backward ring steps [(q_shard, kv_shard, _), ...] in one C call."""
    import torch
    c = _qkv(plan, q, k, v, scale)
    _need(do, torch.bfloat16, "do", q.shape)
    _need(lse, torch.float32, "lse", (q.shape[1], plan.n))
    _need(delta, torch.float32, "delta", (q.shape[1], plan.n))
    _need(dq_acc, torch.float32, "dq_acc", q.shape)
    _need(dk_acc, torch.float32, "dk_acc", k.shape)
    _need(dv_acc, torch.float32, "dv_acc", k.shape)
    n = len(schedule)
    qs = (ctypes.c_int32 * n)(*[int(r) for r, _, _ in schedule])
    ks = (ctypes.c_int32 * n)(*[int(j) for _, j, _ in schedule])
    _call("marble_attn_bwd_steps", plan.handle, ctypes.byref(c), _ptr(do), _ptr(lse),
          _ptr(delta), n, qs, ks, _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), _stream(stream))


def attn_fwd_fused(plan: Plan, q, k, v, state: State, scale: float = 0.0, stream=None):
    """Every forward ring step in one launch, the state on chip between steps
    (marble_attn_fwd_fused)."""
    c = _qkv(plan, q, k, v, scale)
    st = state._c()
    _call("marble_attn_fwd_fused", plan.handle, ctypes.byref(c), ctypes.byref(st),
          _stream(stream))


def attn_bwd_fused(plan: Plan, q, k, v, do, lse, delta, dq_acc, dk_acc, dv_acc,
                   scale: float = 0.0, stream=None):
    """Every backward ring step, one dK/dV launch per kv shard over its ring
    (marble_attn_bwd_fused); accumulators fp32 and caller-zeroed."""
    import torch
    c = _qkv(plan, q, k, v, scale)
    _need(do, torch.bfloat16, "do", q.shape)
    _need(lse, torch.float32, "lse", (q.shape[1], plan.n))
    _need(delta, torch.float32, "delta", (q.shape[1], plan.n))
    _need(dq_acc, torch.float32, "dq_acc", q.shape)
    _need(dk_acc, torch.float32, "dk_acc", k.shape)
    _need(dv_acc, torch.float32, "dv_acc", k.shape)
    _call("marble_attn_bwd_fused", plan.handle, ctypes.byref(c), _ptr(do), _ptr(lse),
          _ptr(delta), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), _stream(stream))


def forward(plan: Plan, q, k, v, state: State, o, lse, needed: bool = False, scale: float = 0.0,
            stream=None, merge: str = "carried", fused: bool = False):
    """All forward ring steps (r-major, keeping shard r's state hot in L2) + finalize;
    ``fused``: the whole ring in one launch (marble_attn_fwd_fused)."""
    if fused:
        if needed or merge not in (None, "carried"):
            raise ValueError("the fused ring carries the fp32 state over the ring steps only")
        attn_fwd_fused(plan, q, k, v, state, scale=scale, stream=stream)
    else:
        attn_steps(plan, q, k, v, ring_schedule(plan.num_shards, needed), state, scale=scale,
                   stream=stream, merge=merge)
    attn_finalize(plan, state, o, lse, stream=stream)


def backward(plan: Plan, q, k, v, o, do, lse, delta, dq_acc, dk_acc, dv_acc,
             needed: bool = False, scale: float = 0.0, stream=None, fused: bool = False):
    """bwd preprocessing + all backward ring steps (accumulators must be zeroed);
    ``fused``: one dK/dV launch per kv shard over its ring (marble_attn_bwd_fused)."""
    attn_bwd_prep(plan, o, do, delta, stream=stream)
    if fused:
        if needed:
            raise ValueError("the fused ring runs the ring steps, not the needed-block mode")
        attn_bwd_fused(plan, q, k, v, do, lse, delta, dq_acc, dk_acc, dv_acc, scale=scale,
                       stream=stream)
    else:
        attn_bwd_steps(plan, q, k, v, do, lse, delta, ring_schedule(plan.num_shards, needed),
                       dq_acc, dk_acc, dv_acc, scale=scale, stream=stream)


def layout_vision_groups(sample, seg):
    """The vision-group layout (marble_layout_vision_groups) of host int32 tracks: returns
    perm (new index -> index), an int32 numpy array."""
    import numpy as np
    s_ = np.ascontiguousarray(sample, dtype=np.int32)
    g_ = np.ascontiguousarray(seg, dtype=np.int32)
    if s_.shape != g_.shape or s_.ndim != 1:
        raise ValueError("sample and seg must be 1-D arrays of one length")
    perm = np.empty(len(s_), np.int32)
    _call("marble_layout_vision_groups", s_.ctypes.data, g_.ctypes.data, len(s_),
          perm.ctypes.data)
    return perm


def chunk_layout_search(block_pairs, num_shards: int, range_cost: int = 0):
    """The chunk-layout search (marble_chunk_layout_search) on a host int64 [nb, nb] matrix
    of work between blocks.  Returns (k, layout cost C, step cost, rank of every chunk)."""
    import numpy as np
    w = np.ascontiguousarray(block_pairs, dtype=np.int64)
    nb = w.shape[0]
    if w.shape != (nb, nb):
        raise ValueError("block_pairs must be square")
    rank = np.zeros(min(nb, 1024), np.int32)
    out = np.zeros(3, np.int64)
    _call("marble_chunk_layout_search", w.ctypes.data, nb, int(num_shards), int(range_cost),
          rank.ctypes.data, out.ctypes.data)
    k = int(out[0])
    return k, int(out[1]), int(out[2]), rank[:k * int(num_shards)].astype(np.int64)


def version() -> str:
    return lib().marble_version().decode()
