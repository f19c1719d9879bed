"""Python binding of libmoe_gb300 (include/moe.h): one MoE-layer forward on a
GB300 GPU -- router top-k/softmax, dispatch, persistent tcgen05 grouped SwiGLU
GEMM, gate-weighted combine -- as hand-written sm_103a CUDA kernels.

This module only marshals arguments: it checks torch tensors' dtype, device,
contiguity and size, passes their device pointers and the current CUDA stream
through ctypes, and turns a non-OK status into an exception. Every step of the
computation runs in the library's kernels; there is no CPU or PyTorch
fallback. Build the library first (``python -c "import __graft_entry__ as g;
g.build()"``); calling into it when it is missing raises ``MoEError``.

Function names follow the C ABI: route, dispatch, expert_ffn, combine,
layer_forward (moe_ prefix dropped).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from .build import LIB_PATH

__all__ = [
    "MoEError", "Shape", "Tuning", "library", "workspace_bytes", "workspace_region", "alloc_workspace",
    "ws_view", "route", "route_scratch_bytes", "alloc_route_scratch", "route_filtered", "dispatch", "expert_ffn", "combine", "layer_forward", "last_device_status",
    "SCHEDULE_INTERLEAVED", "SCHEDULE_EXPERT_WAVE", "ORIENT_DEFAULT", "ORIENT_TOKENS_M", "ORIENT_TOKENS_N", "WS",
    "ROUTER_DEFAULT", "ROUTER_DIRECT", "ROUTER_FILTER_VERIFY",
]

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = \
    range(6)
SCHEDULE_INTERLEAVED, SCHEDULE_EXPERT_WAVE = 0, 1
ORIENT_DEFAULT, ORIENT_TOKENS_M, ORIENT_TOKENS_N = 0, 1, 2
ROUTER_DEFAULT, ROUTER_DIRECT, ROUTER_FILTER_VERIFY = 0, 1, 2


class WS:
    """Workspace region ids (MOE_WS_*)."""
    STATUS, TOPK_IDX, TOPK_GATE, COUNTS, OFFSETS, ROW_OF_SLOT, SLOT_OF_ROW, X_PERM, H, Y_PERM, \
        CHUNK_BASE, L1_DONE, L2_FLAGS = range(13)


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)} (status {status})")


class _CShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int),
                ("top_k", ctypes.c_int), ("ffn", ctypes.c_int), ("num_segments", ctypes.c_int)]


class _CTuning(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int), ("lead_rows", ctypes.c_int), ("num_ctas", ctypes.c_int),
                ("l2_block_n", ctypes.c_int), ("group_rows", ctypes.c_int), ("cta_group", ctypes.c_int),
                ("wait_limit_us", ctypes.c_int), ("unmet_dependency", ctypes.c_int),
                ("trace", ctypes.c_void_p), ("tile_trace", ctypes.c_void_p),
                ("tile_trace_cap", ctypes.c_int), ("orientation", ctypes.c_int),
                ("h_ring_rows", ctypes.c_int), ("fused_combine", ctypes.c_int), ("row_order", ctypes.c_int),
                ("router", ctypes.c_int)]


@dataclass(frozen=True)
class Shape:
    T: int
    d: int
    E: int
    top_k: int
    ffn: int
    num_segments: int = 1

    @property
    def R(self) -> int:
        return self.T * self.top_k

    def c(self) -> _CShape:
        return _CShape(self.T, self.d, self.E, self.top_k, self.ffn, self.num_segments)


TRACE_WORDS = 16  # per-CTA uint64 counters written when Tuning.trace is given
TILE_TRACE_WORDS = 8  # per-tile record words written when Tuning.tile_trace is given
TILE_TRACE_FIELDS = ("tile", "prod_start", "prod_dep_wait", "mma_start", "mma_last_issue",
                     "mma_stage_wait", "epi_start", "epi_end")
TRACE_FIELDS = ("prod_wait_empty", "prod_wait_rows", "prod_cycles", "mma_wait_full", "mma_wait_tmem",
                "mma_cycles", "epi_wait_full", "epi_work", "epi_wait_stores", "epi_cycles", "l1_tiles",
                "l2_tiles", "t_start_ns", "t_end_ns", "unused14", "unused15")


@dataclass(frozen=True)
class Tuning:
    schedule: int = SCHEDULE_INTERLEAVED
    lead_rows: int = 0
    num_ctas: int = 0
    l2_block_n: int = 0
    group_rows: int = 0
    cta_group: int = 0
    wait_limit_us: int = 0
    unmet_dependency: int = 0
    trace: object = None  # optional torch int64 CUDA tensor of >= num_ctas * TRACE_WORDS entries
    tile_trace: object = None  # optional torch int64 CUDA tensor, num_ctas * cap * TILE_TRACE_WORDS
    tile_trace_cap: int = 0
    orientation: int = ORIENT_DEFAULT  # which MMA operand holds the tokens (ORIENT_*)
    h_ring_rows: int = 0  # h as a ring of this many scheduler rows (0 = all rows)
    fused_combine: int = 0  # layer only: combine inside the grouped GEMM (consumer warps)
    row_order: int = 0  # scheduler rows: 0 default, 1 expert order, 2 mixed (single-row experts spread out)
    router: int = ROUTER_DEFAULT  # layer routing: ROUTER_DIRECT or ROUTER_FILTER_VERIFY (same bits)

    def c(self) -> _CTuning:
        tr = None if self.trace is None else _ptr(self.trace, torch.int64, None, "trace")
        tt = None if self.tile_trace is None else _ptr(self.tile_trace, torch.int64, None, "tile_trace")
        return _CTuning(self.schedule, self.lead_rows, self.num_ctas, self.l2_block_n, self.group_rows,
                        self.cta_group, self.wait_limit_us, self.unmet_dependency, tr, tt,
                        self.tile_trace_cap, self.orientation, self.h_ring_rows, self.fused_combine,
                        self.row_order, self.router)


_lib = None


def library():
    """The loaded libmoe_gb300 (ctypes). Raises MoEError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError(MOE_ERR_CUDA, f"libmoe_gb300 is not built ({LIB_PATH} missing); "
                                         "run grouped_gemm_softmax_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, S, sz = ctypes.c_void_p, ctypes.POINTER(_CShape), ctypes.c_size_t
        TU = ctypes.POINTER(_CTuning)
        sig = {
            "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "moe_workspace_bytes": ([S], sz),
            "moe_workspace_region": ([S, ctypes.c_int, ctypes.POINTER(sz), ctypes.POINTER(sz)],
                                     ctypes.c_int),
            "moe_workspace_bytes_tuned": ([S, TU], sz),
            "moe_workspace_region_tuned": ([S, TU, ctypes.c_int, ctypes.POINTER(sz), ctypes.POINTER(sz)],
                                           ctypes.c_int),
            "moe_route": ([S, P, P, P, P, P, P], ctypes.c_int),
            "moe_route_scratch_bytes": ([S], sz),
            "moe_route_filtered": ([S, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_dispatch": ([S, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_expert_ffn": ([S, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_expert_ffn_tuned": ([S, TU, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_combine": ([S, P, P, P, P, P], ctypes.c_int),
            "moe_layer_forward": ([S, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_layer_forward_tuned": ([S, TU, P, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "moe_layer_forward_ex": ([S, TU, P, P, P, P, P, P, P, P, sz, P, P], ctypes.c_int),
            "moe_layer_kernel_launches": ([S, TU], ctypes.c_int),
            "moe_last_device_status": ([P, P], ctypes.c_int),
            "moe_last_device_detail": ([ctypes.POINTER(ctypes.c_uint32)] * 3, None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _status_string(st: int) -> str:
    try:
        return library().moe_status_string(st).decode()
    except MoEError:
        return "status %d" % st


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoEError(st, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype, numel=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return ctypes.c_void_p(t.data_ptr())


def workspace_bytes(shape: Shape, tuning: Tuning | None = None) -> int:
    if tuning is None:
        return int(library().moe_workspace_bytes(ctypes.byref(shape.c())))
    return int(library().moe_workspace_bytes_tuned(ctypes.byref(shape.c()), ctypes.byref(tuning.c())))


def workspace_region(shape: Shape, region: int, tuning: Tuning | None = None):
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    if tuning is None:
        _check(library().moe_workspace_region(ctypes.byref(shape.c()), region, ctypes.byref(off),
                                              ctypes.byref(nb)), "moe_workspace_region")
    else:
        _check(library().moe_workspace_region_tuned(ctypes.byref(shape.c()), ctypes.byref(tuning.c()),
                                                    region, ctypes.byref(off), ctypes.byref(nb)),
               "moe_workspace_region_tuned")
    return off.value, nb.value


def alloc_workspace(shape: Shape, device="cuda", tuning: Tuning | None = None) -> torch.Tensor:
    """Device workspace for one shape (and tuning: an h ring shrinks it)."""
    nb = workspace_bytes(shape, tuning)
    if nb == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_bytes")
    ws = torch.empty(nb, dtype=torch.uint8, device=device)
    ws[:16].zero_()  # device status word
    return ws


def layer_kernel_launches(shape: Shape, tuning: Tuning | None = None) -> int:
    """How many kernels one layer_forward call launches for this shape and tuning."""
    t = ctypes.byref(tuning.c()) if tuning is not None else None
    return int(library().moe_layer_kernel_launches(ctypes.byref(shape.c()), t))


def tile_trace_capacity(shape: Shape, num_ctas: int) -> int:
    """Per-CTA record count for Tuning.tile_trace that holds every tile a CTA can
    run: the tiles of the smallest (128-row) scheduler rows spread over the
    CTAs, plus 64 for the uneven spread of dynamically claimed tiles."""
    rows = (shape.T * shape.top_k + 127) // 128 + shape.E
    return rows * ((shape.ffn + shape.d) // 64) // max(num_ctas, 1) + 64


def ws_view(ws: torch.Tensor, shape: Shape, region: int, dtype, dims) -> torch.Tensor:
    """A typed view of one workspace region (no copy)."""
    off, nb = workspace_region(shape, region)
    esz = torch.empty((), dtype=dtype).element_size()
    n = 1
    for x in dims:
        n *= x
    if n * esz > nb:
        raise ValueError("view larger than the region")
    return ws[off:off + n * esz].view(dtype).view(*dims)


def route(shape: Shape, x, w_router, expert_bias, topk_idx, topk_gate, stream=None):
    T, d, E, k = shape.T, shape.d, shape.E, shape.top_k
    _check(library().moe_route(
        ctypes.byref(shape.c()), _ptr(x, torch.bfloat16, T * d, "x"),
        _ptr(w_router, torch.bfloat16, E * d, "w_router"),
        _ptr(expert_bias, torch.float32, E, "expert_bias", optional=True),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"), _ptr(topk_gate, torch.float32, T * k, "topk_gate"),
        _stream(stream)), "moe_route")


def route_scratch_bytes(shape: Shape) -> int:
    return int(library().moe_route_scratch_bytes(ctypes.byref(shape.c())))


def alloc_route_scratch(shape: Shape, device="cuda") -> torch.Tensor:
    """Zeroed device scratch for route_filtered (its status word starts clear)."""
    nb = route_scratch_bytes(shape)
    if nb == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "invalid shape")
    return torch.zeros(nb, dtype=torch.uint8, device=device)


def route_filtered(shape: Shape, x, w_router, expert_bias, topk_idx, topk_gate, scratch, stream=None):
    """route by filter then verify: the same bits in four launches (see moe.h)."""
    T, d, E, k = shape.T, shape.d, shape.E, shape.top_k
    _check(library().moe_route_filtered(
        ctypes.byref(shape.c()), _ptr(x, torch.bfloat16, T * d, "x"),
        _ptr(w_router, torch.bfloat16, E * d, "w_router"),
        _ptr(expert_bias, torch.float32, E, "expert_bias", optional=True),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"), _ptr(topk_gate, torch.float32, T * k, "topk_gate"),
        _ptr(scratch, torch.uint8, None, "scratch"), scratch.numel(), _stream(stream)), "moe_route_filtered")


def dispatch(shape: Shape, x, topk_idx, expert_counts, expert_offsets, row_of_slot, slot_of_row, x_perm,
             ws, stream=None):
    T, d, E, R = shape.T, shape.d, shape.E, shape.R
    _check(library().moe_dispatch(
        ctypes.byref(shape.c()), _ptr(x, torch.bfloat16, T * d, "x"),
        _ptr(topk_idx, torch.int32, R, "topk_idx"), _ptr(expert_counts, torch.int32, E, "expert_counts"),
        _ptr(expert_offsets, torch.int32, E + 1, "expert_offsets"),
        _ptr(row_of_slot, torch.int32, R, "row_of_slot"), _ptr(slot_of_row, torch.int32, R, "slot_of_row"),
        _ptr(x_perm, torch.bfloat16, R * d, "x_perm"), _ptr(ws, torch.uint8, None, "ws"), ws.numel(),
        _stream(stream)), "moe_dispatch")


def expert_ffn(shape: Shape, x_perm, expert_offsets, w1, w3, w2, y_perm, ws, stream=None,
               tuning: Tuning | None = None):
    R, d, E, F = shape.R, shape.d, shape.E, shape.ffn
    args = (_ptr(x_perm, torch.bfloat16, R * d, "x_perm"),
            _ptr(expert_offsets, torch.int32, E + 1, "expert_offsets"),
            _ptr(w1, torch.bfloat16, E * F * d, "W1"), _ptr(w3, torch.bfloat16, E * F * d, "W3"),
            _ptr(w2, torch.bfloat16, E * d * F, "W2"), _ptr(y_perm, torch.bfloat16, R * d, "y_perm"),
            _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream))
    if tuning is None:
        st = library().moe_expert_ffn(ctypes.byref(shape.c()), *args)
    else:
        st = library().moe_expert_ffn_tuned(ctypes.byref(shape.c()), ctypes.byref(tuning.c()), *args)
    _check(st, "moe_expert_ffn")


def _segments(shape: Shape, out_segments):
    if isinstance(out_segments, torch.Tensor):
        out_segments = [out_segments]
    if len(out_segments) != shape.num_segments:
        raise ValueError(f"expected {shape.num_segments} output segments")
    rows = shape.T // shape.num_segments
    arr = (ctypes.c_void_p * len(out_segments))()
    for i, s in enumerate(out_segments):
        arr[i] = _ptr(s, torch.bfloat16, rows * shape.d, f"out_segments[{i}]").value
    return arr


def combine(shape: Shape, y_perm, topk_gate, row_of_slot, out_segments, stream=None):
    R, d = shape.R, shape.d
    segs = _segments(shape, out_segments)
    _check(library().moe_combine(
        ctypes.byref(shape.c()), _ptr(y_perm, torch.bfloat16, R * d, "y_perm"),
        _ptr(topk_gate, torch.float32, R, "topk_gate"), _ptr(row_of_slot, torch.int32, R, "row_of_slot"),
        ctypes.cast(segs, ctypes.c_void_p), _stream(stream)), "moe_combine")


def layer_forward(shape: Shape, x, w_router, expert_bias, w1, w3, w2, out_segments, ws, stream=None,
                  tuning: Tuning | None = None, stage_events=None):
    """The whole layer. stage_events: optional 5 recorded torch.cuda.Event objects, re-recorded
    by the library before routing and after routing, dispatch, the grouped GEMM and combine."""
    T, d, E, F = shape.T, shape.d, shape.E, shape.ffn
    segs = _segments(shape, out_segments)
    args = (_ptr(x, torch.bfloat16, T * d, "x"), _ptr(w_router, torch.bfloat16, E * d, "w_router"),
            _ptr(expert_bias, torch.float32, E, "expert_bias", optional=True),
            _ptr(w1, torch.bfloat16, E * F * d, "W1"), _ptr(w3, torch.bfloat16, E * F * d, "W3"),
            _ptr(w2, torch.bfloat16, E * d * F, "W2"), ctypes.cast(segs, ctypes.c_void_p),
            _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream))
    if stage_events is not None:
        if len(stage_events) != 5 or any(int(e.cuda_event) == 0 for e in stage_events):
            raise ValueError("stage_events: five torch.cuda.Event objects, each recorded once")
        evs = (ctypes.c_void_p * 5)(*[int(e.cuda_event) for e in stage_events])
        tu = None if tuning is None else ctypes.byref(tuning.c())
        st = library().moe_layer_forward_ex(ctypes.byref(shape.c()), tu, *args,
                                            ctypes.cast(evs, ctypes.c_void_p))
    elif tuning is None:
        st = library().moe_layer_forward(ctypes.byref(shape.c()), *args)
    else:
        st = library().moe_layer_forward_tuned(ctypes.byref(shape.c()), ctypes.byref(tuning.c()), *args)
    _check(st, "moe_layer_forward")


def last_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status in ws."""
    return int(library().moe_last_device_status(_ptr(ws, torch.uint8, None, "ws"), _stream(stream)))


def last_device_detail():
    """(where, block, detail) of the last failure last_device_status read on this thread."""
    w, b, d = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_uint32()
    library().moe_last_device_detail(ctypes.byref(w), ctypes.byref(b), ctypes.byref(d))
    return w.value, b.value, d.value
