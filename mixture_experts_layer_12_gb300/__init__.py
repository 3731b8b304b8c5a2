"""GB300-native fused MoE layer forward: Python binding of libmoe.so.

The entry points mirror the C ABI of ``include/moe.h`` name for name and
only marshal arguments: torch tensors (device memory owned by the caller)
become raw pointers, the stream defaults to torch's current stream, and a
non-zero return code raises :class:`MoEError` with the library's message.
Every step of the layer runs in the library's CUDA kernels; there is no
other code path, and a missing library raises instead of falling back.

The method is the five-step MoE forward of the page "用Ascend C写一个MoE
融合算子", section "MoE的计算流程" (Routing, Gating, Dispatch, Expert,
Combine); ``include/moe.h`` gives each entry point's definition.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_DEVICE = 5
MOE_DEV_TIMEOUT = 0x1
MOE_DEV_BAD_ID = 0x2
MOE_WS_MIN_BYTES = 256

# Every symbol include/moe.h declares.
EXPORTS = ("moe_version", "moe_last_error_string", "moe_expert_capacity", "moe_workspace_size",
           "moe_route", "moe_dispatch", "moe_expert_ffn_combine", "moe_forward",
           "moe_get_device_status", "moe_selftest_wait_timeout", "moe_forward_profiled",
           "moe_expert_ffn_combine_noalloc", "moe_route_workspace_size", "moe_dispatch_rows",
           "moe_expert_ffn", "moe_combine", "moe_forward_plan", "moe_noalloc_device_status",
           "moe_route_plan")
MOE_NOALLOC_SCRATCH_BYTES = 32 << 20


class MoEError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[moe error {code}] {message}")
        self.code = code


MOE_GATE_TOPK_SOFTMAX = 0
MOE_GATE_SOFTMAX_TOPK = 1
MOE_GATE_SOFTMAX_TOPK_RENORM = 2


MOE_EXPERT_GELU = 0
MOE_EXPERT_SWIGLU = 1
_ACTS = {"gelu": MOE_EXPERT_GELU, "swiglu": MOE_EXPERT_SWIGLU}


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
                ("gating", ctypes.c_int32), ("expert_act", ctypes.c_int32)]


def make_shape(T: int, H: int, F: int, E: int, k: int, capacity_factor=None,
               gating: int = MOE_GATE_TOPK_SOFTMAX, act: str = "gelu") -> moe_shape:
    cf = -1.0 if capacity_factor is None else float(capacity_factor)
    return moe_shape(int(T), int(H), int(F), int(E), int(k), cf, int(gating), _ACTS[act])


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libmoe.so not found at {p}; run mixture_experts_layer_12_gb300/build.py "
                              "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(p)
        P, S = ctypes.c_void_p, ctypes.POINTER(moe_shape)
        sig = {
            "moe_version": ([], ctypes.c_int),
            "moe_last_error_string": ([], ctypes.c_char_p),
            "moe_expert_capacity": ([S], ctypes.c_int64),
            "moe_workspace_size": ([S], ctypes.c_size_t),
            "moe_route_workspace_size": ([S], ctypes.c_size_t),
            "moe_route": ([S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "moe_dispatch": ([S, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "moe_expert_ffn_combine": ([S, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "moe_forward": ([S, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "moe_get_device_status": ([P, P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
            "moe_noalloc_device_status": ([P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
            "moe_selftest_wait_timeout": ([P, ctypes.c_size_t, ctypes.c_uint64, P], ctypes.c_int),
            "moe_forward_profiled": ([S, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P],
                                     ctypes.c_int),
            "moe_expert_ffn_combine_noalloc": ([S, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "moe_dispatch_rows": ([S, P, P, P, P, P], ctypes.c_int),
            "moe_expert_ffn": ([S, ctypes.c_int32, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "moe_combine": ([S, P, P, P, P, P], ctypes.c_int),
            "moe_forward_plan": ([S, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
                                 ctypes.c_int),
            "moe_route_plan": ([S, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
                               ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int):
    if rc != MOE_OK:
        msg = load_library().moe_last_error_string().decode(errors="replace")
        raise MoEError(rc, msg)


def _current_cuda_index() -> int:
    return torch.cuda.current_device()


def check_tensor(t, dtype=None, name="tensor", min_numel: int = 0, device_index=None) -> None:
    """Host-side checks of one tensor argument, before anything is launched:
    dtype, contiguity, at least `min_numel` elements (the library indexes
    its buffers from the shape alone, so an undersized tensor would become
    out-of-bounds device accesses), and -- when it holds elements -- that it
    lives on CUDA device `device_index` (the current device, whose stream
    and built-in scratch the call uses)."""
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements; the shape needs at least {min_numel}")
    if t.numel() > 0:
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got device {t.device}")
        if device_index is not None and t.device.index != device_index:
            raise ValueError(f"{name} is on cuda:{t.device.index}, the current device is "
                             f"cuda:{device_index}")


def _ptr(t, dtype=None, name="tensor", min_numel: int = 0):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    dev = _current_cuda_index() if (t.numel() > 0 and t.device.type == "cuda") else None
    check_tensor(t, dtype, name, min_numel, dev)
    return ctypes.c_void_p(t.data_ptr())


def _req(shape, n_segments: int = 0) -> dict:
    """Minimum element counts of every tensor argument for `shape`."""
    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    f1 = 2 * F if shape.expert_act == MOE_EXPERT_SWIGLU else F
    tk = max(T, 0) * k
    return dict(x=T * H, w_router=H * E, b_router=E, ids=tk, weights=tk, counts=E, offsets=E + 1,
                perm=tk, slot=tk, w1=E * H * f1, w2=E * F * H, y=T * H, xp=tk * H, Y=tk * H,
                seg_offsets=n_segments + 1)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ------------------------------------------------------------ C ABI names --

def moe_version() -> int:
    return load_library().moe_version()


def moe_expert_capacity(shape: moe_shape) -> int:
    return int(load_library().moe_expert_capacity(ctypes.byref(shape)))


def moe_workspace_size(shape: moe_shape) -> int:
    n = int(load_library().moe_workspace_size(ctypes.byref(shape)))
    if n == 0:
        _check(MOE_ERR_UNSUPPORTED)
    return n


def moe_forward_plan(shape: moe_shape) -> tuple[bool, bool]:
    """(dispatch runs inside the router launch, combine runs inside the
    second expert GEMM) for this shape."""
    d, c = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().moe_forward_plan(ctypes.byref(shape), ctypes.byref(d), ctypes.byref(c)))
    return bool(d.value), bool(c.value)


def moe_route_plan(shape: moe_shape) -> tuple[int, int]:
    """(tokens per tile, K splits) of the one-launch tensor-core route on
    the current CUDA device, (0, 0) when the shape routes otherwise."""
    tm, sp = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().moe_route_plan(ctypes.byref(shape), ctypes.byref(tm), ctypes.byref(sp)))
    return int(tm.value), int(sp.value)


def moe_route_workspace_size(shape: moe_shape) -> int:
    n = int(load_library().moe_route_workspace_size(ctypes.byref(shape)))
    if n == 0:
        _check(MOE_ERR_UNSUPPORTED)
    return n


def _args(shape, *specs, n_segments: int = 0):
    """ctypes pointers of (tensor, dtype, name) argument specs, each checked
    against the element count the shape needs (see check_tensor)."""
    need = _req(shape, n_segments)
    return [_ptr(t, dt, name, need.get(name, 0)) for t, dt, name in specs]


_BF, _I32, _F32 = torch.bfloat16, torch.int32, torch.float32


def _ws(ws):
    return _ptr(ws, None, "ws"), ws.numel() * ws.element_size()


def moe_route(shape, x, w_router, b_router, ids, weights, counts, offsets, perm, slot, ws,
              stream=None):
    p = _args(shape, (x, _BF, "x"), (w_router, _BF, "w_router"), (b_router, _F32, "b_router"),
              (ids, _I32, "ids"), (weights, _F32, "weights"), (counts, _I32, "counts"),
              (offsets, _I32, "offsets"), (perm, _I32, "perm"), (slot, _I32, "slot"))
    _check(load_library().moe_route(ctypes.byref(shape), *p, *_ws(ws), _stream(stream)))


def moe_dispatch(shape, ids, counts, offsets, perm, slot, ws, stream=None):
    p = _args(shape, (ids, _I32, "ids"), (counts, _I32, "counts"), (offsets, _I32, "offsets"),
              (perm, _I32, "perm"), (slot, _I32, "slot"))
    _check(load_library().moe_dispatch(ctypes.byref(shape), *p, *_ws(ws), _stream(stream)))


def _ffn_combine_specs(x, w1, w2, weights, offsets, perm, slot, y):
    return ((x, _BF, "x"), (w1, _BF, "w1"), (w2, _BF, "w2"), (weights, _F32, "weights"),
            (offsets, _I32, "offsets"), (perm, _I32, "perm"), (slot, _I32, "slot"), (y, _BF, "y"))


def moe_expert_ffn_combine(shape, x, w1, w2, weights, offsets, perm, slot, y, ws, stream=None):
    p = _args(shape, *_ffn_combine_specs(x, w1, w2, weights, offsets, perm, slot, y))
    _check(load_library().moe_expert_ffn_combine(ctypes.byref(shape), *p, *_ws(ws),
                                                 _stream(stream)))


def moe_dispatch_rows(shape, x, perm, offsets, xp, stream=None):
    """xp[r] = x[perm[r] // k] for the kept rows, in dispatch order."""
    p = _args(shape, (x, _BF, "x"), (perm, _I32, "perm"), (offsets, _I32, "offsets"),
              (xp, _BF, "xp"))
    _check(load_library().moe_dispatch_rows(ctypes.byref(shape), *p, _stream(stream)))


def moe_expert_ffn(shape, n_segments, xp, w1, w2, seg_offsets, Y, ws, stream=None):
    """Expert FFN on rows grouped in segments; segment i uses expert i % E."""
    p = _args(shape, (xp, _BF, "xp"), (w1, _BF, "w1"), (w2, _BF, "w2"),
              (seg_offsets, _I32, "seg_offsets"), (Y, _BF, "Y"), n_segments=int(n_segments))
    _check(load_library().moe_expert_ffn(ctypes.byref(shape), int(n_segments), *p, *_ws(ws),
                                         _stream(stream)))


def moe_combine(shape, Y, weights, slot, y, stream=None):
    """y[t] = sum_j weights[t, j] * Y[slot[t, j]] over the kept slots."""
    p = _args(shape, (Y, _BF, "Y"), (weights, _F32, "weights"), (slot, _I32, "slot"),
              (y, _BF, "y"))
    _check(load_library().moe_combine(ctypes.byref(shape), *p, _stream(stream)))


def moe_expert_ffn_combine_noalloc(shape, x, w1, w2, weights, offsets, perm, slot, y, stream=None):
    """moe_expert_ffn_combine without a caller workspace: the library's
    built-in device scratch (MOE_NOALLOC_SCRATCH_BYTES) holds the
    intermediates, for callers that cannot allocate device memory.  Calls
    that overlap on the GPU share that scratch and must be serialised."""
    p = _args(shape, *_ffn_combine_specs(x, w1, w2, weights, offsets, perm, slot, y))
    _check(load_library().moe_expert_ffn_combine_noalloc(ctypes.byref(shape), *p,
                                                         _stream(stream)))


def _forward_specs(x, w_router, b_router, w1, w2, y, ids, weights, counts, offsets, perm, slot):
    return ((x, _BF, "x"), (w_router, _BF, "w_router"), (b_router, _F32, "b_router"),
            (w1, _BF, "w1"), (w2, _BF, "w2"), (y, _BF, "y"), (ids, _I32, "ids"),
            (weights, _F32, "weights"), (counts, _I32, "counts"), (offsets, _I32, "offsets"),
            (perm, _I32, "perm"), (slot, _I32, "slot"))


def moe_forward(shape, x, w_router, b_router, w1, w2, y, ids, weights, counts, offsets, perm,
                slot, ws, stream=None):
    p = _args(shape, *_forward_specs(x, w_router, b_router, w1, w2, y, ids, weights, counts,
                                     offsets, perm, slot))
    _check(load_library().moe_forward(ctypes.byref(shape), *p, *_ws(ws), _stream(stream)))


KERNEL_NAMES = ("router", "dispatch", "permute", "expert_gemm1", "expert_gemm2", "combine")


def moe_forward_profiled(shape, x, w_router, b_router, w1, w2, y, ids, weights, counts, offsets,
                         perm, slot, ws, events, stream=None):
    """moe_forward recording ``events`` (len(KERNEL_NAMES) + 1 torch.cuda.Event
    or None) at the kernel boundaries: before the router, then after each of
    KERNEL_NAMES."""
    n = len(KERNEL_NAMES) + 1
    if len(events) != n:
        raise ValueError(f"moe_forward_profiled takes {n} events, got {len(events)}")
    handles = (ctypes.c_void_p * n)()
    for i, ev in enumerate(events):
        if ev is not None:
            if not ev.cuda_event:
                ev.record()  # materialise the underlying cudaEvent_t
            handles[i] = ev.cuda_event
    p = _args(shape, *_forward_specs(x, w_router, b_router, w1, w2, y, ids, weights, counts,
                                     offsets, perm, slot))
    _check(load_library().moe_forward_profiled(ctypes.byref(shape), *p, *_ws(ws),
                                               _stream(stream), handles))


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word.
    Raises MoEError if a status bit is set."""
    v = ctypes.c_int32(0)
    rc = load_library().moe_get_device_status(_ptr(ws, None, "ws"), _stream(stream), ctypes.byref(v))
    if rc not in (MOE_OK,):
        raise MoEError(rc, load_library().moe_last_error_string().decode(errors="replace"))
    return v.value


def moe_noalloc_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the status word of
    moe_expert_ffn_combine_noalloc's built-in scratch on the current device.
    Raises MoEError if a status bit is set."""
    v = ctypes.c_int32(0)
    rc = load_library().moe_noalloc_device_status(_stream(stream), ctypes.byref(v))
    if rc != MOE_OK:
        raise MoEError(rc, load_library().moe_last_error_string().decode(errors="replace"))
    return v.value


def moe_selftest_wait_timeout(ws, limit_ns: int, stream=None):
    _check(load_library().moe_selftest_wait_timeout(
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), int(limit_ns), _stream(stream)))


# --------------------------------------------------------------- helpers --

@dataclass
class RoutingBuffers:
    ids: torch.Tensor
    weights: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    slot: torch.Tensor


def alloc_routing(T: int, E: int, k: int, device) -> RoutingBuffers:
    i32 = dict(dtype=torch.int32, device=device)
    return RoutingBuffers(ids=torch.empty(T, k, **i32),
                          weights=torch.empty(T, k, dtype=torch.float32, device=device),
                          counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                          perm=torch.empty(max(T * k, 1), **i32), slot=torch.empty(T, k, **i32))


def alloc_workspace(shape: moe_shape, device) -> torch.Tensor:
    """Workspace for moe_forward / moe_expert_ffn_combine (and all others)."""
    n = max(moe_workspace_size(shape), MOE_WS_MIN_BYTES)
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def alloc_route_workspace(shape: moe_shape, device) -> torch.Tensor:
    """Workspace for moe_route / moe_dispatch."""
    n = max(moe_route_workspace_size(shape), MOE_WS_MIN_BYTES)
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


class MoELayer:
    """Holds a layer's weights (device tensors) and reusable buffers; calling
    it runs moe_forward on the current stream."""

    def __init__(self, w_router, w1, w2, k: int, bias=None, capacity_factor=None,
                 gating: int = MOE_GATE_TOPK_SOFTMAX, act: str = "gelu"):
        """act "gelu": w1 [E, H, F]; "swiglu": w1 [E, H, 2F] = [gate | up]."""
        self.w_router, self.w1, self.w2, self.bias = w_router, w1, w2, bias
        self.E, self.H, self.F = w2.shape[0], w2.shape[2], w2.shape[1]
        self.act = act
        self.k = int(k)
        self.capacity_factor = capacity_factor
        self.gating = int(gating)
        self._T = None

    def _ensure(self, T: int, device):
        if self._T == T:
            return
        self.shape = make_shape(T, self.H, self.F, self.E, self.k, self.capacity_factor,
                                self.gating, self.act)
        self.ws = alloc_workspace(self.shape, device)
        self.routing = alloc_routing(T, self.E, self.k, device)
        self.y = torch.empty(T, self.H, dtype=torch.bfloat16, device=device)
        self._T = T

    def __call__(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        self._ensure(x.shape[0], x.device)
        r = self.routing
        moe_forward(self.shape, x, self.w_router, self.bias, self.w1, self.w2, self.y, r.ids,
                    r.weights, r.counts, r.offsets, r.perm, r.slot, self.ws, stream)
        return self.y


def capacity(T: int, E: int, k: int, capacity_factor) -> int:
    """The library's expert capacity (-1 = unlimited), computed by the library."""
    return moe_expert_capacity(make_shape(T, 8, 8, E, k, capacity_factor))


def load_cv(counts) -> float:
    """Coefficient of variation (std / mean) of the per-expert kept counts:
    the load-balance diagnostic of the article's section 4.3 (its auxiliary
    loss is 0.01 * cv(experts_load)).  Host-side arithmetic on an output."""
    c = counts.detach().double().cpu()
    m = c.mean().item()
    return float(c.std(unbiased=False).item() / m) if m > 0 else 0.0


def roofline_flops(N_rows: int, H: int, F: int) -> float:
    """Algorithmic FLOPs of the two expert GEMMs for N_rows kept rows."""
    return 4.0 * N_rows * H * F


__all__ = [n for n in EXPORTS] + ["MoEError", "moe_shape", "make_shape", "load_library",
                                   "alloc_routing", "alloc_workspace", "alloc_route_workspace",
                                   "MoELayer", "RoutingBuffers",
                                   "capacity", "roofline_flops", "load_cv",
                                   "MOE_GATE_TOPK_SOFTMAX", "MOE_GATE_SOFTMAX_TOPK",
                                   "MOE_GATE_SOFTMAX_TOPK_RENORM", "MOE_EXPERT_GELU",
                                   "MOE_EXPERT_SWIGLU"]
