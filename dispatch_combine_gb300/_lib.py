"""ctypes binding of libmoe.so (the C ABI declared in include/moe.h).

Argument marshalling only: every step of the MoE path runs in the CUDA
kernels of libmoe.so.  There is no CPU or PyTorch fallback; if the library is
missing or a call fails, an exception is raised.

Tensors are passed by ``data_ptr()``; the stream is the caller's current
PyTorch CUDA stream unless one is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_SCORE_SIGMOID_BIAS = 0
MOE_SCORE_SOFTMAX = 1
MOE_LAYOUT_CONTIGUOUS = 0
MOE_LAYOUT_MASKED = 1

STATUS_NAMES = {
    0: "MOE_OK",
    1: "MOE_ERR_INVALID_ARG",
    2: "MOE_ERR_UNSUPPORTED",
    3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA",
    5: "MOE_ERR_TIMEOUT",
    6: "MOE_ERR_OVERFLOW",
}

# Every function the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t


class MoeShape(ctypes.Structure):
    """Mirror of moe_shape_t."""
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("G", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("score", ctypes.c_int32), ("bias_scale", ctypes.c_float)]


_PS = ctypes.POINTER(MoeShape)
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_workspace_size": (_I32, [_PS, ctypes.POINTER(_SZ)]),
    "moe_expert_ffn_workspace_size": (_I32, [_PS, _I32, _I32, ctypes.POINTER(_SZ)]),
    "moe_workspace_init": (_I32, [_P, _SZ, _P]),
    "moe_get_device_status": (_I32, [_P, _SZ, _P, ctypes.POINTER(_I32)]),
    "moe_route": (_I32, [_PS, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_from_logits": (_I32, [_PS, _P, _P, _P, _P, _P]),
    "moe_group_topk": (_I32, [_PS, _P, _P, _P]),
    "moe_dispatch": (_I32, [_PS, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_noalloc": (_I32, [_PS, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_replicated_workspace_size": (_I32, [_PS, _I32, ctypes.POINTER(_SZ)]),
    "moe_dispatch_replicated": (_I32, [_PS, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_capacity": (_I32, [_I32, _I32, _I32, ctypes.c_double]),
    "moe_eplb_plan": (_I32, [_P, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_quantize_fp8_rows": (_I32, [_P, ctypes.c_int64, _I32, _P, _P, _P]),
    "moe_expert_ffn_fp8_workspace_size": (_I32, [_PS, _I32, _I32, ctypes.POINTER(_SZ)]),
    "moe_expert_ffn_fp8": (_I32, [_PS, _I32, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _SZ,
                                  _P]),
    "moe_layer_fp8_workspace_size": (_I32, [_PS, ctypes.POINTER(_SZ)]),
    "moe_layer_fp8": (_I32, [_PS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_fp8_blocks": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P]),
    "moe_dispatch_capacity": (_I32, [_PS, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                     _SZ, _P]),
    "moe_layer_capacity_workspace_size": (_I32, [_PS, _I32, ctypes.POINTER(_SZ)]),
    "moe_layer_capacity": (_I32, [_PS, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                  _P]),
    "moe_expert_ffn": (_I32, [_PS, _I32, _P, _P, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_gate_up": (_I32, [_PS, _I32, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "moe_expert_down": (_I32, [_PS, _I32, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I32, [_PS, _P, _P, _P, _P, _P]),
    "moe_layer": (_I32, [_PS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_layer_launch_count": (_I32, [_PS]),
    "moe_layer_yperm_row_bytes": (ctypes.c_int64, [_PS]),
    "moe_route_refined_count": (_I32, [_PS, _P, _SZ, _P, _P]),
    "moe_router_prep_size": (_I32, [_PS, ctypes.POINTER(_SZ)]),
    "moe_router_prepare": (_I32, [_PS, _P, _P, _SZ, _P]),
    "moe_router_release": (_I32, [_P]),
    "moe_selftest_wait_timeout": (_I32, [_P, _SZ, _U64, _P]),
}

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


def lib():
    """Load libmoe.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m dispatch_combine_gb300.build` (the MoE path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def _check(name: str, st: int):
    if st != 0:
        raise MoEError(name, st)


def shape_struct(T, d, E, G, topk_group, k, inter, score, bias_scale=0.15) -> MoeShape:
    return MoeShape(int(T), int(d), int(E), int(G), int(topk_group), int(k), int(inter),
                    int(score), float(bias_scale))


def as_shape(s) -> MoeShape:
    """Accept a MoeShape, a dict or an object with the shape's attributes."""
    if isinstance(s, MoeShape):
        return s
    if isinstance(s, dict):
        return shape_struct(s["T"], s["d"], s["E"], s["G"], s["topk_group"], s["k"],
                            s["inter"], s["score"], s.get("bias_scale", 0.15))
    return shape_struct(s.T, s.d, s.E, s.G, s.topk_group, s.k, s.inter, s.score,
                        getattr(s, "bias_scale", 0.15))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _expect(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------------------
# workspace
# --------------------------------------------------------------------------

class Workspace:
    """Caller-owned device workspace (a uint8 tensor, 256-byte aligned)."""

    def __init__(self, nbytes: int, device=None, stream=None):
        device = torch.device(device if device is not None else "cuda")
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        self.offset = (-base) % 256
        self.ptr = base + self.offset
        _check("moe_workspace_init",
               lib().moe_workspace_init(ctypes.c_void_p(self.ptr), self.nbytes,
                                        _stream(stream)))

    @property
    def c_ptr(self):
        return ctypes.c_void_p(self.ptr)


def moe_workspace_size(shape) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(as_shape(shape)),
                                                          ctypes.byref(out)))
    return out.value


def moe_expert_ffn_workspace_size(shape, layout: int, M_max: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_expert_ffn_workspace_size",
           lib().moe_expert_ffn_workspace_size(ctypes.byref(as_shape(shape)), int(layout),
                                               int(M_max), ctypes.byref(out)))
    return out.value


def moe_get_device_status(ws: Workspace, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check("moe_get_device_status",
           lib().moe_get_device_status(ws.c_ptr, ws.nbytes, _stream(stream),
                                       ctypes.byref(st)))
    return st.value


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_layer_launch_count(shape) -> int:
    return int(lib().moe_layer_launch_count(ctypes.byref(as_shape(shape))))


def moe_layer_yperm_row_bytes(shape) -> int:
    """Bytes per routed row of the layer's down-GEMM output as the combine
    reads it (4*d fp32, or 2*d + d/32 in the compact form)."""
    return int(lib().moe_layer_yperm_row_bytes(ctypes.byref(as_shape(shape))))


def moe_route_refined_count(shape, ws: Workspace, stream=None) -> int:
    """(token, expert) pairs whose fixed-order logit the last screened
    routing in ws computed (-1: the shape is not screened).  Synchronises the
    stream."""
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    _check("moe_route_refined_count",
           lib().moe_route_refined_count(ctypes.byref(as_shape(shape)), ws.c_ptr, ws.nbytes,
                                         _ptr(out), _stream(stream)))
    return int(out.item())


def moe_router_prep_size(shape) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_router_prep_size",
           lib().moe_router_prep_size(ctypes.byref(as_shape(shape)), ctypes.byref(out)))
    return out.value


class RouterPrep:
    """A prepared copy of a router weight (see moe_router_prepare in moe.h).
    Holds its buffer and the weight while recorded; release() (or leaving a
    ``with`` block) drops the record."""

    def __init__(self, shape, w_r, stream=None):
        n = moe_router_prep_size(shape)
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=w_r.device)
        self.ptr = self.buf.data_ptr() + (-self.buf.data_ptr()) % 256
        self.w_r = w_r
        _check("moe_router_prepare",
               lib().moe_router_prepare(ctypes.byref(as_shape(shape)), _ptr(w_r),
                                        ctypes.c_void_p(self.ptr), n, _stream(stream)))

    def release(self):
        if self.w_r is not None:
            _check("moe_router_release", lib().moe_router_release(_ptr(self.w_r)))
            self.w_r = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.release()


def moe_router_prepare(shape, w_r, stream=None) -> RouterPrep:
    return RouterPrep(shape, w_r, stream)


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def moe_route(shape, x, w_r, bias, ws: Workspace, topk_ids=None, topk_w=None,
              logits=None, want_logits=False, stream=None):
    s = as_shape(shape)
    dev = x.device
    if topk_ids is None:
        topk_ids = torch.empty((s.T, s.k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((s.T, s.k), dtype=torch.float32, device=dev)
    if logits is None and want_logits:
        logits = torch.empty((s.T, s.E), dtype=torch.float32, device=dev)
    _expect(x, torch.bfloat16, (s.T, s.d), "x")
    _expect(w_r, torch.bfloat16, (s.d, s.E), "w_r")
    _check("moe_route", lib().moe_route(ctypes.byref(s), _ptr(x), _ptr(w_r), _ptr(bias),
                                        _ptr(topk_ids), _ptr(topk_w), _ptr(logits),
                                        ws.c_ptr, ws.nbytes, _stream(stream)))
    return topk_ids, topk_w, logits


def moe_route_from_logits(shape, logits, bias, topk_ids=None, topk_w=None, stream=None):
    s = as_shape(shape)
    dev = logits.device
    _expect(logits, torch.float32, (s.T, s.E), "logits")
    if topk_ids is None:
        topk_ids = torch.empty((s.T, s.k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((s.T, s.k), dtype=torch.float32, device=dev)
    _check("moe_route_from_logits",
           lib().moe_route_from_logits(ctypes.byref(s), _ptr(logits), _ptr(bias),
                                       _ptr(topk_ids), _ptr(topk_w), _stream(stream)))
    return topk_ids, topk_w


def moe_group_topk(shape, scores, topk_ids=None, stream=None):
    s = as_shape(shape)
    _expect(scores, torch.float32, (s.T, s.E), "scores")
    if topk_ids is None:
        topk_ids = torch.empty((s.T, s.k), dtype=torch.int32, device=scores.device)
    _check("moe_group_topk", lib().moe_group_topk(ctypes.byref(s), _ptr(scores),
                                                  _ptr(topk_ids), _stream(stream)))
    return topk_ids


def moe_dispatch(shape, topk_ids, x, ws: Workspace, stream=None, x_perm_out=None):
    """Returns (counts [E], offsets [E+1], src_token [T*k], dest [T*k], x_perm);
    x_perm is written into x_perm_out when it is given."""
    s = as_shape(shape)
    dev = topk_ids.device
    n = s.T * s.k
    _expect(topk_ids, torch.int32, (s.T, s.k), "topk_ids")
    counts = torch.empty(s.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(s.E + 1, dtype=torch.int32, device=dev)
    src = torch.empty(n, dtype=torch.int32, device=dev)
    dest = torch.empty(n, dtype=torch.int32, device=dev)
    x_perm = None
    if x is not None:
        _expect(x, torch.bfloat16, (s.T, s.d), "x")
        if x_perm_out is not None:
            _expect(x_perm_out, torch.bfloat16, (n, s.d), "x_perm_out")
            x_perm = x_perm_out
        else:
            x_perm = torch.empty((n, s.d), dtype=torch.bfloat16, device=dev)
    _check("moe_dispatch", lib().moe_dispatch(ctypes.byref(s), _ptr(topk_ids), _ptr(x),
                                              _ptr(counts), _ptr(offsets), _ptr(src),
                                              _ptr(dest), _ptr(x_perm), ws.c_ptr, ws.nbytes,
                                              _stream(stream)))
    return counts, offsets, src, dest, x_perm


def moe_dispatch_noalloc(shape, topk_ids, x, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate
    device memory (the library keeps a fixed 1 MiB scratch array per GPU).

    The output tensors are allocated here by PyTorch for convenience; a
    caller that owns its buffers passes them to the C entry point directly.
    Returns (counts [E], offsets [E+1], src_token [T*k], dest [T*k], x_perm).
    """
    s = as_shape(shape)
    dev = topk_ids.device
    n = s.T * s.k
    _expect(topk_ids, torch.int32, (s.T, s.k), "topk_ids")
    counts = torch.empty(s.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(s.E + 1, dtype=torch.int32, device=dev)
    src = torch.empty(n, dtype=torch.int32, device=dev)
    dest = torch.empty(n, dtype=torch.int32, device=dev)
    x_perm = None
    if x is not None:
        _expect(x, torch.bfloat16, (s.T, s.d), "x")
        x_perm = torch.empty((n, s.d), dtype=torch.bfloat16, device=dev)
    _check("moe_dispatch_noalloc",
           lib().moe_dispatch_noalloc(ctypes.byref(s), _ptr(topk_ids), _ptr(x), _ptr(counts),
                                      _ptr(offsets), _ptr(src), _ptr(dest), _ptr(x_perm),
                                      _stream(stream)))
    return counts, offsets, src, dest, x_perm


def moe_dispatch_replicated_workspace_size(shape, num_physical: int) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_dispatch_replicated_workspace_size",
           lib().moe_dispatch_replicated_workspace_size(ctypes.byref(as_shape(shape)),
                                                        int(num_physical), ctypes.byref(out)))
    return out.value


def moe_dispatch_replicated(shape, phys_expert, topk_ids, x, ws: Workspace, stream=None):
    """Dispatch onto physical expert copies (phys_expert [P] int32: the
    logical expert of each physical slot).  Returns (counts_phys [P],
    offsets_phys [P+1], src_token [T*k], dest [T*k], x_perm or None)."""
    s = as_shape(shape)
    dev = topk_ids.device
    n = s.T * s.k
    P = int(phys_expert.numel())
    _expect(topk_ids, torch.int32, (s.T, s.k), "topk_ids")
    if phys_expert.dtype != torch.int32:
        raise TypeError("phys_expert: expected torch.int32")
    counts = torch.empty(P, dtype=torch.int32, device=dev)
    offsets = torch.empty(P + 1, dtype=torch.int32, device=dev)
    src = torch.empty(n, dtype=torch.int32, device=dev)
    dest = torch.empty(n, dtype=torch.int32, device=dev)
    x_perm = None
    if x is not None:
        _expect(x, torch.bfloat16, (s.T, s.d), "x")
        x_perm = torch.empty((n, s.d), dtype=torch.bfloat16, device=dev)
    _check("moe_dispatch_replicated",
           lib().moe_dispatch_replicated(ctypes.byref(s), P, _ptr(phys_expert), _ptr(topk_ids),
                                         _ptr(x), _ptr(counts), _ptr(offsets), _ptr(src),
                                         _ptr(dest), _ptr(x_perm), ws.c_ptr, ws.nbytes,
                                         _stream(stream)))
    return counts, offsets, src, dest, x_perm


def moe_expert_ffn(shape, layout, x_in, seg, M_max, w_gate_up, w_down, ws: Workspace,
                   y_out=None, stream=None):
    s = as_shape(shape)
    if y_out is None:
        y_out = torch.empty(tuple(x_in.shape[:-1]) + (s.d,), dtype=torch.float32,
                            device=x_in.device)
    _expect(w_gate_up, torch.bfloat16, (s.E, 2 * s.inter, s.d), "w_gate_up")
    _expect(w_down, torch.bfloat16, (s.E, s.d, s.inter), "w_down")
    _check("moe_expert_ffn",
           lib().moe_expert_ffn(ctypes.byref(s), int(layout), _ptr(x_in), _ptr(seg),
                                int(M_max), _ptr(w_gate_up), _ptr(w_down), _ptr(y_out),
                                ws.c_ptr, ws.nbytes, _stream(stream)))
    return y_out


def moe_expert_gate_up(shape, layout, x_in, seg, M_max, w_gate_up, ws: Workspace,
                       h_out=None, stream=None):
    s = as_shape(shape)
    if h_out is None:
        h_out = torch.empty(tuple(x_in.shape[:-1]) + (s.inter,), dtype=torch.bfloat16,
                            device=x_in.device)
    _expect(w_gate_up, torch.bfloat16, (s.E, 2 * s.inter, s.d), "w_gate_up")
    _check("moe_expert_gate_up",
           lib().moe_expert_gate_up(ctypes.byref(s), int(layout), _ptr(x_in), _ptr(seg),
                                    int(M_max), _ptr(w_gate_up), _ptr(h_out), ws.c_ptr,
                                    ws.nbytes, _stream(stream)))
    return h_out


def moe_expert_down(shape, layout, h_in, seg, M_max, w_down, ws: Workspace, y_out=None,
                    stream=None):
    s = as_shape(shape)
    if y_out is None:
        y_out = torch.empty(tuple(h_in.shape[:-1]) + (s.d,), dtype=torch.float32,
                            device=h_in.device)
    _expect(w_down, torch.bfloat16, (s.E, s.d, s.inter), "w_down")
    _check("moe_expert_down",
           lib().moe_expert_down(ctypes.byref(s), int(layout), _ptr(h_in), _ptr(seg),
                                 int(M_max), _ptr(w_down), _ptr(y_out), ws.c_ptr, ws.nbytes,
                                 _stream(stream)))
    return y_out


def moe_combine(shape, y_perm, dest, topk_w, y=None, stream=None):
    s = as_shape(shape)
    _expect(y_perm, torch.float32, (s.T * s.k, s.d), "y_perm")
    if y is None:
        y = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=y_perm.device)
    _check("moe_combine", lib().moe_combine(ctypes.byref(s), _ptr(y_perm), _ptr(dest),
                                            _ptr(topk_w), _ptr(y), _stream(stream)))
    return y


def _event_array(events):
    """Host array of 6 cudaEvent_t handles from torch.cuda.Event objects."""
    if events is None:
        return None
    if len(events) != 6:
        raise ValueError("moe_layer takes 6 stage events")
    handles = []
    for ev in events:
        if ev.cuda_event == 0:  # torch creates the event on first record
            ev.record()
        handles.append(ev.cuda_event)
    return (ctypes.c_void_p * 6)(*handles)


def moe_layer(shape, x, w_r, bias, w_gate_up, w_down, ws: Workspace, y=None,
              topk_ids=None, topk_w=None, counts=None, stage_events=None, stream=None):
    s = as_shape(shape)
    _expect(x, torch.bfloat16, (s.T, s.d), "x")
    _expect(w_r, torch.bfloat16, (s.d, s.E), "w_r")
    _expect(w_gate_up, torch.bfloat16, (s.E, 2 * s.inter, s.d), "w_gate_up")
    _expect(w_down, torch.bfloat16, (s.E, s.d, s.inter), "w_down")
    if y is None:
        y = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=x.device)
    _check("moe_layer", lib().moe_layer(ctypes.byref(s), _ptr(x), _ptr(w_r), _ptr(bias),
                                        _ptr(w_gate_up), _ptr(w_down), _ptr(y),
                                        _ptr(topk_ids), _ptr(topk_w), _ptr(counts),
                                        ws.c_ptr, ws.nbytes, _event_array(stage_events),
                                        _stream(stream)))
    return y


MOE_OVERFLOW_DROP = 0
MOE_OVERFLOW_SECOND_ROUND = 1


def moe_expert_capacity(T: int, k: int, E: int, c: float) -> int:
    """C = ceil(c * T * k / E)."""
    return int(lib().moe_expert_capacity(int(T), int(k), int(E), float(c)))


def moe_dispatch_capacity(shape, capacity, overflow, topk_ids, x, ws: Workspace, stream=None):
    """Returns (counts [E], kept [E], ovf_offsets [E+1], dest [T*k],
    src_row [E*C + T*k], x_rows [E*C + T*k, d] or None)."""
    s = as_shape(shape)
    dev = topk_ids.device
    n = s.T * s.k
    rows = s.E * int(capacity) + n
    _expect(topk_ids, torch.int32, (s.T, s.k), "topk_ids")
    counts = torch.empty(s.E, dtype=torch.int32, device=dev)
    kept = torch.empty(s.E, dtype=torch.int32, device=dev)
    ovf = torch.empty(s.E + 1, dtype=torch.int32, device=dev)
    dest = torch.empty(n, dtype=torch.int32, device=dev)
    src = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    x_rows = None
    if x is not None:
        _expect(x, torch.bfloat16, (s.T, s.d), "x")
        x_rows = torch.empty((rows, s.d), dtype=torch.bfloat16, device=dev)
    _check("moe_dispatch_capacity",
           lib().moe_dispatch_capacity(ctypes.byref(s), int(capacity), int(overflow),
                                       _ptr(topk_ids), _ptr(x), _ptr(counts), _ptr(kept),
                                       _ptr(ovf), _ptr(dest), _ptr(src), _ptr(x_rows),
                                       ws.c_ptr, ws.nbytes, _stream(stream)))
    return counts, kept, ovf, dest, src, x_rows


def moe_layer_capacity_workspace_size(shape, capacity) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_layer_capacity_workspace_size",
           lib().moe_layer_capacity_workspace_size(ctypes.byref(as_shape(shape)), int(capacity),
                                                   ctypes.byref(out)))
    return int(out.value)


def moe_layer_capacity(shape, capacity, overflow, x, w_r, bias, w_gate_up, w_down,
                       ws: Workspace, y=None, counts=None, kept=None, stream=None):
    s = as_shape(shape)
    _expect(x, torch.bfloat16, (s.T, s.d), "x")
    _expect(w_r, torch.bfloat16, (s.d, s.E), "w_r")
    _expect(w_gate_up, torch.bfloat16, (s.E, 2 * s.inter, s.d), "w_gate_up")
    _expect(w_down, torch.bfloat16, (s.E, s.d, s.inter), "w_down")
    if y is None:
        y = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=x.device)
    _check("moe_layer_capacity",
           lib().moe_layer_capacity(ctypes.byref(s), int(capacity), int(overflow), _ptr(x),
                                    _ptr(w_r), _ptr(bias), _ptr(w_gate_up), _ptr(w_down),
                                    _ptr(y), _ptr(counts), _ptr(kept), ws.c_ptr, ws.nbytes,
                                    _stream(stream)))
    return y


def moe_eplb_plan(load, num_groups: int, num_nodes: int, num_gpus: int, num_physical: int):
    """Expert placement (host).  load: per-expert loads (numpy).  Returns
    (gpu_slots [num_gpus, num_physical // num_gpus], replicas [E]) as numpy."""
    import numpy as np
    load = np.ascontiguousarray(load, dtype=np.float64)
    E = load.size
    slots = np.empty(num_physical, dtype=np.int32)
    reps = np.empty(E, dtype=np.int32)
    _check("moe_eplb_plan",
           lib().moe_eplb_plan(load.ctypes.data_as(ctypes.c_void_p), E, int(num_groups),
                               int(num_nodes), int(num_gpus), int(num_physical),
                               slots.ctypes.data_as(ctypes.c_void_p),
                               reps.ctypes.data_as(ctypes.c_void_p)))
    return slots.reshape(num_gpus, num_physical // num_gpus), reps


def moe_quantize_fp8_rows(x, stream=None):
    """x [rows, cols] bf16 -> (q [rows, cols] uint8 e4m3 codes, scales [rows, cols/128] fp32)."""
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    sc = torch.empty((rows, cols // 128), dtype=torch.float32, device=x.device)
    _check("moe_quantize_fp8_rows",
           lib().moe_quantize_fp8_rows(_ptr(x), rows, cols, _ptr(q), _ptr(sc), _stream(stream)))
    return q, sc


def moe_quantize_fp8_blocks(w, stream=None):
    """w [mats, rows, cols] bf16 -> (q uint8 codes, scales [mats, rows/128, cols/128] fp32)."""
    mats, rows, cols = w.shape
    q = torch.empty((mats, rows, cols), dtype=torch.uint8, device=w.device)
    sc = torch.empty((mats, rows // 128, cols // 128), dtype=torch.float32, device=w.device)
    _check("moe_quantize_fp8_blocks",
           lib().moe_quantize_fp8_blocks(_ptr(w), mats, rows, cols, _ptr(q), _ptr(sc),
                                         _stream(stream)))
    return q, sc


def moe_expert_ffn_fp8_workspace_size(shape, layout, M_max=0) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_expert_ffn_fp8_workspace_size",
           lib().moe_expert_ffn_fp8_workspace_size(ctypes.byref(as_shape(shape)), int(layout),
                                                   int(M_max), ctypes.byref(out)))
    return int(out.value)


def moe_expert_ffn_fp8(shape, layout, x_q, x_scale, seg, M_max, w_gu_q, w_gu_s, w_dn_q,
                       w_dn_s, ws: Workspace, y_out=None, stream=None):
    s = as_shape(shape)
    rows = x_q.shape[0] if x_q.dim() == 2 else x_q.shape[0] * x_q.shape[1]
    if y_out is None:
        y_out = torch.empty(tuple(x_q.shape[:-1]) + (s.d,), dtype=torch.float32,
                            device=x_q.device)
    _check("moe_expert_ffn_fp8",
           lib().moe_expert_ffn_fp8(ctypes.byref(s), int(layout), _ptr(x_q), _ptr(x_scale),
                                    _ptr(seg), int(M_max), _ptr(w_gu_q), _ptr(w_gu_s),
                                    _ptr(w_dn_q), _ptr(w_dn_s), _ptr(y_out), ws.c_ptr,
                                    ws.nbytes, _stream(stream)))
    return y_out


def moe_layer_fp8_workspace_size(shape) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_layer_fp8_workspace_size",
           lib().moe_layer_fp8_workspace_size(ctypes.byref(as_shape(shape)), ctypes.byref(out)))
    return int(out.value)


def moe_layer_fp8(shape, x, w_r, bias, w_gu_q, w_gu_s, w_dn_q, w_dn_s, ws: Workspace, y=None,
                  counts=None, stream=None):
    s = as_shape(shape)
    _expect(x, torch.bfloat16, (s.T, s.d), "x")
    _expect(w_r, torch.bfloat16, (s.d, s.E), "w_r")
    _expect(w_gu_q, torch.uint8, (s.E, 2 * s.inter, s.d), "w_gate_up_q")
    _expect(w_dn_q, torch.uint8, (s.E, s.d, s.inter), "w_down_q")
    if y is None:
        y = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=x.device)
    _check("moe_layer_fp8",
           lib().moe_layer_fp8(ctypes.byref(s), _ptr(x), _ptr(w_r), _ptr(bias), _ptr(w_gu_q),
                               _ptr(w_gu_s), _ptr(w_dn_q), _ptr(w_dn_s), _ptr(y), _ptr(counts),
                               ws.c_ptr, ws.nbytes, _stream(stream)))
    return y


def moe_selftest_wait_timeout(ws: Workspace, limit_ns: int, stream=None):
    _check("moe_selftest_wait_timeout",
           lib().moe_selftest_wait_timeout(ws.c_ptr, ws.nbytes, int(limit_ns),
                                           _stream(stream)))
