"""CPU oracle of the single-GPU MoE layer path (test infrastructure only).

This package is the independent reference that the CUDA path is checked
against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it.  It shares no code with the CUDA library and
never calls it.  The arithmetic lives in ``moe_oracle.c`` (plain C, compiled
with ``-O2 -ffp-contract=off``, no fast-math); this module only marshals numpy
arrays through ctypes.

bf16 tensors are passed as ``numpy.uint16`` arrays holding the raw bit
patterns (the top 16 bits of the fp32 value).

Pinned against (tests/test_oracle_*.py, no GPU):
  * router_logits: an fp64 dot product within the fp32 error bound, exact
    integer sums, and a hand-derived value that only the stated summation
    order produces;
  * exp/sigmoid: fp64 exp within 2 ulp over the clamped range;
  * select: the routing simulation printed on the "ep-deploy" handbook page
    (section "EPLB 与路由约束": busiest-GPU ratio 2.87 / 3.97, nodes per token
    3.18 / 3.96), brute-force enumeration of group and expert subsets, and
    plain top-k when there is one group;
  * dispatch: a brute-force sort by (expert, assignment) and its invariants;
  * expert FFN: numpy float64 matmuls of the same definition, and a closed
    form with identity-like weights;
  * combine: identity experts return x, one-hot weights select one expert.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCORE_SIGMOID_BIAS = 0
SCORE_SOFTMAX = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        sig = {
            "oracle_num_threads": (I, []),
            "oracle_set_num_threads": (None, [I]),
            "oracle_router_logits": (None, [P, P, I, I, I, P]),
            "oracle_exp": (F, [F]),
            "oracle_sigmoid": (F, [F]),
            "oracle_exp_array": (None, [P, P, ctypes.c_int64]),
            "oracle_sigmoid_array": (None, [P, P, ctypes.c_int64]),
            "oracle_select": (None, [P, I, I, I, I, I, I, P]),
            "oracle_route_from_logits": (None, [P, P, I, I, I, I, I, I, F, P, P, P]),
            "oracle_route": (None, [P, P, P, I, I, I, I, I, I, I, F, P, P, P]),
            "oracle_dispatch": (I, [P, I, I, I, P, P, P, P]),
            "oracle_dispatch_replicated": (I, [P, I, I, I, I, P, P, P, P, P]),
            "oracle_expert_ffn_rows": (None, [P, P, I, I, I, P, P, I, P, P]),
            "oracle_combine": (None, [P, P, P, I, I, I, P]),
            "oracle_layer_tokens": (None, [P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                           P, I, P, P, P]),
            "oracle_layer_tokens_keep": (None, [P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                                P, I, P, P, P, P]),
            "oracle_expert_capacity": (I, [I, I, I, ctypes.c_double]),
            "oracle_eplb_place": (I, [P, I, I, I, I, I, P, P]),
            "oracle_e4m3_to_float": (F, [ctypes.c_uint8]),
            "oracle_float_to_e4m3": (ctypes.c_uint8, [F]),
            "oracle_quantize_rows_fp8": (None, [P, ctypes.c_int64, I, P, P]),
            "oracle_quantize_blocks_fp8": (None, [P, I, I, I, P, P]),
            "oracle_expert_ffn_rows_fp8": (None, [P, P, P, I, I, I, P, P, P, P, P, P]),
            "oracle_dispatch_capacity": (I, [P, I, I, I, I, I, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 bit patterns must be uint16, got {a.dtype}")
    return a


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------
# bf16 conversions (bit-level, round to nearest even)
# --------------------------------------------------------------------------

def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Router
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """Canonical-order fp32 logits [T,E] of x [T,d] (bf16) and w_r [d,E] (bf16)."""
    x = _u16(x)
    w_r = _u16(w_r)
    T, d = x.shape
    d2, E = w_r.shape
    assert d == d2
    out = np.empty((T, E), dtype=np.float32)
    if T:
        _load().oracle_router_logits(_p(x), _p(w_r), T, d, E, _p(out))
    return out


def exp(y) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.empty_like(y)
    _load().oracle_exp_array(_p(y), _p(out), y.size)
    return out


def sigmoid(l) -> np.ndarray:
    l = _c(l, np.float32)
    out = np.empty_like(l)
    _load().oracle_sigmoid_array(_p(l), _p(out), l.size)
    return out


def select(scores: np.ndarray, G: int, topk_group: int, k: int,
           group_sum_f32: bool) -> np.ndarray:
    """Group-limited top-k on float64 scores [T,E]; returns ids [T,k] int32."""
    s = _c(scores, np.float64)
    T, E = s.shape
    ids = np.empty((T, k), dtype=np.int32)
    if T:
        _load().oracle_select(_p(s), T, E, G, topk_group, k, int(bool(group_sum_f32)),
                              _p(ids))
    return ids


def route_from_logits(logits: np.ndarray, bias, G: int, topk_group: int, k: int,
                      score: int, bias_scale: float = 0.15):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = _c(bias if bias is not None else np.zeros(E), np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    sel = np.empty((T, E), dtype=np.float32)
    if T:
        _load().oracle_route_from_logits(_p(logits), _p(b), T, E, G, topk_group, k,
                                         score, bias_scale, _p(ids), _p(w), _p(sel))
    return ids, w, sel


def route(x, w_r, bias, G, topk_group, k, score, bias_scale=0.15):
    """Full router: returns (ids [T,k] int32, weights [T,k] fp32, logits [T,E])."""
    logits = router_logits(x, w_r)
    ids, w, _ = route_from_logits(logits, bias, G, topk_group, k, score, bias_scale)
    return ids, w, logits


# --------------------------------------------------------------------------
# Dispatch / FFN / combine
# --------------------------------------------------------------------------

def dispatch(ids: np.ndarray, E: int):
    """Stable counting sort: returns counts [E], offsets [E+1], dest [T*k], src [T*k]."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    n = T * k
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    dest = np.empty(n, dtype=np.int32)
    src = np.empty(n, dtype=np.int32)
    rc = _load().oracle_dispatch(_p(ids), T, k, E, _p(counts), _p(offsets), _p(dest),
                                 _p(src))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, offsets, dest, src


def dispatch_replicated(ids: np.ndarray, E: int, phys_expert: np.ndarray):
    """Dispatch onto physical expert copies (reading R15): phys_expert [P] is
    the logical expert of each physical slot.  Returns counts_phys [P],
    offsets_phys [P+1], dest [T*k], src [T*k]."""
    ids = _c(ids, np.int32)
    pe = _c(phys_expert, np.int32)
    T, k = ids.shape
    P = pe.size
    counts = np.empty(P, dtype=np.int32)
    offsets = np.empty(P + 1, dtype=np.int32)
    dest = np.empty(T * k, dtype=np.int32)
    src = np.empty(T * k, dtype=np.int32)
    rc = _load().oracle_dispatch_replicated(_p(ids), T, k, E, P, _p(pe), _p(counts),
                                            _p(offsets), _p(dest), _p(src))
    if rc != 0:
        raise ValueError("expert id out of range or expert without a copy")
    return counts, offsets, dest, src


def expert_ffn_rows(x_rows, row_expert, w_gu, w_down, round_h_bf16=False,
                    return_h=False):
    """SwiGLU FFN of each row with its expert; returns y [n,d] fp32 (and h)."""
    x_rows = _u16(x_rows)
    row_expert = _c(row_expert, np.int32)
    w_gu = _u16(w_gu)
    w_down = _u16(w_down)
    n, d = x_rows.shape
    E, two_inter, d2 = w_gu.shape
    inter = two_inter // 2
    assert d2 == d and w_down.shape == (E, d, inter)
    if n and (row_expert.min() < 0 or row_expert.max() >= E):
        raise ValueError("expert id out of range")
    y = np.empty((n, d), dtype=np.float32)
    h = np.empty((n, inter), dtype=np.float32)
    if n:
        _load().oracle_expert_ffn_rows(_p(x_rows), _p(row_expert), n, d, inter,
                                       _p(w_gu), _p(w_down), int(bool(round_h_bf16)),
                                       _p(h), _p(y))
    return (y, h) if return_h else y


def combine(y_perm, dest, w, T: int, k: int) -> np.ndarray:
    """Weighted combine to token order; returns y [T,d] float64."""
    y_perm = _c(y_perm, np.float32)
    dest = _c(dest, np.int32)
    w = _c(w, np.float32)
    d = y_perm.shape[1]
    y = np.empty((T, d), dtype=np.float64)
    if T:
        _load().oracle_combine(_p(y_perm), _p(dest), _p(w), T, k, d, _p(y))
    return y


def expert_capacity(T, k, E, c):
    """C = ceil(c * T * k / E) (capacity per expert)."""
    return int(_load().oracle_expert_capacity(int(T), int(k), int(E), float(c)))


def dispatch_capacity(ids, E, C, policy):
    """Capacity dispatch (policy 0 drop, 1 second round); returns
    (counts, kept, ovf_offsets, dest, src_row)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    ovf = np.empty(E + 1, np.int32)
    dest = np.empty(T * k, np.int32)
    src = np.empty(E * C + T * k, np.int32)
    rc = _load().oracle_dispatch_capacity(_p(ids), T, k, E, int(C), int(policy), _p(counts),
                                          _p(kept), _p(ovf), _p(dest), _p(src))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, kept, ovf, dest, src


def e4m3_to_float(code: int) -> float:
    return float(_load().oracle_e4m3_to_float(int(code)))


def float_to_e4m3(x: float) -> int:
    return int(_load().oracle_float_to_e4m3(float(x)))


def quantize_rows_fp8(x_bits):
    """Per (row, 128 columns) e4m3 codes and fp32 scales of bf16 rows."""
    x = _u16(x_bits)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    _load().oracle_quantize_rows_fp8(_p(x), rows, cols, _p(q), _p(s))
    return q, s


def quantize_blocks_fp8(w_bits):
    """Per 128 x 128 block e4m3 codes and fp32 scales of [mats, rows, cols] bf16."""
    w = _u16(w_bits)
    mats, rows, cols = w.shape
    q = np.empty((mats, rows, cols), np.uint8)
    s = np.empty((mats, rows // 128, cols // 128), np.float32)
    _load().oracle_quantize_blocks_fp8(_p(w), mats, rows, cols, _p(q), _p(s))
    return q, s


def expert_ffn_rows_fp8(xq, xs, row_expert, wgu_q, wgu_s, wd_q, wd_s, return_h=False):
    """FP8 SwiGLU FFN of each row; returns y [n,d] fp32 (and h as fp32 of its bf16)."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    row_expert = _c(row_expert, np.int32)
    n, d = xq.shape
    inter = wgu_q.shape[1] // 2
    y = np.empty((n, d), np.float32)
    h = np.empty((n, inter), np.float32) if return_h else None
    _load().oracle_expert_ffn_rows_fp8(_p(xq), _p(xs), _p(row_expert), n, d, inter,
                                       _p(_c(wgu_q, np.uint8)), _p(_c(wgu_s, np.float32)),
                                       _p(_c(wd_q, np.uint8)), _p(_c(wd_s, np.float32)),
                                       None if h is None else _p(h), _p(y))
    return (y, h) if return_h else y


def eplb_place(load, groups, nodes, gpus, phys):
    """Expert placement (nodes = 0: global).  Returns (gpu_slots [gpus, phys//gpus]
    logical expert ids, replicas [E])."""
    load = _c(load, np.float64)
    E = load.size
    slots = np.empty(phys, np.int32)
    reps = np.empty(E, np.int32)
    rc = _load().oracle_eplb_place(_p(load), E, int(groups), int(nodes), int(gpus), int(phys),
                                   _p(slots), _p(reps))
    if rc != 0:
        raise ValueError("sizes do not divide")
    return slots.reshape(gpus, phys // gpus), reps


def layer_tokens(x, w_r, bias, w_gu, w_down, shape: dict, tokens, keep=None):
    """Whole layer for the listed tokens; returns (y [n,d] f64, ids, weights).
    keep [n, k] (optional): assignments that add their term (capacity drop)."""
    x = _u16(x)
    w_r = _u16(w_r)
    w_gu = _u16(w_gu)
    w_down = _u16(w_down)
    tokens = _c(tokens, np.int32)
    T, d = x.shape
    E = w_r.shape[1]
    k = shape["k"]
    inter = w_gu.shape[1] // 2
    n = tokens.size
    b = _c(bias if bias is not None else np.zeros(E), np.float32)
    ids = np.empty((n, k), dtype=np.int32)
    wts = np.empty((n, k), dtype=np.float32)
    y = np.empty((n, d), dtype=np.float64)
    kp = None if keep is None else _c(keep, np.uint8)
    if n:
        _load().oracle_layer_tokens_keep(_p(x), _p(w_r), _p(b), _p(w_gu), _p(w_down), T, d,
                                         E, shape["G"], shape["topk_group"], k, inter,
                                         shape["score"], float(shape.get("bias_scale", 0.15)),
                                         _p(tokens), n, None if kp is None else _p(kp),
                                         _p(ids), _p(wts), _p(y))
    return y, ids, wts
