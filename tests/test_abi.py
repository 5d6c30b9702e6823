"""The C-ABI library loads and exports every symbol include/moe.h declares;
host-side validation answers without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from dispatch_combine_gb300 import _lib
from dispatch_combine_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(
        r"(?:moe_status_t|int32_t|int64_t|size_t|void|const\s+char\s*\*)\s*\*?\s*(moe_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                     "moe_layer", "moe_workspace_size", "moe_get_device_status",
                     "moe_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows the signature of each one
    assert sorted(_lib.SIGNATURES) == names


def _shape(**kw):
    base = dict(T=64, d=256, E=16, G=4, topk_group=2, k=2, inter=128, score=0,
                bias_scale=0.15)
    base.update(kw)
    return _lib.as_shape(base)


def _ws_size(lib, shape):
    out = ctypes.c_size_t(0)
    st = lib.moe_workspace_size(ctypes.byref(shape), ctypes.byref(out))
    return st, out.value


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name


def test_workspace_size_valid_and_monotone(lib):
    st, small = _ws_size(lib, _shape())
    assert st == 0 and small > 0 and small % 256 == 0
    st, big = _ws_size(lib, _shape(T=640))
    assert st == 0 and big > small
    # layer workspace holds at least x_perm (bf16) and y_perm (fp32)
    s = _shape(T=512, d=7168, E=256, G=8, topk_group=4, k=8, inter=2048)
    st, n = _ws_size(lib, s)
    assert st == 0 and n >= 512 * 8 * 7168 * 6


@pytest.mark.parametrize("bad", [
    dict(E=15),                   # E % G != 0
    dict(topk_group=5),           # topk_group > G
    dict(topk_group=0),
    dict(k=9),                    # k > topk_group * E / G
    dict(k=0),
    dict(d=100),                  # d % 8 != 0
    dict(E=2048, G=32, topk_group=4),  # E > 1024
    dict(G=64, E=128),            # G > 32
    dict(score=7),
    dict(T=-1),
])
def test_invalid_shapes_rejected(lib, bad):
    st, _ = _ws_size(lib, _shape(**bad))
    assert st == 1  # MOE_ERR_INVALID_ARG


def test_null_pointers_rejected_before_any_launch(lib):
    s = _shape()
    st = lib.moe_route(ctypes.byref(s), None, None, None, None, None, None, None, 0, None)
    assert st == 1
    st = lib.moe_layer(ctypes.byref(s), None, None, None, None, None, None, None, None, None,
                       None, 0, None, None)
    assert st == 1


def test_ffn_unsupported_shapes(lib):
    s = _shape(d=200, inter=128)
    out = ctypes.c_size_t(0)
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(s), 0, 0, ctypes.byref(out)) == 0
    dummy = ctypes.c_void_p(256)
    st = lib.moe_expert_ffn(ctypes.byref(s), 0, dummy, dummy, 0, dummy, dummy, dummy, dummy,
                            1 << 30, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED: d % 64 != 0
    s = _shape(inter=96)
    st = lib.moe_expert_ffn(ctypes.byref(s), 0, dummy, dummy, 0, dummy, dummy, dummy, dummy,
                            1 << 30, None)
    assert st == 2


def test_workspace_checks(lib):
    s = _shape()
    _, need = _ws_size(lib, s)
    dummy = ctypes.c_void_p(256)
    # too small
    st = lib.moe_layer(ctypes.byref(s), dummy, dummy, dummy, dummy, dummy, dummy, None, None,
                       None, dummy, need - 256, None, None)
    assert st == 3
    # misaligned
    st = lib.moe_layer(ctypes.byref(s), dummy, dummy, dummy, dummy, dummy, dummy, None, None,
                       None, ctypes.c_void_p(512 + 16), need, None, None)
    assert st == 3


def test_zero_tokens_is_a_noop(lib):
    s = _shape(T=0)
    st = lib.moe_layer(ctypes.byref(s), None, None, None, None, None, None, None, None, None,
                       None, 0, None, None)
    assert st == 0
    assert lib.moe_layer_launch_count(ctypes.byref(s)) == 0
    # router: screened (d, E multiples of 64: transpose, tensor-core logits,
    # screen, listed logits, listed selection) or logits (1 with the weights
    # resident in shared memory, else a padded copy + the tiled kernel) +
    # select; then count, scan, scatter, gather, gate_up, down, combine
    assert lib.moe_layer_launch_count(ctypes.byref(_shape())) == 9
    decode = _shape(T=512, d=7168, E=256, G=8, topk_group=4, k=8, inter=2048, score=1)
    prefill = _shape(T=16384, d=7168, E=256, G=8, topk_group=4, k=8, inter=2048, score=1)
    few_large = _shape(T=2048, d=4096, E=8, G=1, topk_group=1, k=2, inter=14336)
    e32 = _shape(T=100, d=512, E=32, G=1, topk_group=1, k=4, inter=128)
    assert lib.moe_layer_launch_count(ctypes.byref(decode)) == 12
    assert lib.moe_layer_launch_count(ctypes.byref(prefill)) == 12
    assert lib.moe_layer_launch_count(ctypes.byref(few_large)) == 9
    assert lib.moe_layer_launch_count(ctypes.byref(e32)) == 10


def test_masked_layout_arguments(lib):
    s = _shape()
    out = ctypes.c_size_t(0)
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(s), 1, -1, ctypes.byref(out)) == 1
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(s), 3, 0, ctypes.byref(out)) == 1
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(s), 1, 256, ctypes.byref(out)) == 0
    assert out.value >= 16 * 256 * 128 * 2


def test_layer_yperm_row_bytes(lib):
    # the layers keep their down-GEMM rows compact (fp16 + a code byte per 32
    # columns) where d is a multiple of 256 (whole 256-column down tiles)
    lib.moe_layer_yperm_row_bytes.restype = ctypes.c_int64
    prefill = _shape(T=16384, d=7168, E=256, G=8, topk_group=4, k=8, inter=2048, score=1)
    decode = _shape(T=512, d=7168, E=256, G=8, topk_group=4, k=8, inter=2048, score=1)
    few_large = _shape(T=2048, d=4096, E=8, G=1, topk_group=1, k=2, inter=14336)
    odd_d = _shape(T=2048, d=4160, E=8, G=1, topk_group=1, k=2, inter=1024)
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(prefill)) == 2 * 7168 + 7168 // 32
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(few_large)) == 2 * 4096 + 4096 // 32
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(decode)) == 2 * 7168 + 7168 // 32
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(_shape())) == 2 * 256 + 256 // 32
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(odd_d)) == 4 * 4160
    bad = _shape(T=-1)
    assert lib.moe_layer_yperm_row_bytes(ctypes.byref(bad)) == 0
