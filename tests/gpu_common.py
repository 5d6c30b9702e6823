"""Shared helpers of the GPU parity tests: cached seeded inputs on the device,
host copies for the oracle, and the tolerance checks stated for the path.

Tolerances:
  * routing (ids, counts, offsets, permutation): bit-exact;
  * router logits: bit-exact (same fixed-order fp32 arithmetic);
  * combine weights: within 1e-6 relative;
  * FFN and layer outputs vs the fp64 oracle: relative Frobenius error
    <= 1e-2 and per element |got - ref| <= 2e-2 + (half a bf16 ulp of ref
    when the result is stored in bf16).
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import dispatch_combine_gb300 as moe
from dispatch_combine_gb300 import build as build_mod
import moe_inputs
from moe_inputs import CONFIGS

MAX_ABS = 2e-2
REL_FRO = 1e-2


def ensure_lib():
    build_mod.build()
    return moe.lib()


def bits(t: torch.Tensor) -> np.ndarray:
    return moe_inputs.bf16_bits(t)


@functools.lru_cache(maxsize=None)
def layer_inputs(name: str, seed: int = 0, n_tokens: int | None = None):
    """Device tensors of a named workload (cached per process)."""
    cfg = CONFIGS[name]
    return moe_inputs.make_layer_tensors(cfg, device="cuda", seed=seed, n_tokens=n_tokens)


@functools.lru_cache(maxsize=None)
def host_bits(name: str, key: str, seed: int = 0, n_tokens: int | None = None):
    return bits(layer_inputs(name, seed, n_tokens)[key])


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def check_close(got, ref, bf16_output: bool, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    bound = MAX_ABS + (half_ulp_bf16(ref) if bf16_output else 0.0)
    worst = float((diff - bound).max()) if diff.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert worst <= 0.0, f"{what}: max excess {worst:.3e} (max abs {diff.max():.3e})"
    assert rel <= REL_FRO, f"{what}: rel Frobenius {rel:.3e}"
    return float(diff.max()), rel


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)
