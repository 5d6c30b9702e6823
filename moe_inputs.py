"""Seeded synthetic inputs for the MoE layer (shared by the tests, the bench and
the oracle checks).

This module draws random tensors and nothing else: it holds none of the
layer's arithmetic (no routing, no dispatch, no FFN, no combine).  Every
workload named here is synthetic; no dataset or trained weight is used.

Workloads (hidden d, experts E in G groups, topk_group, k, SwiGLU width inter):

* ``tiny``       T=64,    d=256,  E=16 in G=4,  topk_group=2, k=2, inter=128,
                 sigmoid router with 0.15-scaled per-expert bias.
* ``few_large``  T=2048,  d=4096, E=8,  G=1,    topk_group=1, k=2, inter=14336,
                 softmax router over the logits.
* ``decode``     T=512,   d=7168, E=256 in G=8, topk_group=4, k=8, inter=2048,
                 sigmoid + 0.15 bias (the DeepSeek-V3 shape of the group-limited
                 routing on the "ep-deploy" handbook page).
* ``prefill``    T=16384, rest as ``decode``.
* ``masked_ep``  8 local experts of the ``decode`` weights; per-expert token
                 counts come from routing 4096 ``decode``-router tokens and
                 keeping experts 0-7 (the masked per-rank expert slice of the
                 MoE-TP/EP comparison page).
* ``masked_tp``  256 experts whose SwiGLU width is sliced to 64 (gate_up N=128),
                 the same weight bytes as ``masked_ep``; counts from all 4096
                 routed tokens.

Distributions: x ~ N(0,1); router weight W_r [d,E] and expert weights
~ N(0, 0.02), all cast to bf16; the router bias ~ N(0,1) stays fp32.
Draw order, one generator seeded once: W_r, bias, W_gate_up (one draw per
expert, expert order), W_down (one draw per expert), x.  With this order the
``decode``, ``prefill`` and ``masked_*`` workloads share their router and
expert weights and differ only in x.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, asdict

import torch

SCORE_SIGMOID_BIAS = 0
SCORE_SOFTMAX = 1


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    G: int
    topk_group: int
    k: int
    inter: int
    score: int
    bias_scale: float = 0.15

    def shape(self) -> dict:
        s = asdict(self)
        s.pop("name")
        return s

    def replace(self, **kw) -> "LayerConfig":
        s = asdict(self)
        s.update(kw)
        return LayerConfig(**s)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=64, d=256, E=16, G=4, topk_group=2, k=2, inter=128,
                        score=SCORE_SIGMOID_BIAS),
    "few_large": LayerConfig("few_large", T=2048, d=4096, E=8, G=1, topk_group=1, k=2,
                             inter=14336, score=SCORE_SOFTMAX),
    "decode": LayerConfig("decode", T=512, d=7168, E=256, G=8, topk_group=4, k=8,
                          inter=2048, score=SCORE_SIGMOID_BIAS),
    "prefill": LayerConfig("prefill", T=16384, d=7168, E=256, G=8, topk_group=4, k=8,
                           inter=2048, score=SCORE_SIGMOID_BIAS),
}

# masked per-rank slices: routed with the decode router over this many tokens
MASKED_ROUTE_TOKENS = 4096
MASKED_EP_EXPERTS = 8
MASKED_TP_INTER = 64


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_layer_tensors(cfg: LayerConfig, device="cpu", seed: int = 0,
                       n_tokens: int | None = None, with_x: bool = True,
                       extra_x: dict | None = None, keep_experts=None) -> dict:
    """Draw W_r, bias, W_gate_up, W_down and x for ``cfg`` (see module doc).

    Returns a dict of torch tensors on ``device``:
      x [T,d] bf16, w_r [d,E] bf16, bias [E] fp32,
      w_gate_up [E, 2*inter, d] bf16 (rows 0..inter-1 gate, inter.. up),
      w_down [E, d, inter] bf16.
    ``n_tokens`` overrides T for x only (weights are unchanged).
    ``extra_x`` maps names to token counts: each gets its own x drawn from
    the generator state that follows the weights, i.e. the x that
    ``make_layer_tensors`` gives a workload with the same weights and that
    many tokens (returned as ``out["x_" + name]``).
    ``keep_experts`` (a list of expert indices) keeps only those experts'
    weights, in that order: every expert is still drawn, so x and the kept
    weights are the ones the full draw gives.
    """
    device = torch.device(device)
    g = _gen(device, seed)
    d, E, inter = cfg.d, cfg.E, cfg.inter
    T = cfg.T if n_tokens is None else n_tokens
    w_r = _normal_bf16((d, E), 0.02, g, device)
    bias = torch.randn(E, generator=g, device=device, dtype=torch.float32)
    keep = list(range(E)) if keep_experts is None else [int(e) for e in keep_experts]
    slot = {e: i for i, e in enumerate(keep)}
    w_gu = torch.empty((len(keep), 2 * inter, d), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w = _normal_bf16((2 * inter, d), 0.02, g, device)
        if e in slot:
            w_gu[slot[e]] = w
    w_down = torch.empty((len(keep), d, inter), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w = _normal_bf16((d, inter), 0.02, g, device)
        if e in slot:
            w_down[slot[e]] = w
    out = {"w_r": w_r, "bias": bias, "w_gate_up": w_gu, "w_down": w_down}
    state = g.get_state()
    if with_x:
        out["x"] = _normal_bf16((T, d), 1.0, g, device)
    for name, n in (extra_x or {}).items():
        g.set_state(state)
        out["x_" + name] = _normal_bf16((n, d), 1.0, g, device)
    return out


def make_tensors_for_shape(T: int, d: int, E: int, inter: int, device="cpu",
                           seed: int = 0, x_std: float = 1.0,
                           w_std: float = 0.02) -> dict:
    """Same draw order as ``make_layer_tensors`` for an arbitrary small shape."""
    device = torch.device(device)
    g = _gen(device, seed)
    w_r = _normal_bf16((d, E), w_std, g, device)
    bias = torch.randn(E, generator=g, device=device, dtype=torch.float32)
    w_gu = _normal_bf16((E, 2 * inter, d), w_std, g, device)
    w_down = _normal_bf16((E, d, inter), w_std, g, device)
    x = _normal_bf16((T, d), x_std, g, device)
    return {"x": x, "w_r": w_r, "bias": bias, "w_gate_up": w_gu, "w_down": w_down}


def random_ids(T: int, k: int, E: int, seed: int = 0, skew: float = 0.0) -> torch.Tensor:
    """Random expert ids [T,k] int32, k distinct per row (CPU).

    ``skew`` > 0 draws experts with weights exp(skew * N(0,1)) so that a few
    experts are hot; 0 gives uniform choice.
    """
    g = _gen("cpu", seed)
    if skew > 0:
        logw = torch.randn(E, generator=g) * skew
        p = torch.softmax(logw, 0).expand(T, E)
    else:
        p = torch.full((T, E), 1.0 / E)
    return torch.multinomial(p, k, replacement=False, generator=g).to(torch.int32)


def random_weights(T: int, k: int, seed: int = 0) -> torch.Tensor:
    """Positive random combine weights [T,k] fp32 (CPU), rows not normalised."""
    g = _gen("cpu", seed)
    return torch.rand(T, k, generator=g) + 0.05


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (copied to host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def sha256_of(*tensors: torch.Tensor) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()
