"""Benchmark of the single-GPU MoE layer (router -> dispatch -> SwiGLU experts
-> combine) on GB300.

One step = one moe_layer call over one batch of T synthetic tokens, with
inputs resident in HBM.  Prints ONE JSON line (rank 0):
  metric  "MoE-layer tokens/s (1 GB300); % of HBM / bf16 tensor roofline per stage"
  value   whole-job tokens/s over the K timed steps (max time over ranks)
  e2e     the same metric through the C-ABI call with host buffers: every step
          copies x from pinned host memory and reads y back
  roofline  for the dominant kernel, achieved vs the measured peak
  stages  per-stage time and roofline fraction (CUDA events inside moe_layer)
  cpu_baseline  the CPU oracle on a bounded token sample (host cores)

Multi-GPU (torchrun, N ranks): each rank runs its own replica of the layer on
its own batch (data-parallel replicas, no collective on the data path); the
only collectives are the timing barrier and the max-over-ranks reduction.

``--impl reference`` times the CPU oracle instead (rank 0 only), on a bounded
token sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_inputs import CONFIGS, SCORE_SIGMOID_BIAS  # noqa: E402

METRIC = "MoE-layer tokens/s (1 GB300); % of HBM / bf16 tensor roofline per stage"
UNIT = "tokens/s"
DEFAULT_CONFIG = "prefill"
# timed in the same run when the default workload is: same weights, decode batch
DEFAULT_ALSO = {"prefill": "decode"}
L2_BYTES = 126 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FMA peak from the unit counts: 152 SMs x 128 fp32 lanes x 2 FLOP per
# fused multiply-add x 2.07 GHz (the maximum SM clock)
FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# --------------------------------------------------------------------------
# algorithmic work (the arithmetic below is pinned by tests/test_arith_pins.py)
# --------------------------------------------------------------------------

def expert_weight_bytes(c) -> int:
    """gate, up and down weights of one expert, bf16."""
    return 3 * c.d * c.inter * 2


# timed steps that carry the six stage events (every STAGE_EVERY-th)
STAGE_EVERY = 8


def ffn_flops_per_row(c) -> int:
    """gate_up (2*d*2*inter) + down (2*inter*d) per routed row."""
    return 6 * c.d * c.inter


def stage_bytes(c, yperm_row_bytes=None) -> dict:
    """Algorithmic bytes of the bandwidth stages for one layer call.

    router:   read x and W_r, write ids + weights
    dispatch: read ids and x, write x_perm (bf16) and dest + src_token
    combine:  read y_perm and dest + weights, write y (bf16); y_perm rows of
              yperm_row_bytes (moe_layer_yperm_row_bytes: 4*d fp32, or
              2*d + d/32 in the compact form; default fp32)
    """
    T, d, E, k = c.T, c.d, c.E, c.k
    yb = 4 * d if yperm_row_bytes is None else int(yperm_row_bytes)
    return {
        "router": T * d * 2 + d * E * 2 + T * k * 8,
        "dispatch": T * k * 4 + T * d * 2 + T * k * d * 2 + T * k * 8,
        "combine": T * k * yb + T * k * 8 + T * d * 2,
    }


def ffn_work(c, n_touched: int) -> dict:
    rows = c.T * c.k
    return {
        "gate_up": {"flops": 4 * c.d * c.inter * rows,
                    "bytes": n_touched * 2 * c.inter * c.d * 2},
        "down": {"flops": 2 * c.d * c.inter * rows, "bytes": n_touched * c.d * c.inter * 2},
    }


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# DRAM traffic of one launch of a kernel, from an ncu capture summarised in
# profiles/dram_traffic.md; valid only while the kernel's sources are the
# ones the capture was taken from.
KERNEL_SOURCES = {
    "gate_up": ["gemm.cu", "common.cuh"], "down": ["gemm.cu", "common.cuh"],
    "router": ["router.cu", "common.cuh"], "dispatch": ["dispatch.cu", "common.cuh"],
    "combine": ["combine.cu", "common.cuh"],
}


def kernel_source_hash(stage: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[stage]:
        with open(os.path.join(ROOT, "dispatch_combine_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, stage: str):
    """Bytes per launch (DRAM read + write) if profiles/dram_traffic.md holds a
    capture of this stage's kernel at this workload from the current sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        rows = open(path).read().splitlines()
    except OSError:
        return None
    want = kernel_source_hash(stage)
    for ln in rows:
        cells = [x.strip().strip("`") for x in ln.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == workload and cells[1] == stage and cells[2] == want:
            try:
                return float(cells[3])
            except ValueError:
                return None
    return None


def workload_desc(c) -> str:
    score = "sigmoid+0.15*bias" if c.score == SCORE_SIGMOID_BIAS else "softmax"
    g = f"E={c.E} in G={c.G} groups, topk_group={c.topk_group}" if c.G > 1 else f"E={c.E}, G=1"
    return (f"{c.name}: T={c.T}, d={c.d}, {g}, k={c.k}, {score} router, "
            f"SwiGLU inter={c.inter}, bf16")


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = getattr(self, "t_start", 0.0)
        t1 = getattr(self, "t_end", float("inf"))
        inside = [ln for ts, ln in self.lines if t0 <= ts <= t1]
        if not inside:  # region shorter than the sampling period: the nearest sample
            near = min(self.lines, key=lambda tl: abs(tl[0] - 0.5 * (t0 + t1)), default=None)
            inside = [near[1]] if near else []
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() in ("active", "1", "0x1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples taken while the timed region ran
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# distributed helpers (replicas; only timing collectives)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_value(tokens_per_rank: int, world: int, seconds: float, steps: int) -> float:
    """Whole-job throughput: tokens processed by all ranks / wall time."""
    return tokens_per_rank * world * steps / seconds


# --------------------------------------------------------------------------
# CPU oracle timing (reported baseline and the reference arm)
# --------------------------------------------------------------------------

def time_oracle(c, host: dict, n_tokens: int, seed: int = 0) -> dict:
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(c.T, size=min(n_tokens, c.T), replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.layer_tokens(host["x"], host["w_r"], host["bias"], host["w_gate_up"],
                        host["w_down"], c.shape(), toks)
    dt = time.perf_counter() - t0
    return {"value": len(toks) / dt, "seconds": dt, "tokens": int(len(toks)),
            "cores": oracle.num_threads()}


def oracle_sample_size(c, host: dict, seconds: float) -> int:
    """Tokens of oracle work that take about `seconds` on this host: an
    8-token sample is timed first and the count scaled from it."""
    probe = time_oracle(c, host, 8, seed=999)
    per_token = probe["seconds"] / max(probe["tokens"], 1)
    return max(1, min(c.T, int(seconds / per_token)))


def host_inputs(t: dict) -> dict:
    from moe_inputs import bf16_bits
    return {"x": bf16_bits(t["x"]), "w_r": bf16_bits(t["w_r"]),
            "bias": t["bias"].detach().cpu().numpy(), "w_gate_up": bf16_bits(t["w_gate_up"]),
            "w_down": bf16_bits(t["w_down"])}


def run_reference(args, c):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import oracle
    from moe_inputs import make_layer_tensors
    # inputs drawn on the GPU when there is one (faster for the large
    # workloads; drawing is not timed), then copied to the host
    t = make_layer_tensors(c, device="cuda" if torch.cuda.is_available() else "cpu", seed=0)
    host = host_inputs(t)
    del t
    # each step a bounded token sample; the whole run stays within
    # --ref-total-s however many steps are asked for (at least one token a step)
    per_step_s = min(args.ref_step_s, args.ref_total_s / max(args.steps, 1))
    n = oracle_sample_size(c, host, per_step_s)
    for w in range(args.warmup):  # untimed warm-up steps (one token each)
        time_oracle(c, host, 1, seed=1000 + w)
    total_s, total_tok = 0.0, 0
    for s in range(args.steps):
        r = time_oracle(c, host, n, seed=s)
        total_s += r["seconds"]
        total_tok += r["tokens"]
    value = total_tok / total_s
    sample = (f"{n} of {c.T} tokens per step (seeded), full layer per token: canonical "
              f"router, k={c.k} SwiGLU experts in fp64, combine")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(c), "T": c.T, "d": c.d, "E": c.E, "k": c.k,
                   "inter": c.inter},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del torch
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

# a timed region shorter than this is taken against the burst tensor peak
# (the GPU has not reached its power cap yet), a longer one against the
# sustained peak
BURST_REGION_S = 1.0


def tensor_peak(peaks: dict, peak_src: str, region_s: float) -> tuple[float, str]:
    """The bf16 tensor peak that applies to a timed region of region_s seconds."""
    if region_s < BURST_REGION_S:
        return peaks["bf16_tflops"], (f"{peak_src} bf16 burst (timed region {region_s:.2f} s "
                                      f"< {BURST_REGION_S:.0f} s)")
    return peaks["bf16_tflops_sustained"], (f"{peak_src} bf16 sustained (timed region "
                                            f"{region_s:.2f} s)")


def layer_bytes(c, n_touched: int, yperm_row_bytes=None) -> int:
    """Algorithmic HBM bytes of one layer call: the bandwidth stages plus the
    touched experts' weights streamed once."""
    sb = stage_bytes(c, yperm_row_bytes)
    return sb["router"] + sb["dispatch"] + sb["combine"] + n_touched * expert_weight_bytes(c)


def measure_layer(args, c, t, ws, device, world: int, steps: int, warmup: int) -> dict:
    """Time `steps` moe_layer calls of workload c after `warmup` untimed ones
    (CUDA events on the launching stream, clocks sampled inside the timed
    region, max over ranks) and derive the per-stage roofline record."""
    import torch
    import dispatch_combine_gb300 as moe

    x = t["x"]
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    shape = c.shape()
    y = torch.empty(c.T, c.d, dtype=torch.bfloat16, device=device)
    counts = torch.empty(c.E, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    def step(events=None):
        moe.moe_layer(shape, x, t["w_r"], bias, t["w_gate_up"], t["w_down"], ws, y=y,
                      counts=counts, stage_events=events)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit(f"device status error during warm-up ({c.name})")

    K = steps
    # stage events on every STAGE_EVERY-th timed step (an event between two
    # kernels stops the next one from launching early, so the other steps
    # run without them); the stage times are the averages over those steps
    sampled = list(range(0, K, STAGE_EVERY))
    evs = {s: [torch.cuda.Event(enable_timing=True) for _ in range(6)] for s in sampled}
    for row in evs.values():  # create the events before the timed region
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(device.index or 0)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler.mark("t_start")
    start.record(stream)
    for s in range(K):
        step(evs.get(s))
    end.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t_end")
    barrier(world)
    clocks = sampler.stop()
    ms_total = start.elapsed_time(end)
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit(f"device status error in the timed region ({c.name})")
    ms_total_max = max_over_ranks(ms_total, world, device)
    value = job_value(c.T, world, ms_total_max / 1000.0, K)

    # per-stage durations (events recorded on the launching stream)
    names = ["router", "dispatch", "gate_up", "down", "combine"]
    stage_ms = {n: 0.0 for n in names}
    for row in evs.values():
        for i, n in enumerate(names):
            stage_ms[n] += row[i].elapsed_time(row[i + 1])
    stage_ms = {n: v / len(evs) for n, v in stage_ms.items()}

    n_refined = moe.moe_route_refined_count(shape, ws)
    cnt = counts.cpu()
    n_touched = int((cnt > 0).sum())
    mean = float(cnt.float().mean())
    r_imb = float(cnt.max()) / mean if mean > 0 else 0.0
    m_tiles = int(((cnt + 127) // 128).sum())
    tile_fill = float(cnt.sum()) / (128.0 * m_tiles) if m_tiles else 0.0

    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    region_s = ms_total / 1000.0
    tpeak, tpeak_src = tensor_peak(peaks, peak_src, region_s)
    tensor = tpeak * 1e12
    yrb = moe.moe_layer_yperm_row_bytes(shape)
    sb = stage_bytes(c, yrb)
    fw = ffn_work(c, n_touched)
    stages = {}
    for n in ("router", "dispatch", "combine"):
        sec = stage_ms[n] / 1000.0
        stages[n] = {"us": stage_ms[n] * 1000.0, "bound": "hbm", "bytes": sb[n],
                     "achieved_gbs": sb[n] / sec / 1e9, "frac": sb[n] / hbm / sec}
    stages["combine"]["yperm_row_bytes"] = yrb
    # screened router: tensor-core logits, then the fixed-order logits of the
    # experts each token's intervals leave open (at least its k selected;
    # their weight rows come from L2); its HBM bytes stay those of the stage
    r_flops = 2.0 * c.T * c.d * c.E
    if n_refined >= 0:
        stages["router"].update({"screened": True, "refined_pairs": n_refined,
                                 "refined_per_token": n_refined / c.T, "tc_flops": r_flops,
                                 "refine_l2_bytes": n_refined * c.d * 2})
    # otherwise the logits are fp32 multiply-adds on CUDA cores (fixed order):
    # at large T they bound the stage, not its bytes
    elif r_flops / (FP32_TFLOPS * 1e12) > sb["router"] / hbm:
        sec = stage_ms["router"] / 1000.0
        stages["router"].update({"bound": "alu", "flops": r_flops,
                                 "achieved_tflops": r_flops / sec / 1e12,
                                 "peak_tflops_fp32": FP32_TFLOPS,
                                 "frac": r_flops / sec / (FP32_TFLOPS * 1e12)})
    for n in ("gate_up", "down"):
        sec = stage_ms[n] / 1000.0
        t_hbm, t_tc = fw[n]["bytes"] / hbm, fw[n]["flops"] / tensor
        stages[n] = {"us": stage_ms[n] * 1000.0,
                     "bound": "tensor" if t_tc >= t_hbm else "hbm",
                     "flops": fw[n]["flops"], "weight_bytes": fw[n]["bytes"],
                     "achieved_tflops": fw[n]["flops"] / sec / 1e12,
                     "achieved_gbs": fw[n]["bytes"] / sec / 1e9,
                     "frac": max(t_hbm, t_tc) / sec}
    ffn_sec = (stage_ms["gate_up"] + stage_ms["down"]) / 1000.0
    ffn_flops = fw["gate_up"]["flops"] + fw["down"]["flops"]
    ffn_wbytes = fw["gate_up"]["bytes"] + fw["down"]["bytes"]
    ffn_bound = "tensor" if ffn_flops / tensor >= ffn_wbytes / hbm else "hbm"
    ffn = {"us": ffn_sec * 1e6, "bound": ffn_bound,
           "frac": max(ffn_wbytes / hbm, ffn_flops / tensor) / ffn_sec,
           "tensor_frac": ffn_flops / tensor / ffn_sec, "hbm_frac": ffn_wbytes / hbm / ffn_sec,
           "n_touched_experts": n_touched, "r_imbalance": r_imb,
           "m_tiles_128": m_tiles, "tile_fill": tile_fill}
    # the whole layer against its own floor: max(all algorithmic HBM bytes,
    # FFN FLOPs at the tensor peak) over the measured time per layer
    lb = layer_bytes(c, n_touched, yrb)
    layer_s = ms_total_max / 1000.0 / K
    layer = {"us": layer_s * 1e6, "bytes": lb, "flops": ffn_flops,
             "hbm_frac": lb / hbm / layer_s, "tensor_frac": ffn_flops / tensor / layer_s,
             "bound": "tensor" if ffn_flops / tensor >= lb / hbm else "hbm"}
    layer["frac"] = max(layer["hbm_frac"], layer["tensor_frac"])

    dominant = max(names, key=lambda n: stage_ms[n])
    dom = stages[dominant]
    if dom["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dom["achieved_tflops"], "peak": tpeak,
                "unit": "TFLOP/s", "frac": dom["achieved_tflops"] / tpeak}
        roof["peak_source"] = tpeak_src
    else:
        ach = dom.get("weight_bytes", dom.get("bytes")) / (stage_ms[dominant] / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
        roof["peak_source"] = f"{peak_src} HBM copy"
    roof["traffic"] = measured_traffic(c.name, dominant)
    roof["kernel"] = dominant
    return {"value": value, "ms_total": ms_total_max, "ms_per_step": ms_total_max / K,
            "steps": K, "warmup": warmup, "roofline": roof, "stages": stages, "ffn": ffn,
            "layer": layer, "clocks": clocks, "y": y, "launches": moe.moe_layer_launch_count(shape) * K}


def run_gpu(args, c):
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import make_layer_tensors

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the MoE path has no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    moe.lib()  # raises if libmoe.so is missing

    # workloads that share this one's weights and are timed in the same run
    also = [a for a in (args.also.split(",") if args.also else []) if a and a != c.name]
    for a in also:
        o = CONFIGS[a]
        if (o.d, o.E, o.G, o.inter, o.score) != (c.d, c.E, c.G, c.inter, c.score):
            raise SystemExit(f"--also {a}: its weights differ from {c.name}'s")
    t = make_layer_tensors(c, device=device, seed=0, extra_x={a: CONFIGS[a].T for a in also})
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    shape = c.shape()
    ws_bytes = max(moe.moe_workspace_size(CONFIGS[n].shape()) for n in [c.name] + also)
    ws = moe.Workspace(ws_bytes, device=device)
    stream = torch.cuda.current_stream(device)
    # the router weight's prepared copy (transposed, with column norms) is
    # made once, like any one-time weight layout step, and used by every call
    router_prep = None
    try:
        router_prep = moe.moe_router_prepare(shape, t["w_r"])
    except moe.MoEError as e:
        if e.status != 2:  # MOE_ERR_UNSUPPORTED: this shape is not screened
            raise

    main = measure_layer(args, c, t, ws, device, world, args.steps, args.warmup)
    y = main["y"]

    # end to end through the C ABI with host buffers: every step copies its
    # x from pinned host memory and reads its y back, on two copy streams
    # with double-buffered device tensors, so step s+1's upload and step
    # s-1's read-back overlap step s's layer; all copies lie inside the
    # timed region
    e2e = None
    e2e_steps = args.steps if args.e2e_steps is None else args.e2e_steps
    if e2e_steps > 0:
        x_host = t["x"].cpu().pin_memory()
        y_host = [torch.empty(c.T, c.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(t["x"]) for _ in range(2)]
        y_dev = [torch.empty_like(y) for _ in range(2)]
        h2d = torch.cuda.Stream(device)
        d2h = torch.cuda.Stream(device)
        ev_up = [torch.cuda.Event() for _ in range(2)]     # x_dev[b] filled
        ev_done = [torch.cuda.Event() for _ in range(2)]   # layer on buffer b done
        ev_back = [torch.cuda.Event() for _ in range(2)]   # y_dev[b] read back
        for b in range(2):  # recorded once so that the first waits are no-ops
            ev_done[b].record(stream)
            ev_back[b].record(stream)

        def e2e_step(i):
            b = i % 2
            h2d.wait_event(ev_done[b])  # the layer of step i-2 has read x_dev[b]
            with torch.cuda.stream(h2d):
                x_dev[b].copy_(x_host, non_blocking=True)
            ev_up[b].record(h2d)
            stream.wait_event(ev_up[b])
            stream.wait_event(ev_back[b])  # y_dev[b] of step i-2 is back on the host
            moe.moe_layer(shape, x_dev[b], t["w_r"], bias, t["w_gate_up"], t["w_down"], ws,
                          y=y_dev[b], stream=stream)
            ev_done[b].record(stream)
            d2h.wait_event(ev_done[b])
            with torch.cuda.stream(d2h):
                y_host[b].copy_(y_dev[b], non_blocking=True)
            ev_back[b].record(d2h)

        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d.wait_event(e0)
        d2h.wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i)
        for b in range(2):  # the region ends when the last read-backs are done
            stream.wait_event(ev_back[b])
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        e2e = {"value": job_value(c.T, world, ms / 1000.0, e2e_steps), "unit": UNIT,
               "h2d_bytes_per_step": c.T * c.d * 2, "d2h_bytes_per_step": c.T * c.d * 2,
               "steps": e2e_steps}
        del x_host, y_host, x_dev, y_dev

    # the other workloads of the same weights (the decode batch beside the
    # prefill one): full stage records of their own, nested in this line
    also_rec = {}
    for a in also:
        ca = CONFIGS[a]
        ta = dict(t)
        ta["x"] = t["x_" + a]
        r = measure_layer(args, ca, ta, ws, device, world, args.also_steps or args.steps,
                          args.warmup)
        r.pop("y")
        also_rec[a] = {"workload": workload_desc(ca), "metric": METRIC, "unit": UNIT, **r}
        main["launches"] += r.pop("launches")
        also_rec[a].pop("launches", None)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_sample_s > 0:
        import oracle
        host = host_inputs(t)
        n = oracle_sample_size(c, host, args.cpu_sample_s)
        r = time_oracle(c, host, n)
        cpu = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['tokens']} of {c.T} tokens (seeded), full layer per token, "
                         f"{r['seconds']:.1f} s"}

    if router_prep is not None:
        router_prep.release()
    l2_note = ("inputs larger than L2 (expert weights "
               f"{c.E * expert_weight_bytes(c) / 1e9:.2f} GB)"
               if c.E * expert_weight_bytes(c) > L2_BYTES else
               "all inputs fit in L2 (hot-L2 timing)")
    line = {
        "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_desc(c), "T": c.T, "d": c.d, "E": c.E, "G": c.G,
                   "topk_group": c.topk_group, "k": c.k, "inter": c.inter,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": l2_note,
                   "router_weight": ("prepared once (transposed copy + column norms)"
                                     if router_prep is not None else "used as given")},
        "roofline": main["roofline"],
        "stages": main["stages"],
        "ffn": main["ffn"],
        "layer": main["layer"],
        "clocks": main["clocks"],
        "e2e": e2e,
        "gpu_launches": main["launches"],
        "cpu_baseline": cpu,
    }
    if also_rec:
        line["also"] = also_rec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# masked per-rank expert slices (expert FFN only)
# --------------------------------------------------------------------------

def run_masked(args):
    """Time the masked expert FFN on a per-rank slice (its own JSON line).

    Token counts come from routing 4096 tokens through the decode router on
    the GPU (moe_route + moe_dispatch); "ep" keeps experts 0-7 of the decode
    weights (d=7168, inter=2048), "tp" keeps all 256 experts with the SwiGLU
    width sliced to 64 (gate_up N=128), the same weight bytes.  Reported:
    gate_up+SwiGLU alone and the whole FFN (gate_up + down), in microseconds
    and as a fraction of the HBM roofline of the weight bytes.
    """
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import (MASKED_EP_EXPERTS, MASKED_ROUTE_TOKENS, MASKED_TP_INTER,
                            make_layer_tensors)
    torch.cuda.set_device(0)
    cfg = CONFIGS["decode"]
    t = make_layer_tensors(cfg, device="cuda", seed=0, n_tokens=MASKED_ROUTE_TOKENS)
    rshape = cfg.replace(T=MASKED_ROUTE_TOKENS).shape()
    ws = moe.Workspace(moe.moe_workspace_size(rshape))
    ids, _, _ = moe.moe_route(rshape, t["x"], t["w_r"], t["bias"], ws)
    counts, offsets, src, _, _ = moe.moe_dispatch(rshape, ids, None, ws)
    counts_h, offsets_h = counts.cpu(), offsets.cpu()
    if args.masked == "ep":
        experts = list(range(MASKED_EP_EXPERTS))
        w_gu = t["w_gate_up"][:MASKED_EP_EXPERTS].contiguous()
        w_down = t["w_down"][:MASKED_EP_EXPERTS].contiguous()
        inter = cfg.inter
    else:
        experts = list(range(cfg.E))
        i0 = MASKED_TP_INTER
        w_gu = torch.cat([t["w_gate_up"][:, :i0], t["w_gate_up"][:, cfg.inter:cfg.inter + i0]],
                         dim=1).contiguous()
        w_down = t["w_down"][:, :, :i0].contiguous()
        inter = i0
    del t["w_gate_up"], t["w_down"]
    mm_h = counts_h[experts]
    M_max = max(128, int((int(mm_h.max()) + 127) // 128 * 128))
    buf = torch.zeros(len(experts), M_max, cfg.d, dtype=torch.bfloat16, device="cuda")
    for i, e in enumerate(experts):
        rows = src[int(offsets_h[e]):int(offsets_h[e + 1])].long()
        buf[i, :rows.numel()] = t["x"][rows]
    mm = mm_h.to(torch.int32).cuda()
    shape = dict(T=1, d=cfg.d, E=len(experts), G=1, topk_group=1, k=1, inter=inter, score=1,
                 bias_scale=0.15)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_MASKED, M_max))
    h = torch.empty(len(experts), M_max, inter, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(len(experts), M_max, cfg.d, dtype=torch.float32, device="cuda")

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / args.steps

    us_gu = timed(lambda: moe.moe_expert_gate_up(shape, moe.MOE_LAYOUT_MASKED, buf, mm, M_max,
                                                 w_gu, fws, h_out=h))
    us_ffn = timed(lambda: moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_MASKED, buf, mm, M_max,
                                              w_gu, w_down, fws, y_out=y))
    if moe.moe_get_device_status(fws) != 0:
        raise SystemExit("device status error")
    peaks, src_p = load_peaks()
    touched = [i for i, e in enumerate(experts) if int(mm_h[i]) > 0]
    gu_bytes = len(touched) * 2 * inter * cfg.d * 2
    dn_bytes = len(touched) * cfg.d * inter * 2
    rows = int(mm_h.sum())
    line = {
        "metric": f"masked expert FFN ({args.masked}) us", "impl": "gb300",
        "value": us_ffn, "unit": "us", "higher_is_better": False, "steps": args.steps,
        "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": (f"masked per-rank slice '{args.masked}': {len(experts)} experts, "
                                f"d={cfg.d}, inter={inter} (gate_up N={2 * inter}), M_max={M_max}"),
                   "rows": rows, "masked_m_min": int(mm_h.min()), "masked_m_max": int(mm_h.max()),
                   "masked_m_mean": float(mm_h.float().mean()), "touched_experts": len(touched)},
        "gate_up_us": us_gu,
        "gate_up_hbm_frac": gu_bytes / (peaks["hbm_gbs"] * 1e9) / (us_gu * 1e-6),
        "ffn_hbm_frac": (gu_bytes + dn_bytes) / (peaks["hbm_gbs"] * 1e9) / (us_ffn * 1e-6),
        "weight_bytes": gu_bytes + dn_bytes, "peak_source": src_p,
    }
    print(json.dumps(line), flush=True)
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", choices=sorted(CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--also", default=None,
                    help="comma-separated workloads with the same weights, timed in the same "
                         "run and nested in the line under 'also' (default: decode beside "
                         "prefill; '' for none)")
    ap.add_argument("--also-steps", type=int, default=None,
                    help="timed steps of the --also workloads (default: --steps)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="timed steps of the end-to-end measurement (default: --steps, so both "
                         "reach the same clocks; 0 = skip)")
    ap.add_argument("--cpu-sample-s", type=float, default=15.0,
                    help="seconds of CPU oracle work for cpu_baseline (0 = skip)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the layer with FP8 experts (own line)")
    ap.add_argument("--eplb", action="store_true",
                    help="plan expert placements on the routed loads (own line)")
    ap.add_argument("--capacity", type=float, default=None,
                    help="time the capacity variant with this capacity factor (own line)")
    ap.add_argument("--overflow", choices=["drop", "second"], default="drop")
    ap.add_argument("--masked", choices=["ep", "tp"], default=None,
                    help="time the masked expert FFN of a per-rank slice instead")
    ap.add_argument("--ref-step-s", type=float, default=4.0,
                    help="seconds of oracle work per step of --impl reference at most")
    ap.add_argument("--ref-total-s", type=float, default=120.0,
                    help="seconds of oracle work over all steps of --impl reference (about; "
                         "each step runs at least one token)")
    ap.add_argument("--stage-only", choices=["dispatch", "combine"], default=None,
                    help="time one bandwidth stage alone on seeded ids (own line)")
    ap.add_argument("--route-only", action="store_true",
                    help="time the router alone (screened and fixed-order; own line)")
    ap.add_argument("--ffn-counts", default=None, metavar="WORKLOAD:N",
                    help="time the expert FFN alone on N of the workload's touched experts with "
                         "their real row counts (own line)")
    ap.add_argument("--ffn-rows", default=None, metavar="E,R",
                    help="time the expert FFN alone on E experts x R rows at the workload's "
                         "d and inter (bf16, or FP8 with --fp8; own line)")
    a = ap.parse_args(argv)
    if a.also is None:
        a.also = DEFAULT_ALSO.get(a.config, "")
    return a


def run_route_only(args):
    """The router alone on the workload's x and W_r (no expert weights on the
    device): moe_route without logits (screened where the shape allows) and
    with logits (the fixed-order path), each timed over the steps."""
    import torch
    import dispatch_combine_gb300 as moe
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    g = torch.Generator(device="cuda").manual_seed(0)
    w_r = (torch.randn(c.d, c.E, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    bias = torch.randn(c.E, device="cuda", generator=g, dtype=torch.float32)
    x = torch.randn(c.T, c.d, device="cuda", generator=g).to(torch.bfloat16)
    shape = c.shape()
    b = bias if c.score == SCORE_SIGMOID_BIAS else None
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    ids = torch.empty(c.T, c.k, dtype=torch.int32, device="cuda")
    w = torch.empty(c.T, c.k, dtype=torch.float32, device="cuda")
    lg = torch.empty(c.T, c.E, dtype=torch.float32, device="cuda")
    out = {}
    router_prep = None
    try:
        router_prep = moe.moe_router_prepare(shape, w_r)
    except moe.MoEError as e:
        if e.status != 2:  # not screened
            raise
    for label, logits in (("screened", None), ("fixed_order", lg)):
        def step():
            moe.moe_route(shape, x, w_r, b, ws, topk_ids=ids, topk_w=w, logits=logits)
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        out[label] = e0.elapsed_time(e1) * 1000.0 / args.steps
        if logits is None:
            out["refined_pairs"] = moe.moe_route_refined_count(shape, ws)
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status error")
    if router_prep is not None:
        router_prep.release()
    line = {
        "metric": "router alone: us per call", "impl": "gb300", "value": out["screened"],
        "unit": "us", "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(c)},
        "fixed_order_us": out["fixed_order"], "refined_pairs": out["refined_pairs"],
        "tokens_per_s": c.T / (out["screened"] * 1e-6),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_stage_only(args):
    """One bandwidth stage alone at the workload's T, k, d, E, with its inputs
    larger than L2: "dispatch" (moe_dispatch with the row gather, on seeded
    random expert ids with a mild hot-expert skew) or "combine" (moe_combine
    of a seeded fp32 y_perm).  Reports us per call and the algorithmic bytes
    over that time against the measured copy bandwidth (own line)."""
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import random_ids
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    shape = c.shape()
    n = c.T * c.k
    g = torch.Generator(device="cuda").manual_seed(0)
    ids = random_ids(c.T, c.k, c.E, seed=0, skew=1.0).cuda()
    # the dispatch's part of a workspace (status, chunk histograms) is small;
    # the layer's x_perm / y_perm regions are not needed here
    ws = moe.Workspace(16 << 20)
    if args.stage_only == "dispatch":
        x = torch.randn(c.T, c.d, device="cuda", generator=g).to(torch.bfloat16)
        xp = torch.empty(n, c.d, dtype=torch.bfloat16, device="cuda")

        def step():
            moe.moe_dispatch(shape, ids, x, ws, x_perm_out=xp)
    else:
        _, _, _, dest, _ = moe.moe_dispatch(shape, ids, None, ws)
        y_perm = torch.randn(n, c.d, device="cuda", generator=g, dtype=torch.float32)
        w = torch.rand(c.T, c.k, device="cuda", generator=g, dtype=torch.float32)
        y = torch.empty(c.T, c.d, dtype=torch.bfloat16, device="cuda")

        def step():
            moe.moe_combine(shape, y_perm, dest, w, y=y)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status error")
    us = e0.elapsed_time(e1) * 1000.0 / args.steps
    nbytes = stage_bytes(c)[args.stage_only]
    peaks, peak_src = load_peaks()
    line = {
        "metric": f"{args.stage_only} alone: us per call", "impl": "gb300", "value": us,
        "unit": "us", "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16" if args.stage_only == "dispatch" else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(c), "ids": "seeded random, skew 1.0"},
        "bytes": nbytes, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
        "hbm_fraction": nbytes / (us * 1e-6) / (peaks["hbm_gbs"] * 1e9),
        "peak_source": peak_src,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ffn_only(args):
    """Expert FFN alone (gate_up + SwiGLU, down) on E experts of R rows each,
    contiguous layout, at the workload's d and inter: the GEMM kernels
    without routing or dispatch, with a small device footprint (own line)."""
    import torch
    import dispatch_combine_gb300 as moe
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    E, R = (int(v) for v in args.ffn_rows.split(","))
    d, inter = c.d, c.inter
    g = torch.Generator(device="cuda").manual_seed(0)
    w_gu = (torch.randn(E, 2 * inter, d, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    w_dn = (torch.randn(E, d, inter, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(E * R, d, device="cuda", generator=g).to(torch.bfloat16)
    offsets = torch.arange(E + 1, dtype=torch.int32, device="cuda") * R
    shape = dict(T=E * R, d=d, E=E, G=1, topk_group=1, k=1, inter=inter, score=1,
                 bias_scale=0.15)
    y = torch.empty(E * R, d, dtype=torch.float32, device="cuda")
    if args.fp8:
        gq, gs = moe.moe_quantize_fp8_blocks(w_gu)
        dq, ds = moe.moe_quantize_fp8_blocks(w_dn)
        del w_gu, w_dn
        xq, xs = moe.moe_quantize_fp8_rows(x)
        ws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))

        def step():
            moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_CONTIGUOUS, xq, xs, offsets, 0, gq, gs,
                                   dq, ds, ws, y_out=y)
        wbytes = E * 3 * d * inter
    else:
        ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))

        def step():
            moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x, offsets, 0, w_gu, w_dn, ws,
                               y_out=y)
        wbytes = E * 3 * d * inter * 2
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status error")
    sec = e0.elapsed_time(e1) / 1000.0 / args.steps
    flops = 6.0 * E * R * d * inter
    peaks, peak_src = load_peaks()
    line = {
        "metric": "expert FFN alone: weight GB/s and TFLOP/s", "impl": "gb300",
        "value": wbytes / sec / 1e9, "unit": "GB/s", "higher_is_better": True,
        "steps": args.steps, "warmup": args.warmup, "us_per_step": sec * 1e6,
        "dtype": "e4m3" if args.fp8 else "bf16", "data": "synthetic",
        "config": {"workload": f"{E} experts x {R} rows, d={d}, inter={inter} "
                               f"(from {c.name})", "weight_bytes": wbytes},
        "tflops": flops / sec / 1e12,
        "hbm_fraction": wbytes / sec / (peaks["hbm_gbs"] * 1e9),
        "peak_source": peak_src,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ffn_counts(args):
    """Expert FFN alone on a subset of a workload's experts with their real
    row counts (own line): the workload's tokens are routed on the GPU, the
    touched experts ranked by count, and every (touched / n)-th of them kept,
    so the subset's count mix follows the full launch's; the rows are the
    tokens those experts received, in dispatch order.  Small enough on the
    device for an ncu capture (weights of n experts only)."""
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import make_layer_tensors
    torch.cuda.set_device(0)
    name, n_sub = args.ffn_counts.split(":")
    c = CONFIGS[name]
    n_sub = int(n_sub)
    t = make_layer_tensors(c, device="cuda", seed=0, keep_experts=[])
    shape = c.shape()
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    ids, _, _ = moe.moe_route(shape, t["x"], t["w_r"], bias, ws)
    counts, offsets, src, _, _ = moe.moe_dispatch(shape, ids, None, ws)
    cnt = counts.cpu()
    touched = [int(e) for e in torch.argsort(cnt, descending=True, stable=True) if cnt[e] > 0]
    step = max(1, len(touched) // n_sub)
    sub = sorted(touched[::step][:n_sub])
    del ws
    tw = make_layer_tensors(c, device="cuda", seed=0, with_x=False, keep_experts=sub)
    off_h = offsets.cpu()
    rows = torch.cat([src[int(off_h[e]):int(off_h[e + 1])] for e in sub]).long()
    x = t["x"][rows].contiguous()
    sub_counts = torch.tensor([int(cnt[e]) for e in sub], dtype=torch.int32)
    offs = torch.zeros(len(sub) + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(sub_counts, 0)
    offs = offs.cuda()
    fshape = dict(T=int(rows.numel()), d=c.d, E=len(sub), G=1, topk_group=1, k=1,
                  inter=c.inter, score=1, bias_scale=0.15)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(fshape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = torch.empty(rows.numel(), c.d, dtype=torch.float32, device="cuda")
    del t

    def step_fn():
        moe.moe_expert_ffn(fshape, moe.MOE_LAYOUT_CONTIGUOUS, x, offs, 0, tw["w_gate_up"],
                           tw["w_down"], fws, y_out=y)

    for _ in range(args.warmup):
        step_fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step_fn()
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(fws) != 0:
        raise SystemExit("device status error")
    us = e0.elapsed_time(e1) * 1000.0 / max(args.steps, 1)
    R = int(rows.numel())
    gu_w = len(sub) * 2 * c.inter * c.d * 2
    dn_w = len(sub) * c.d * c.inter * 2
    line = {
        "metric": "expert FFN on a real-count expert subset: us per call", "impl": "gb300",
        "value": us, "unit": "us", "higher_is_better": False, "steps": args.steps,
        "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{len(sub)} of the {len(touched)} experts touched by "
                               f"{workload_desc(c)}, every {step}-th by count",
                   "experts": sub, "counts": sub_counts.tolist(), "rows": R},
        # algorithmic bytes of each GEMM launch on the subset: weights once,
        # rows in, result out (h bf16; y fp32)
        "algorithmic_bytes": {"gate_up": gu_w + R * c.d * 2 + R * c.inter * 2,
                              "down": dn_w + R * c.inter * 2 + R * c.d * 4},
        "full_launch_algorithmic_bytes": {
            "gate_up": len(touched) * 2 * c.inter * c.d * 2 + c.T * c.k * (c.d + c.inter) * 2,
            "down": len(touched) * c.d * c.inter * 2 + c.T * c.k * (c.inter * 2 + c.d * 4)},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_capacity(args):
    """Time the capacity variant of the layer (its own JSON line): capacity
    C = ceil(c*T*k/E) per expert, overflow dropped or run in a second round."""
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import make_layer_tensors
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    t = make_layer_tensors(c, device="cuda", seed=0)
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    shape = c.shape()
    C = moe.moe_expert_capacity(c.T, c.k, c.E, args.capacity)
    policy = moe.MOE_OVERFLOW_DROP if args.overflow == "drop" else moe.MOE_OVERFLOW_SECOND_ROUND
    ws = moe.Workspace(moe.moe_layer_capacity_workspace_size(shape, C))
    y = torch.empty(c.T, c.d, dtype=torch.bfloat16, device="cuda")
    counts = torch.empty(c.E, dtype=torch.int32, device="cuda")
    kept = torch.empty(c.E, dtype=torch.int32, device="cuda")

    def step():
        moe.moe_layer_capacity(shape, C, policy, t["x"], t["w_r"], bias, t["w_gate_up"],
                               t["w_down"], ws, y=y, counts=counts, kept=kept)

    router_prep = None
    try:
        router_prep = moe.moe_router_prepare(shape, t["w_r"])  # once, like the main line
    except moe.MoEError as e:
        if e.status != 2:  # MOE_ERR_UNSUPPORTED: this shape is not screened
            raise
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status error")
    ms = e0.elapsed_time(e1) / args.steps
    n = c.T * c.k
    dropped = int((counts - kept).sum()) if policy == moe.MOE_OVERFLOW_DROP else 0
    line = {
        "metric": METRIC + f" (capacity factor {args.capacity}, overflow {args.overflow})",
        "impl": "gb300", "value": c.T / (ms / 1000.0), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(c), "capacity": C, "capacity_factor": args.capacity,
                   "overflow": args.overflow, "padded_rows": c.E * C,
                   "overflow_rows": int((counts - kept).sum()),
                   "dropped_fraction": dropped / n},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fp8(args):
    """Time the FP8 layer (its own JSON line): e4m3 weights with 128 x 128
    block scales (quantized once, outside the timed region), activations
    quantized per row and 128 columns inside the layer."""
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import make_layer_tensors
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    t = make_layer_tensors(c, device="cuda", seed=0)
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    shape = c.shape()
    gq, gs = moe.moe_quantize_fp8_blocks(t["w_gate_up"])
    dq, ds = moe.moe_quantize_fp8_blocks(t["w_down"])
    del t["w_gate_up"], t["w_down"]
    ws = moe.Workspace(moe.moe_layer_fp8_workspace_size(shape))
    y = torch.empty(c.T, c.d, dtype=torch.bfloat16, device="cuda")
    counts = torch.empty(c.E, dtype=torch.int32, device="cuda")

    def step():
        moe.moe_layer_fp8(shape, t["x"], t["w_r"], bias, gq, gs, dq, ds, ws, y=y, counts=counts)

    router_prep = None
    try:
        router_prep = moe.moe_router_prepare(shape, t["w_r"])  # once, like the main line
    except moe.MoEError as e:
        if e.status != 2:  # MOE_ERR_UNSUPPORTED: this shape is not screened
            raise
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler.mark("t_start")
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    sampler.mark("t_end")
    clocks = sampler.stop()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status error")
    ms = e0.elapsed_time(e1) / args.steps
    cnt = counts.cpu()
    touched = int((cnt > 0).sum())
    w_bytes = touched * 3 * c.d * c.inter          # e4m3: one byte per weight
    flops = 6.0 * c.T * c.k * c.d * c.inter
    peaks, peak_src = load_peaks()
    # the FP8 expert FFN alone (both GEMMs and the h quantization between
    # them) on the same routing's rows in dispatch order
    rws = moe.Workspace(moe.moe_workspace_size(shape))
    ids, _, _ = moe.moe_route(shape, t["x"], t["w_r"], bias, rws)
    _, offsets, _, _, x_perm = moe.moe_dispatch(shape, ids, t["x"], rws)
    xq_p, xs_p = moe.moe_quantize_fp8_rows(x_perm)
    del x_perm, rws
    fshape = dict(T=c.T * c.k, d=c.d, E=c.E, G=1, topk_group=1, k=1, inter=c.inter, score=1,
                  bias_scale=0.15)
    fws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(fshape,
                                                              moe.MOE_LAYOUT_CONTIGUOUS))
    y_f = torch.empty(c.T * c.k, c.d, dtype=torch.float32, device="cuda")

    def ffn_step():
        moe.moe_expert_ffn_fp8(fshape, moe.MOE_LAYOUT_CONTIGUOUS, xq_p, xs_p, offsets, 0, gq, gs,
                               dq, ds, fws, y_out=y_f)

    for _ in range(args.warmup):
        ffn_step()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        ffn_step()
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(fws) != 0:
        raise SystemExit("device status error")
    ffn_s = e0.elapsed_time(e1) / 1000.0 / args.steps
    # algorithmic bytes of the FFN: the touched weights once; gate_up reads
    # the FP8 rows and their scales and writes h's codes and scales (h is
    # quantized in its epilogue); down reads those and writes the fp32 rows
    n = c.T * c.k
    h_bytes = n * (c.inter + 4 * (c.inter // 128))
    ffn_bytes = w_bytes + n * (c.d + 4 * (c.d // 128)) + 2 * h_bytes + n * c.d * 4
    line = {
        "metric": METRIC + " (FP8 e4m3 experts, block scales)", "impl": "gb300",
        "value": c.T / (ms / 1000.0), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": workload_desc(c), "weights": "e4m3, power-of-two fp32 scale per 128x128 block",
                   "activations": "e4m3, power-of-two fp32 scale per row and 128 columns (h: in the gate_up epilogue)",
                   "touched_experts": touched},
        "layer_weight_bytes_fp8": w_bytes,
        "layer_hbm_fraction_of_weights": w_bytes / (ms / 1000.0) / (peaks["hbm_gbs"] * 1e9),
        "layer_tflops": flops / (ms / 1000.0) / 1e12,
        # expert FFN alone, fp32 output rows (the layer writes compact rows):
        # the touched experts' FP8 weight bytes over HBM, and its FLOPs
        "ffn": {"us": ffn_s * 1e6,
                "hbm_fraction_of_weights": w_bytes / ffn_s / (peaks["hbm_gbs"] * 1e9),
                "algorithmic_bytes": ffn_bytes,
                "hbm_fraction": ffn_bytes / ffn_s / (peaks["hbm_gbs"] * 1e9),
                "tflops": flops / ffn_s / 1e12,
                "fp8_tensor_fraction": flops / ffn_s / 1e12 / (2.0 * peaks["bf16_tflops"]),
                "peak_source": peak_src + " (fp8 peak: 2 x the bf16 measured burst, the nominal ratio)"},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_eplb(args):
    """Expert placement on the loads of a routed batch (its own JSON line):
    route the workload's tokens on the GPU, count assignments per expert,
    plan global and hierarchical placements on the host (moe_eplb_plan) and
    report the planner time and the busiest/mean GPU load."""
    import torch
    import dispatch_combine_gb300 as moe
    from moe_inputs import make_layer_tensors
    torch.cuda.set_device(0)
    c = CONFIGS[args.config]
    t = make_layer_tensors(c, device="cuda", seed=0)
    ws = moe.Workspace(moe.moe_workspace_size(c.shape()))
    bias = t["bias"] if c.score == SCORE_SIGMOID_BIAS else None
    ids, _, _ = moe.moe_route(c.shape(), t["x"], t["w_r"], bias, ws)
    counts = torch.bincount(ids.flatten().long(), minlength=c.E).double().cpu().numpy()
    results = []
    for nodes, gpus, phys in ((4, 32, c.E + 32), (8, 64, c.E + 64)):
        for hier in (0, 1):
            if c.G % nodes or c.E % gpus:
                continue
            reps = max(1, args.steps)
            t0 = time.perf_counter()
            for _ in range(reps):
                slots, rep = moe.moe_eplb_plan(counts, c.G, nodes if hier else 0, gpus, phys)
            us = (time.perf_counter() - t0) / reps * 1e6
            per_gpu = [sum(counts[e] / rep[e] for e in row) for row in slots]
            results.append({"nodes": nodes, "gpus": gpus, "physical": phys,
                            "placement": "hierarchical" if hier else "global",
                            "plan_us": us,
                            "busiest_over_mean": max(per_gpu) / (sum(per_gpu) / len(per_gpu))})
    line = {"metric": "EPLB plan time (host) and busiest/mean GPU load", "impl": "gb300",
            "value": max(r["plan_us"] for r in results) if results else None, "unit": "us",
            "higher_is_better": False, "steps": args.steps, "data": "synthetic",
            "config": {"workload": workload_desc(c), "loads": "assignment counts of the routed batch"},
            "plans": results}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    c = CONFIGS[args.config]
    if args.ffn_rows:
        return run_ffn_only(args)
    if args.ffn_counts:
        return run_ffn_counts(args)
    if args.route_only:
        return run_route_only(args)
    if args.stage_only:
        return run_stage_only(args)
    if args.fp8:
        return run_fp8(args)
    if args.eplb:
        return run_eplb(args)
    if args.capacity is not None:
        return run_capacity(args)
    if args.masked:
        return run_masked(args)
    if args.impl == "reference":
        return run_reference(args, c)
    return run_gpu(args, c)


if __name__ == "__main__":
    sys.exit(main())
