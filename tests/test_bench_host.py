"""Host-side logic of bench.py (no GPU): the max-over-ranks timing reduction
with two gloo ranks, whole-job throughput, clock parsing, and the JSON line of
the reference arm (the CPU oracle) on the tiny workload."""
import contextlib
import io
import json
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # each replica reports its own elapsed time; the job time is the max
    t = bench.max_over_ranks(10.0 + rank * 5.0, world, "cpu")
    v = bench.job_value(tokens_per_rank=1000, world=world, seconds=t / 1000.0, steps=4)
    dist.destroy_process_group()
    q.put((rank, t, v))


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == 15.0
        # 2 ranks x 1000 tokens x 4 steps in 15 ms
        assert v == pytest.approx(2 * 1000 * 4 / 0.015)


def test_job_value_single():
    assert bench.job_value(2048, 1, 0.5, 10) == pytest.approx(40960.0)


def test_clock_parsing():
    cs = bench.ClockSampler(0)
    cs.proc = None
    assert cs.stop()["reasons"] == ["nvidia-smi unavailable"]

    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs = bench.ClockSampler(0)
    cs.proc = _P()
    cs.t_start, cs.t_end = 100.0, 101.0
    cs.lines = [
        (99.0, "300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (100.2, "1900, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (100.6, "1950, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (100.9, "2000, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
    ]
    r = cs.stop()
    assert r["sm_mhz"] == 1950.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_reference_arm_json_line(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2",
                         "--warmup", "1", "--ref-step-s", "0.2"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_total_time_is_bounded(monkeypatch):
    # however many steps are asked for, the token sample per step shrinks so
    # that all steps together take about --ref-total-s
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny", "--steps", "50",
                         "--warmup", "1", "--ref-total-s", "0.5"])
    assert rc == 0
    d = json.loads([ln for ln in buf.getvalue().splitlines() if ln.strip()][0])
    assert d["steps"] == 50
    assert d["ms_per_step"] * d["steps"] / 1000.0 < 2.0


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1"])
    assert rc == 0 and buf.getvalue() == ""


def test_tensor_peak_follows_timed_region_length():
    peaks = {"hbm_gbs": 6784.5, "bf16_tflops": 1854.8, "bf16_tflops_sustained": 1699.2}
    p, src = bench.tensor_peak(peaks, "measured", 0.17)
    assert p == 1854.8 and "burst" in src
    p, src = bench.tensor_peak(peaks, "measured", 5.2)
    assert p == 1699.2 and "sustained" in src


def test_layer_bytes_prefill():
    c = bench.CONFIGS["prefill"]
    sb = bench.stage_bytes(c)
    # weights of 100 touched experts (88.08 MB each) plus the bandwidth stages
    assert bench.layer_bytes(c, 100) == sum(sb.values()) + 100 * 3 * 7168 * 2048 * 2


def test_default_line_is_prefill_with_decode_nested():
    a = bench.parse_args([])
    assert a.config == "prefill" and a.also == "decode"
    a = bench.parse_args(["--config", "few_large"])
    assert a.also == ""
