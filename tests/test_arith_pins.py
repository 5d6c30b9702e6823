"""Closed-form arithmetic the pages print, used for the algorithmic byte and
FLOP counts of the benchmark (no GPU)."""
import math

from moe_inputs import CONFIGS
import bench


def test_dispatch_volume_example_first_page():
    # "第十五章" section 3.4 worked example: 8-rank EP group, T=4096 tokens,
    # top-2, H=8192, bf16 (b=2).
    T, k, H, b, P = 4096, 2, 8192, 2, 8
    MiB = 2 ** 20
    assert T * k * H * b == 128 * MiB                      # dispatch T*k*H*b
    assert T * k * H * b * (P - 1) // P == 112 * MiB       # remote share 7/8
    assert 2 * T * k * H * b * (P - 1) // P == 224 * MiB   # dispatch + combine
    assert 2 * T * k * H * b * (P - 1) // P // P == 28 * MiB  # per rank
    assert T * k * H * b // P ** 2 == 2 * MiB              # per source-dest pair
    # top-16 instead of top-2: x8 -> 1.75 GiB remote dispatch + combine
    assert 2 * T * 16 * H * b * (P - 1) // P == int(1.75 * 2 ** 30)


def test_activation_buffer_size_second_page():
    # MoE-TP/EP comparison: at B=512 the [B*k, d] buffer is about 59 MB
    # (k=8, d=7168, bf16).
    assert round(512 * 8 * 7168 * 2 / 1e6) == 59


def test_tokens_per_expert_formulas():
    # M_e = B_local * P * k / E: B_local=128, P=32, k=8, E=256 -> 128
    assert 128 * 32 * 8 // 256 == 128
    # "第十五章" 4.1: 16T/896 = T/56
    assert 16 * 5600 / 896 == 5600 / 56 == 100
    # capacity C = ceil(c*T*k/E): T=5600, k=16, E=896 -> 100, c=1.2 -> 120
    assert math.ceil(1.0 * 5600 * 16 / 896) == 100
    assert math.ceil(1.2 * 5600 * 16 / 896) == 120


def test_expert_weight_bytes_and_flops():
    c = CONFIGS["decode"]
    # 3 * d * inter parameters per expert (gate, up, down) = 44 M -> 88 MB bf16
    assert 3 * c.d * c.inter == 44040192
    assert bench.expert_weight_bytes(c) == 3 * c.d * c.inter * 2
    # FLOPs per routed row: 2*d*2*inter + 2*inter*d = 6*d*inter
    assert bench.ffn_flops_per_row(c) == 6 * c.d * c.inter
    # masked slice: 8 experts x 7168 x 4096 gate_up (the second page's 235 MB
    # at 1 byte per weight) = 469.8 MB at bf16
    assert 8 * 7168 * 4096 * 2 == 469762048


def test_stage_algorithmic_bytes():
    c = CONFIGS["decode"]
    T, d, E, k = c.T, c.d, c.E, c.k
    b = bench.stage_bytes(c)
    assert b["router"] == T * d * 2 + d * E * 2 + T * k * 8
    assert b["dispatch"] == T * k * 4 + T * d * 2 + T * k * d * 2 + T * k * 8
    assert b["combine"] == T * k * d * 4 + T * k * 8 + T * d * 2
