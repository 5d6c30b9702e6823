"""Oracle pins for the FP8 path (e4m3 with power-of-two block scales): the
e4m3 decoder against the format's definition, the encoder against a
brute-force nearest search with ties to the even code, the block quantizers
against a numpy restatement whose scale is found by brute force over every
exponent, and the FP8 FFN against float64 matmuls of the dequantized
operands."""
import numpy as np
import pytest

import oracle
from moe_inputs import bf16_bits


def _e4m3_def(c):
    c = int(c)
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return float("nan")
    v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


FINITE = np.array([_e4m3_def(c) for c in range(127)])   # codes 0..126, increasing


def _nearest_code(x):
    a = abs(float(x))
    if a > 448.0:
        c = 126
    else:
        d = np.abs(FINITE - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if best.size == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if np.signbit(x) else 0)


def test_decoder_matches_format_definition():
    for c in range(256):
        got, want = oracle.e4m3_to_float(c), _e4m3_def(c)
        assert (np.isnan(got) and np.isnan(want)) or got == want, c
    assert oracle.e4m3_to_float(0x7e) == 448.0 and oracle.e4m3_to_float(1) == 2.0 ** -9


def test_encoder_is_nearest_with_ties_to_even():
    g = np.random.default_rng(0)
    xs = list(g.normal(0, 30, 4000)) + list(g.normal(0, 0.01, 2000))
    xs += list((FINITE[1:] + FINITE[:-1]) / 2)          # exact midpoints: ties
    xs += [0.0, -0.0, 448.0, 449.0, 470.0, 1e6, -1e6, 2.0 ** -10, 3 * 2.0 ** -10]
    for x in xs:
        x32 = float(np.float32(x))
        assert oracle.float_to_e4m3(x32) == _nearest_code(x32), x32


def _pow2_scale(amax):
    """The block scale by its definition: the smallest power of two 2^e,
    e in [-127, 127], with amax <= 448 * 2^e (brute force over every e; the
    float64 products are exact); 1 for an all-zero block."""
    amax = float(amax)
    if amax == 0.0:
        return np.float32(1.0)
    for e in range(-127, 128):
        if amax <= 448.0 * 2.0 ** e:
            return np.float32(2.0 ** e)
    raise AssertionError(amax)


def _quant_rows_np(xf32):
    """x: [rows, cols] float32 values of bf16; per-128 block power-of-two scale."""
    rows, cols = xf32.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    for r in range(rows):
        for b in range(cols // 128):
            blk = xf32[r, b * 128:(b + 1) * 128]
            sc = _pow2_scale(np.abs(blk).max())
            s[r, b] = sc
            # x / s is exact (s a power of two): the code is the nearest one
            q[r, b * 128:(b + 1) * 128] = [_nearest_code(float(v) / float(sc)) for v in blk]
    return q, s


def _bf16(a):
    import torch
    t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    return bf16_bits(t), t.float().numpy()


def test_row_quantizer_matches_numpy_restatement():
    g = np.random.default_rng(1)
    x = g.normal(0, 1, (5, 384)) * np.array([1e-3, 1.0, 50.0])[None, :].repeat(128, 1)
    x[2, 128:256] = 0.0                                   # all-zero block: scale 1
    bits, xf = _bf16(x)
    q, s = oracle.quantize_rows_fp8(bits)
    q2, s2 = _quant_rows_np(xf)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    assert s[2, 1] == 1.0 and not q[2, 128:256].any()
    # every scale is a power of two, and the largest magnitude of a nonzero
    # block lands in (224, 448]: codes 118 (224) .. 126 (448)
    m, _ = np.frexp(s)
    assert np.all(m == 0.5)
    for r in range(5):
        for b in range(3):
            blk = q[r, b * 128:(b + 1) * 128]
            if blk.any():
                assert 118 <= (blk & 0x7f).max() <= 126


def test_row_quantizer_scale_boundaries_and_clamp():
    # one block per row: amax exactly 448 * 2^k keeps e = k (the max maps to
    # 448); the next bf16 above it moves to e = k + 1; magnitudes below
    # 448 * 2^-127 (bf16 subnormals among them) clamp to 2^-127
    amaxes = [448.0, 448.0 * 2.0 ** -20, 450.0, 1.0, 2.0 ** -130, 1e-38, 3.0e38]
    x = np.zeros((len(amaxes), 128), np.float32)
    x[:, 5] = amaxes
    x[:, 9] = -0.75 * np.array(amaxes)
    bits, xf = _bf16(x)
    q, s = oracle.quantize_rows_fp8(bits)
    assert s[0, 0] == 1.0 and q[0, 5] == 126
    assert s[1, 0] == np.float32(2.0 ** -20) and q[1, 5] == 126
    assert s[2, 0] == 2.0                      # bf16(450) = 450 > 448
    assert s[3, 0] == np.float32(2.0 ** -8)   # 1 / 2^-8 = 256 <= 448 < 512
    assert s[4, 0] == np.float32(2.0 ** -127) and s[5, 0] == np.float32(2.0 ** -127)
    assert s[6, 0] == np.float32(2.0 ** 120)
    for r, a in enumerate(xf[:, 5]):
        assert s[r, 0] == _pow2_scale(a)
        assert q[r, 9] == _nearest_code(float(xf[r, 9]) / float(s[r, 0]))


def test_block_quantizer_is_the_row_quantizer_on_128x128_blocks():
    g = np.random.default_rng(2)
    w = g.normal(0, 0.02, (2, 256, 384))
    bits, wf = _bf16(w)
    q, s = oracle.quantize_blocks_fp8(bits)
    assert q.shape == (2, 256, 384) and s.shape == (2, 2, 3)
    for m in range(2):
        for i in range(2):
            for j in range(3):
                blk = wf[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                sc = _pow2_scale(np.abs(blk).max())
                assert s[m, i, j] == sc
                codes = np.array([[_nearest_code(float(v) / float(sc)) for v in row]
                                  for row in blk])
                assert np.array_equal(q[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128], codes)


def test_fp8_ffn_matches_float64_of_dequantized_operands():
    g = np.random.default_rng(3)
    E, d, inter, n = 2, 256, 128, 6
    xb, xf = _bf16(g.normal(0, 1, (n, d)))
    wgb, _ = _bf16(g.normal(0, 1, (E, 2 * inter, d)) / d ** 0.5)
    wdb, _ = _bf16(g.normal(0, 1, (E, d, inter)) / inter ** 0.5)
    xq, xs = oracle.quantize_rows_fp8(xb)
    gq, gs = oracle.quantize_blocks_fp8(wgb)
    dq, ds = oracle.quantize_blocks_fp8(wdb)
    row_e = np.array([0, 1, 1, 0, 1, 0], np.int32)
    y, h = oracle.expert_ffn_rows_fp8(xq, xs, row_e, gq, gs, dq, ds, return_h=True)
    dec = np.vectorize(_e4m3_def)
    xd = dec(xq) * np.repeat(xs, 128, 1)
    gd = dec(gq) * np.repeat(np.repeat(gs, 128, 1), 128, 2)
    dd = dec(dq) * np.repeat(np.repeat(ds, 128, 1), 128, 2)
    for r in range(n):
        e = row_e[r]
        gu = gd[e] @ xd[r]
        hv = gu[:inter] / (1 + np.exp(-gu[:inter])) * gu[inter:]
        hb, hf = _bf16(hv[None, :])
        assert np.array_equal(h[r], hf[0])
        hq, hs = _quant_rows_np(hf)
        hdq = dec(hq[0]) * np.repeat(hs[0], 128)
        want = dd[e] @ hdq
        assert np.allclose(y[r], want, rtol=1e-6, atol=1e-7)
