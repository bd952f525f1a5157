"""Pins of the oracle's FP4/FP8 formats (DeepSeek-V4.1-Flash walkthrough 1.(5).4
"FP4 Main KV Cache"; release summary "CSA2").  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines, parse_float


def test_code_values_match_golden_table():
    n = 0
    for line in golden_lines("e4m3_e2m1_values.txt"):
        kind, code, val = line.split()
        code = int(code, 0)
        got = oracle.e2m1_value(code) if kind == "e2m1" else oracle.e4m3_value(code)
        if val == "nan":
            assert math.isnan(got)
        else:
            want = float(val)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (kind, code)
        n += 1
    assert n > 20


def test_e2m1_magnitudes_are_the_eight_point_grid():
    assert [oracle.e2m1_value(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_decode_matches_torch_for_every_byte():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    for b in range(256):
        got = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b], b


def _e4m3_probe_points():
    """Every finite E4M3 value, every midpoint between neighbours, and the fp32
    numbers just below and above each midpoint."""
    vals = sorted({oracle.e4m3_value(b) for b in range(0x7F)})
    pts = []
    for a, b in zip(vals, vals[1:]):
        mid = np.float32((a + b) / 2)              # midpoints have <= 5 bits: exact
        pts += [a, b, mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1000))]
    return np.array(pts, dtype=np.float32)


def test_e4m3_encode_rne_matches_torch_cast_at_codes_midpoints_and_neighbours():
    # torch casts fp32 -> e4m3 with round-to-nearest-even; feed it fp32 values
    # (its fp64 path first rounds to fp32, a double rounding the oracle avoids)
    pts = _e4m3_probe_points()
    pts = np.concatenate([pts, -pts])
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in pts])
    assert (got == ref).all()


def test_e4m3_encode_rounds_the_exact_value_not_an_fp32_copy():
    # 2^-10 is the midpoint of 0 and 2^-9: exactly on it -> even (0), a hair above -> 2^-9
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(float.fromhex("0x1.0000000000001p-10")) == 0x01


def test_e4m3_encode_saturates_at_448():
    for v in (448.0, 449.0, 464.0, 480.0, 1e6, math.inf):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_e2m1_encode_ties_go_to_even_code():
    # midpoints of the grid and the code they round to
    for q, code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert oracle.e2m1_encode_magnitude(q) == code
        below = oracle.e2m1_encode_magnitude(np.nextafter(q, 0))
        above = oracle.e2m1_encode_magnitude(np.nextafter(q, 10))
        assert oracle.e2m1_value(below) < q < oracle.e2m1_value(above)
    assert oracle.e2m1_encode_magnitude(100.0) == 7
    assert oracle.e2m1_encode_magnitude(0.0) == 0


def test_row_is_288_bytes_for_512_channels():
    # 512 four-bit codes + 512/16 one-byte scales
    assert oracle.fp4_row_bytes(512) == 288


def _golden_blocks():
    out = []
    for line in golden_lines("fp4_blocks.txt"):
        vals, scale, codes = (p.strip() for p in line.split("|"))
        x = np.array([parse_float(t) for t in vals.split()], dtype=np.float32)
        assert x.size == 16
        out.append((x, int(scale, 16), bytes(int(t, 16) for t in codes.split())))
    return out


def test_quantise_golden_blocks():
    blocks = _golden_blocks()
    assert len(blocks) >= 7
    # place each block at a different position of a 512-channel row
    for pos in (0, 5, 31):
        for x, scale, codes in blocks:
            row = np.zeros((1, 512), np.float32)
            row[0, 16 * pos:16 * pos + 16] = x
            q = oracle.quantize_kv_fp4(row)[0]
            assert q[256 + pos] == scale
            assert bytes(q[8 * pos:8 * pos + 8]) == codes
            # the other blocks are all-zero: scale 0, codes 0
            others = [b for b in range(32) if b != pos]
            assert (q[256 + np.array(others)] == 0).all()


def test_largest_magnitude_2688_round_trips():
    row = np.zeros((1, 512), np.float32)
    row[0, 0] = 2688.0
    row[0, 17] = -2688.0
    d = oracle.dequantize_kv_fp4(oracle.quantize_kv_fp4(row), 512)
    assert d[0, 0] == 2688.0 and d[0, 17] == -2688.0
    assert np.abs(d).max() == 448 * 6


def test_each_code_is_the_nearest_grid_point_of_the_exact_quotient():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 512)) * rng.choice([1e-3, 0.1, 1, 10, 100], (64, 1))).astype(np.float32)
    q = oracle.quantize_kv_fp4(x)
    scales = np.array([[oracle.e4m3_value(b) for b in row[256:]] for row in q])  # [64][32]
    s = np.repeat(scales, 16, axis=1)
    codes = np.empty((64, 512), np.int64)
    codes[:, 0::2] = q[:, :256] & 15
    codes[:, 1::2] = q[:, :256] >> 4
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s > 0, np.abs(x.astype(np.float64)) / np.where(s > 0, s, 1), 0.0)
    dist = np.abs(ratio[..., None] - grid)                  # distance to every grid point
    chosen = dist[np.arange(64)[:, None], np.arange(512)[None], codes & 7]
    assert (chosen <= dist.min(-1) + 0).all()
    assert ((codes >> 3) == np.signbit(x)).all()
    # scale is the E4M3 value nearest absmax/6
    amax = np.abs(x.reshape(64, 32, 16)).max(-1).astype(np.float64)
    e4 = np.array([oracle.e4m3_value(b) for b in range(0x7F)])
    best = np.abs(amax[..., None] / 6 - e4).min(-1)
    assert (np.abs(amax / 6 - scales) == best).all()


def test_quantise_of_dequantised_row_is_identity():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 512)).astype(np.float32)
    q = oracle.quantize_kv_fp4(x)
    d = oracle.dequantize_kv_fp4(q, 512).astype(np.float32)   # exact in fp32
    assert (oracle.quantize_kv_fp4(d) == q).all()


def test_dequantise_is_code_value_times_scale():
    row = np.zeros(288, np.uint8)
    row[:8] = np.arange(16, dtype=np.uint8)[0::2] | (np.arange(16, dtype=np.uint8)[1::2] << 4)
    row[256] = 0x3C  # 1.5
    d = oracle.dequantize_kv_fp4(row[None], 512)[0]
    assert list(d[:16]) == [1.5 * v for v in (0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6)]
    assert (d[16:] == 0).all()
