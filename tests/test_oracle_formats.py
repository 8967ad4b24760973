"""Pins for the oracle's number formats (CPU only)."""
import math

import numpy as np
import pytest
import torch

from conftest import golden
from oracle import oracle as O


def test_e2m1_decode_matches_hand_worked_table():
    rows = golden("e2m1_codes.txt")
    assert len(rows) == 16
    codes = np.array([int(r[0]) for r in rows])
    want = np.array([float(r[1]) for r in rows])
    got = O.e2m1_decode(codes)
    assert np.array_equal(got, want)
    # signed zero is kept as a distinct code
    assert math.copysign(1.0, got[8]) == -1.0


def test_e2m1_encode_hand_worked_rounding():
    for v, code in golden("e2m1_rounding.txt"):
        assert int(O.e2m1_encode(np.float32(float(v)))) == int(code), v


def test_e2m1_encode_is_nearest_by_brute_force():
    # dense grid of float32 inputs incl. every midpoint and its neighbours
    grid = O.e2m1_decode(np.arange(8))
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([np.linspace(-8, 8, 4001), mids, -mids,
                          np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.nextafter(mids.astype(np.float32), np.float32(9))]).astype(np.float32)
    codes = O.e2m1_encode(pts)
    vals = O.e2m1_decode(codes)
    allv = O.e2m1_decode(np.arange(16))
    for p, c, v in zip(pts.astype(np.float64), codes, vals):
        d = np.abs(allv - min(max(p, -6.0), 6.0))
        best = d.min()
        assert abs(v - min(max(p, -6.0), 6.0)) == best
        if np.count_nonzero(d == best) > 1 and best > 0:  # a true tie: even mantissa
            assert (c & 1) == 0


def test_e4m3_decode_matches_torch_float8_for_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).float().double().numpy()
    got = O.e4m3_decode(b)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # hand-worked anchors: smallest subnormal, smallest normal, one, largest
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x38) == 1.0
    assert O.e4m3_decode(0x7E) == 448.0


def test_e4m3_encode_matches_torch_rounding_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 0.01,
                        rng.standard_normal(20000) * 10,
                        rng.uniform(0, 448, 20000),
                        O.e4m3_decode(np.arange(1, 126)) * 1.0625,
                        (O.e4m3_decode(np.arange(0, 126)) + O.e4m3_decode(np.arange(1, 127))) / 2]
                       ).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v)
    # torch keeps -0 for negative underflow too; compare bytes exactly
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates():
    assert int(O.e4m3_encode(np.float32(1e6))) == 0x7E
    assert int(O.e4m3_encode(np.float32(460.0))) == 0x7E
    assert int(O.e4m3_encode(np.float32(-1e6))) == 0xFE


def test_ue8m0_decode():
    assert O.ue8m0_decode(127) == 1.0
    assert O.ue8m0_decode(0) == 2.0 ** -127
    assert O.ue8m0_decode(254) == 2.0 ** 127
    assert np.isnan(O.ue8m0_decode(255))


def test_bf16_round_matches_torch_on_float32():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(50000), rng.standard_normal(1000) * 1e-39,
                        rng.standard_normal(1000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.bf16_round_bits(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_round_single_rounding_from_float64():
    # 1 + 2^-8 is the exact midpoint between 1 and 1 + 2^-7: ties to even -> 1;
    # one float64 ulp above it must round up (a float32 detour would lose it).
    assert O.bf16_round(1.0 + 2.0 ** -8) == 1.0
    assert O.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
