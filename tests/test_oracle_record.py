"""Pins for the expert record layout and the block quantiser (CPU only)."""
import numpy as np
import pytest

from conftest import golden
from oracle import oracle as O

G = {r[0]: float(r[1]) for r in golden("record_bytes.txt")}


def test_qwen_record_byte_count_from_page():
    assert O.record_bytes(2560, 640, O.FMT_NVFP4) == int(G["qwen_record"])
    assert O.record_bytes(2560, 640, O.FMT_NVFP4) == int(G["qwen_record_pages_4k"]) * 4096


def test_qwen_record_parts_are_4k_aligned():
    lay = O.record_layout(2560, 640, O.FMT_NVFP4)
    for name in ("gate", "up", "down", "gate_s", "up_s", "down_s", "total"):
        assert lay[name] % 4096 == 0, name
    # order gate | up | down | scales, as the page lists it
    assert lay["gate"] < lay["up"] < lay["down"] < lay["gate_s"] < lay["up_s"] < lay["down_s"]


def test_deepseek_record_from_page():
    lay = O.record_layout(4096, 2880, O.FMT_MXFP4)
    codes_mb = lay["gate_s"] / 1e6
    scales_mb = (lay["total"] - lay["gate_s"]) / 1e6
    assert round(codes_mb, 1) == G["deepseek_codes_mb"]
    assert round(scales_mb, 1) == G["deepseek_scales_mb"]
    assert round(lay["total"] / 2 ** 20, 2) == G["deepseek_record_mib"]


def test_bytes_per_token_from_pages():
    q = O.expert_bytes_per_token(48, 10, 2560, 640, O.FMT_NVFP4)
    assert round(q / 1e9, 2) == G["qwen_token_bytes_gb"]
    d = O.expert_bytes_per_token(40, 6, 4096, 2880, O.FMT_MXFP4)
    assert round(d / 2 ** 30, 1) == G["deepseek_token_gib"]


def _blocks(rng, rows, K, std=0.02):
    return (rng.standard_normal((rows, K)) * std).astype(np.float32)


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_MXFP4])
def test_quantiser_picks_nearest_grid_point(fmt):
    rng = np.random.default_rng(3 + fmt)
    W = _blocks(rng, 16, 128)
    W[3, :] = 0.0                      # all-zero blocks
    W[4, :32] = np.float32(1e-8)       # tiny: NVFP4 scale underflows to 0
    W[5, :] *= 1000                    # large
    codes, scales = O.quantize_matrix(W, fmt)
    Gs = O.block_size(fmt)
    sdec = O.e4m3_decode(scales) if fmt == O.FMT_NVFP4 else O.ue8m0_decode(scales)
    el = np.empty(W.shape, dtype=np.uint8)
    el[:, 0::2] = codes & 0xF
    el[:, 1::2] = codes >> 4
    allv = O.e2m1_decode(np.arange(8))
    for r in range(W.shape[0]):
        for c in range(W.shape[1]):
            s = sdec[r, c // Gs]
            v = O.e2m1_decode(el[r, c])
            if s == 0:
                assert el[r, c] == 0
                continue
            # brute force: |v*s - x| is minimal over the 8 magnitudes (with
            # the x/s ratio clamped to the top of the grid)
            if fmt == O.FMT_NVFP4:
                ratio = float(np.float32(W[r, c]) / np.float32(s))
            else:
                ratio = float(np.float32(W[r, c]) * np.float32(1.0 / s))
            target = min(abs(ratio), 6.0)
            assert abs(abs(v) - target) == np.min(np.abs(allv - target))
            if v != 0 or el[r, c] == 8:
                assert np.signbit(v) == np.signbit(np.float32(W[r, c]))


def test_nvfp4_scale_is_rounded_amax_over_six():
    rng = np.random.default_rng(7)
    W = _blocks(rng, 8, 64)
    _, scales = O.quantize_matrix(W, O.FMT_NVFP4)
    amax = np.abs(W.reshape(8, 4, 16)).max(axis=2)
    allv = O.e4m3_decode(np.arange(127))
    for r in range(8):
        for b in range(4):
            want = np.float32(amax[r, b]) / np.float32(6.0)
            d = np.abs(allv - want)
            assert abs(O.e4m3_decode(scales[r, b]) - want) == d.min()


def test_mxfp4_scale_is_smallest_power_of_two_that_fits():
    rng = np.random.default_rng(8)
    W = _blocks(rng, 8, 128, std=3.0)
    W[0, :32] = 6.0 * 2.0 ** -3   # exactly representable amax: E = -3
    _, scales = O.quantize_matrix(W, O.FMT_MXFP4)
    amax = np.abs(W.reshape(8, 4, 32)).max(axis=2).astype(np.float64)
    E = scales.astype(np.int64) - 127
    assert np.all(6.0 * np.ldexp(1.0, E) >= amax)
    assert np.all(6.0 * np.ldexp(1.0, E - 1) < amax)
    assert scales[0, 0] == 127 - 3


def test_nibble_order_low_nibble_first():
    W = np.zeros((1, 32), dtype=np.float32)
    W[0, 0] = 6 * 0.5    # element 0 -> code for 3.0 after scaling by amax/6
    W[0, 1] = 6 * 1.0    # element 1 -> 6.0 (the block max)
    codes, scales = O.quantize_matrix(W, O.FMT_NVFP4)
    assert O.e4m3_decode(scales[0, 0]) == 1.0
    assert codes[0, 0] == (5 | (7 << 4))


def test_pack_unpack_roundtrip_equals_dequantised_parts():
    rng = np.random.default_rng(9)
    H, I = 64, 32
    gate, up, down = _blocks(rng, I, H), _blocks(rng, I, H), _blocks(rng, H, I)
    for fmt in (O.FMT_NVFP4, O.FMT_MXFP4):
        rec = O.pack_expert(gate, up, down, fmt)
        assert rec.size == O.record_bytes(H, I, fmt)
        Wg, Wu, Wd = O.unpack_expert(rec, H, I, fmt)
        for W, D in ((gate, Wg), (up, Wu), (down, Wd)):
            c, s = O.quantize_matrix(W, fmt)
            assert np.array_equal(O.dequantize_matrix(c, s, W.shape[1], fmt), D)
            # error bound: half the coarsest grid step (2) times the scale, or
            # the clipped part above 6*s when the scale itself rounded down
            Gs = O.block_size(fmt)
            sdec = O.e4m3_decode(s) if fmt == O.FMT_NVFP4 else O.ue8m0_decode(s)
            amax = np.abs(W.reshape(W.shape[0], -1, Gs)).max(axis=2)
            bound = np.maximum(sdec, amax - 6 * sdec)
            assert np.all(np.abs(D - W) <= np.repeat(bound, Gs, axis=1) * (1 + 1e-9))
