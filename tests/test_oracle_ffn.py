"""Pins for the oracle's expert FFN, bucketing, RMS chaining and FP8 GEMV
(CPU only)."""
import math
import struct

import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import synth
from conftest import golden
from oracle import oracle as O

E2M1 = {int(r[0]): float(r[1]) for r in golden("e2m1_codes.txt")}


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _e4m3(b):
    return float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def _brute_dequant(rec, off, soff, rows, K, fmt):
    """Element-by-element decode straight from the record bytes."""
    Gs = 16 if fmt == O.FMT_NVFP4 else 32
    out = [[0.0] * K for _ in range(rows)]
    for r in range(rows):
        for c in range(K):
            byte = int(rec[off + (r * K + c) // 2])
            code = byte & 0xF if c % 2 == 0 else byte >> 4
            sb = int(rec[soff + (r * K + c) // Gs])
            s = _e4m3(sb) if fmt == O.FMT_NVFP4 else 2.0 ** (sb - 127)
            out[r][c] = E2M1[code] * s
    return out


def _brute_layer(xb, idx, w, recs, H, I, fmt):
    lay = O.record_layout(H, I, fmt)
    x = [[float(v) for v in row] for row in O.bf16_bits_to_f32(xb)]
    T, k = idx.shape
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            rec = recs[int(idx[t, j])]
            Wg = _brute_dequant(rec, lay["gate"], lay["gate_s"], I, H, fmt)
            Wu = _brute_dequant(rec, lay["up"], lay["up_s"], I, H, fmt)
            Wd = _brute_dequant(rec, lay["down"], lay["down_s"], H, I, fmt)
            g = [math.fsum(Wg[i][h] * x[t][h] for h in range(H)) for i in range(I)]
            u = [math.fsum(Wu[i][h] * x[t][h] for h in range(H)) for i in range(I)]
            hh = [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(I)]
            for n in range(H):
                y[t][n] += w[t, j] * math.fsum(Wd[n][i] * hh[i] for i in range(I))
    return np.array(y)


def _pool(E, H, I, fmt, seed):
    recs = []
    for e in range(E):
        g, u, d = synth.expert_weights(H, I, seed + e, std=0.5)
        recs.append(O.pack_expert(g.numpy(), u.numpy(), d.numpy(), fmt))
    return recs


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_MXFP4])
def test_decode_layer_matches_brute_force(fmt):
    H, I, E, k, T = 32, 32, 6, 3, 2
    recs = _pool(E, H, I, fmt, 100)
    xb = _bits(synth.activations(T, H, 21))
    idx = np.array([[4, 0, 2], [1, 5, 3]], dtype=np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.6, 0.25, 0.15]])
    got = O.moe_layer_decode(xb, idx, w, recs, H, I, fmt)
    want = _brute_layer(xb, idx, w, recs, H, I, fmt)
    assert O.rel_l2(got, want) < 1e-7


def test_pointer_table_permutation_invariance_and_zero_record():
    H, I, E = 64, 32, 5
    recs = _pool(E, H, I, O.FMT_NVFP4, 200)
    xb = _bits(synth.activations(3, H, 22))
    idx = np.array([[0, 1], [2, 3], [4, 0]], dtype=np.int32)
    w = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1]])
    base = O.moe_layer_decode(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    perm = [3, 0, 4, 1, 2]                       # slot s holds expert perm[s]
    table = {perm[s]: recs[perm[s]] for s in range(E)}
    assert np.array_equal(O.moe_layer_decode(xb, idx, w, table, H, I, O.FMT_NVFP4), base)
    zero = dict(enumerate(recs))
    zero[4] = np.zeros_like(recs[4])
    y = O.moe_layer_decode(xb, idx, w, zero, H, I, O.FMT_NVFP4)
    only0 = O.moe_layer_decode(xb[2:3], np.array([[0]]), np.array([[0.1]]), recs, H, I, O.FMT_NVFP4)
    assert np.allclose(y[2], only0[0], rtol=1e-6, atol=0)


def test_k1_weight1_is_single_expert_ffn():
    H, I = 64, 32
    g, u, d = synth.expert_weights(H, I, 300, std=0.5)
    rec = O.pack_expert(g.numpy(), u.numpy(), d.numpy(), O.FMT_NVFP4)
    Wg, Wu, Wd = O.unpack_expert(rec, H, I, O.FMT_NVFP4)
    xb = _bits(synth.activations(1, H, 23))
    x = O.bf16_bits_to_f32(xb)[0].astype(np.float64)
    gg, uu = Wg @ x, Wu @ x
    want = Wd @ (gg * uu * scipy_expit(gg))
    y = O.moe_layer_decode(xb, np.array([[0]]), np.array([[1.0]]), [rec], H, I, O.FMT_NVFP4)
    assert np.allclose(y[0], want, rtol=1e-6, atol=1e-12)


def scipy_expit(v):
    import scipy.special
    return scipy.special.expit(v)


def _controls_setup():
    H, I, E = 64, 32, 4
    recs = _pool(E, H, I, O.FMT_NVFP4, 400)
    xb = _bits(synth.activations(2, H, 24))
    idx = np.array([[0, 1], [2, 3]], dtype=np.int32)
    w = np.array([[0.6, 0.4], [0.8, 0.2]])
    return H, I, recs, xb, idx, w


def test_negative_control_nibble_swap_breaks_output():
    H, I, recs, xb, idx, w = _controls_setup()
    base = O.moe_layer_decode(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    lay = O.record_layout(H, I, O.FMT_NVFP4)
    bad = []
    for r in recs:
        r = r.copy()
        c = r[: lay["gate_s"]]
        r[: lay["gate_s"]] = ((c & 0xF) << 4) | (c >> 4)
        bad.append(r)
    assert O.rel_l2(O.moe_layer_decode(xb, idx, w, bad, H, I, O.FMT_NVFP4), base) > 0.1


def test_negative_control_gate_up_swap_breaks_output():
    H, I, recs, xb, idx, w = _controls_setup()
    base = O.moe_layer_decode(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    lay = O.record_layout(H, I, O.FMT_NVFP4)
    bad = []
    for r in recs:
        r = r.copy()
        a = r[lay["gate"]:lay["up"]].copy()
        r[lay["gate"]:lay["up"]] = r[lay["up"]:lay["down"]]
        r[lay["up"]:lay["down"]] = a
        bad.append(r)
    assert O.rel_l2(O.moe_layer_decode(xb, idx, w, bad, H, I, O.FMT_NVFP4), base) > 0.1


def test_negative_control_wrong_scale_format_breaks_output():
    H, I, recs, xb, idx, w = _controls_setup()
    base = O.moe_layer_decode(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    Wg, Wu, Wd = O.unpack_expert(recs[0], H, I, O.FMT_NVFP4)
    lay = O.record_layout(H, I, O.FMT_NVFP4)
    c = recs[0][lay["gate"]:lay["up"]].reshape(I, H // 2)
    s = recs[0][lay["gate_s"]:lay["up_s"]].reshape(I, H // 16)
    as_ue8m0 = O.e2m1_decode(np.stack([c & 0xF, c >> 4], -1).reshape(I, H)) * \
        np.repeat(O.ue8m0_decode(s), 16, axis=1)
    assert O.rel_l2(as_ue8m0, Wg) > 0.5


def test_grouped_k1_close_to_decode_and_by_expert_equal():
    H, I, E = 64, 64, 4
    recs = _pool(E, H, I, O.FMT_NVFP4, 500)
    xb = _bits(synth.activations(6, H, 25))
    idx = np.array([[0], [1], [2], [3], [0], [1]], dtype=np.int32)
    w = np.ones((6, 1))
    dec = O.moe_layer_decode(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    grp = O.moe_layer_grouped(xb, idx, w, recs, H, I, O.FMT_NVFP4)
    assert O.rel_l2(grp, dec) < 2e-3
    assert O.rel_l2(grp, dec) > 0          # the BF16 rounding of h is visible
    idx2 = np.array([[0, 1], [1, 2], [2, 3], [3, 0], [0, 2], [1, 3]], dtype=np.int32)
    w2 = np.full((6, 2), 0.5)
    a = O.moe_layer_grouped(xb, idx2, w2, recs, H, I, O.FMT_NVFP4)
    b = O.moe_layer_grouped_by_expert(xb, idx2, w2, recs, H, I, O.FMT_NVFP4)
    assert O.rel_l2(a, b) < 1e-6


def test_expert_restriction_sums_to_the_whole_layer():
    # the parts restricted to disjoint expert sets add up to the full layer,
    # and the worker-split helper the full-size GPU tests use agrees with the
    # serial oracle
    from helpers import oracle_layer_split
    H, I, E, k, T = 64, 32, 8, 3, 5
    recs = dict(enumerate(_pool(E, H, I, O.FMT_NVFP4, 600)))
    xb = _bits(synth.activations(T, H, 61))
    rng = np.random.default_rng(62)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T)
    for fn in ("moe_layer_decode", "moe_layer_grouped_by_expert"):
        whole = getattr(O, fn)(xb, idx, w, recs, H, I, O.FMT_NVFP4)
        parts = sum(getattr(O, fn)(xb, idx, w, recs, H, I, O.FMT_NVFP4, experts=g).astype(np.float64)
                    for g in ([0, 3, 5], [1, 2], [4, 6, 7]))
        assert O.rel_l2(parts, whole) < 1e-7
        assert not np.any(getattr(O, fn)(xb, idx, w, recs, H, I, O.FMT_NVFP4, experts=[]))
        split = oracle_layer_split(fn, xb, idx, w, recs, H, I, O.FMT_NVFP4, parts=3)
        assert O.rel_l2(split, whole) < 1e-7


def test_bucketing_brute_force():
    rng = np.random.default_rng(9)
    T, k, E = 37, 4, 11
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, pairs = O.bucket_by_expert(idx, E)
    want = []
    for e in range(E):
        grp = [t * k + j for t in range(T) for j in range(k) if idx[t, j] == e]
        assert counts[e] == len(grp)
        assert offsets[e] == len(want)
        want += grp
    assert offsets[E] == T * k
    assert list(pairs) == want


def _f32(v):
    """A Python float rounded to FP32 (round to nearest even)."""
    return struct.unpack("<f", struct.pack("<f", v))[0]


def _bf16_bits_of_f32(v):
    """FP32 value -> BF16 bit pattern, ties to even, from the FP32 bits."""
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF


def _rms_rows_brute_force(y, eps, nparts=256, stride=True, tree="halves"):
    """The fixed FP32 order of the RMS chaining written out with Python floats
    rounded to FP32 after every operation.  The default arguments are the
    documented reading; the others plant plausible mistakes (a contiguous split
    instead of a strided one, another partial count, adjacent pairing in the
    tree) so that a test can show the pin catches them."""
    T, H = y.shape
    sums, rs, xs = [], [], []
    for t in range(T):
        row = [float(v) for v in y[t]]
        part = [0.0] * nparts
        if stride:
            for i in range(H):
                part[i % nparts] = _f32(part[i % nparts] + _f32(row[i] * row[i]))
        else:
            per = -(-H // nparts)
            for i in range(H):
                part[i // per] = _f32(part[i // per] + _f32(row[i] * row[i]))
        w = nparts // 2
        while w >= 1:
            if tree == "halves":
                part = [_f32(part[j] + part[j + w]) if j < w else part[j] for j in range(nparts)]
            else:  # adjacent pairs, then the survivors packed to the front
                part = [_f32(part[2 * j] + part[2 * j + 1]) for j in range(w)] + [0.0] * (nparts - w)
            w //= 2
        mean = _f32(part[0] / float(H))
        r = _f32(1.0 / _f32(math.sqrt(_f32(mean + _f32(eps)))))
        sums.append(part[0])
        rs.append(r)
        xs.append([_bf16_bits_of_f32(_f32(v * r)) for v in row])
    return (np.array(sums, dtype=np.float32), np.array(rs, dtype=np.float32),
            np.array(xs, dtype=np.uint16))


def _rms_inputs():
    # widths of the Qwen- and DeepSeek-shaped layers and a ragged one (not a
    # multiple of 256); magnitudes spread over several binades so that the
    # order of the FP32 additions shows in the last bits of the sum
    rng = np.random.default_rng(31)
    out = []
    for H in (2560, 4096, 1000):
        y = rng.standard_normal((6, H)) * np.exp2(rng.integers(-1, 2, (6, H)))
        out.append(y.astype(np.float32))
    return out


def test_rms_fixed_order_brute_force():
    for y in _rms_inputs():
        s_want, r_want, x_want = _rms_rows_brute_force(y, 1e-6)
        assert np.array_equal(O.rms_sumsq_fixed_order(y).view(np.uint32), s_want.view(np.uint32))
        assert np.array_equal(O.rms_inv_fixed_order(y, 1e-6).view(np.uint32), r_want.view(np.uint32))
        assert np.array_equal(O.rmsnorm_bf16(y, 1e-6), x_want)


def test_rms_pin_catches_planted_order_mistakes():
    # each planted order gives another FP32 sum of squares on at least one
    # row, so the brute-force pin above would fail an oracle that used it
    ys = _rms_inputs()
    for kw in ({"stride": False}, {"nparts": 128}, {"nparts": 512}, {"tree": "adjacent"}):
        differs = 0
        for y in ys:
            s_bad, _, _ = _rms_rows_brute_force(y, 1e-6, **kw)
            differs += int(np.sum(O.rms_sumsq_fixed_order(y).view(np.uint32) != s_bad.view(np.uint32)))
        assert differs >= 2, kw


def test_rmsnorm_within_one_bf16_unit_of_the_definition():
    # the fixed FP32 order against the float64 definition: the FP32 factor r
    # is within a few FP32 units of the exact one, so x moves across a BF16
    # rounding point only rarely, and then by one unit
    rng = np.random.default_rng(10)
    for H in (2560, 4096):
        y = (rng.standard_normal((8, H)) * 0.3).astype(np.float32)
        got = O.rmsnorm_bf16(y, 1e-6)
        want = O.rmsnorm_bf16_f64(y, 1e-6)
        diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
        assert diff.max() <= 1 and np.count_nonzero(diff) <= 8
        r = O.rms_inv_fixed_order(y, 1e-6).astype(np.float64)
        y64 = y.astype(np.float64)
        r_exact = 1.0 / np.sqrt(np.mean(y64 * y64, axis=1) + 1e-6)
        assert np.all(np.abs(r / r_exact - 1.0) <= 16 * 2.0 ** -24)


def test_rmsnorm_definition_matches_torch_float64():
    # the float64 definition against torch's own RMS norm in float64
    rng = np.random.default_rng(13)
    y = (rng.standard_normal((4, 2560)) * 0.3).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(y).double(), (2560,), eps=1e-6)
    assert np.array_equal(O.rmsnorm_bf16_f64(y, 1e-6), O.bf16_round_bits(ref.numpy()))
    xs = O.bf16_bits_to_f32(O.rmsnorm_bf16(y, 1e-6)).astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(xs * xs, axis=1)), 1.0, atol=1e-2)


def test_rmsnorm_special_cases():
    # constant rows: every element maps to sign(c) / sqrt(1 + eps/c^2)
    y = np.array([[2.0] * 512, [-0.5] * 512], dtype=np.float32)
    x = O.bf16_bits_to_f32(O.rmsnorm_bf16(y, 1e-6))
    assert np.all(x[0] == 1.0) and np.all(x[1] == -1.0)
    # a zero row stays zero (r = 1/sqrt(eps) times 0)
    z = O.rmsnorm_bf16(np.zeros((1, 256), dtype=np.float32), 1e-6)
    assert np.all(z == 0)
    # scale invariance up to rounding: y and 4y (exact power of two) agree bit for bit
    rng = np.random.default_rng(12)
    y = rng.standard_normal((2, 768)).astype(np.float32)
    assert np.array_equal(O.rmsnorm_bf16(y, 0.0), O.rmsnorm_bf16(4 * y, 0.0))


def test_fp8_gemv_brute_force():
    rng = np.random.default_rng(11)
    M, K = 9, 48
    W = rng.integers(0, 256, (M, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x11                 # no NaN codes
    s = rng.uniform(0.5, 2.0, M).astype(np.float32)
    xb = _bits(synth.activations(1, K, 26))[0]
    got = O.fp8_rowscale_gemv(W, s, xb)
    x = O.bf16_bits_to_f32(xb)
    for m in range(M):
        want = float(s[m]) * math.fsum(_e4m3(int(W[m, c])) * float(x[c]) for c in range(K))
        assert np.float32(want) == got[m] or abs(want - got[m]) <= 1e-6 * abs(want)
