"""Pins for the oracle's router logits, top-k and softmax weights (CPU only)."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from block_scaled_fp4_softmax_gb300 import synth
from oracle import oracle as O


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _inputs(T, E, H, seed):
    x = synth.activations(T, H, seed)
    w = synth.router_weights(E, H, seed + 1)
    return _bits(x), _bits(w)


def test_logits_close_to_exact_dot_within_fp32_bound():
    xb, wb = _inputs(5, 40, 256, 11)
    l32 = O.router_logits(xb, wb)
    l64 = O.router_logits_f64(xb, wb)
    x = O.bf16_bits_to_f32(xb).astype(np.float64)
    w = O.bf16_bits_to_f32(wb).astype(np.float64)
    absdot = np.abs(x) @ np.abs(w).T
    # 64 + 5 rounding steps at most on any path: |err| <= 70 * 2^-24 * sum|x w|
    assert np.all(np.abs(l32 - l64) <= 70 * 2.0 ** -24 * absdot)


def test_logits_summation_order_brute_force():
    # the slot / chunk order written out with Python floats rounded to FP32
    xb, wb = _inputs(2, 3, 512, 12)
    x = O.bf16_bits_to_f32(xb)
    w = O.bf16_bits_to_f32(wb)
    got = O.router_logits(xb, wb)
    f32 = lambda v: float(np.float32(v))
    for t in range(2):
        for e in range(3):
            slots = [0.0] * 32
            for c in range(512 // 8):
                for i in range(8):
                    h = 8 * c + i
                    slots[c % 32] = f32(slots[c % 32] + float(x[t, h]) * float(w[e, h]))
            for d in (16, 8, 4, 2, 1):
                slots = [f32(slots[j] + slots[j ^ d]) for j in range(32)]
            assert np.float32(slots[0]) == got[t, e]


def test_bias_is_added_after_the_sum():
    xb, wb = _inputs(2, 8, 64, 13)
    b = np.linspace(-1, 1, 8).astype(np.float32)
    assert np.array_equal(O.router_logits(xb, wb, b), O.router_logits(xb, wb) + b)


def test_topk_matches_full_sort_brute_force():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((20, 64)).astype(np.float32)
    L[3, 10] = L[3, 20] = L[3, 30] = 5.0        # exact ties
    L[4, 7] = np.nan                            # NaN ranks last
    idx, w = O.topk_softmax(L, 10)
    for t in range(20):
        def key(e):
            v = float(L[t, e])
            return (1, 0.0, e) if math.isnan(v) else (0, -v, e)
        want = sorted(range(64), key=key)[:10]
        assert list(idx[t]) == want
    assert list(idx[3, :3]) == [10, 20, 30]
    assert 7 not in idx[4]


def test_duplicated_router_rows_tie_to_lower_index():
    xb, wb = _inputs(3, 16, 128, 14)
    wb = wb.copy()
    wb[9] = wb[2]
    wb[15] = wb[2]
    L = O.router_logits(xb, wb)
    assert np.array_equal(L[:, 2], L[:, 9]) and np.array_equal(L[:, 2], L[:, 15])
    idx, _ = O.topk_softmax(L, 16)
    for t in range(3):
        order = list(idx[t])
        assert order.index(2) < order.index(9) < order.index(15)


def test_weights_sum_to_one_and_k_equals_e_is_full_softmax():
    rng = np.random.default_rng(6)
    L = (rng.standard_normal((7, 12)) * 3).astype(np.float32)
    idx, w = O.topk_softmax(L, 4)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)
    idx, w = O.topk_softmax(L, 12)
    full = scipy.special.softmax(L.astype(np.float64), axis=1)
    for t in range(7):
        assert np.allclose(w[t], full[t, idx[t]], rtol=1e-14, atol=0)


def test_renormalised_topk_equals_restricted_full_softmax():
    rng = np.random.default_rng(8)
    L = rng.standard_normal((5, 30)).astype(np.float32)
    idx, w = O.topk_softmax(L, 6)
    full = scipy.special.softmax(L.astype(np.float64), axis=1)
    for t in range(5):
        sel = full[t, idx[t]]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-13)


def test_zipf_bias_profile():
    b = synth.zipf_bias(512, seed=3).numpy().astype(np.float64)
    p = np.exp(b / 0.5)
    assert abs(p.sum() - 1.0) < 1e-5
    ps = np.sort(p)[::-1]
    assert abs(ps[0] / ps[1] - 2 ** 1.1) < 1e-4
