"""moe_experts_grouped (tcgen05 path) vs the oracle's BF16-intermediate
layer: rel-L2 <= 2e-3."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits, oracle_pack_many
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _run(pool, x, idx, w, st=None):
    return moe.moe_experts_grouped(x.cuda(), torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda(),
                                   torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda(),
                                   pool.ptrs, pool.shape, dev_status=st)


def _route(T, E, H, k, seed, bias=None):
    x = synth.activations(T, H, seed)
    wr = synth.router_weights(E, H, seed + 1)
    idx, w = O.topk_softmax(O.router_logits(bits(x), bits(wr), bias), k)
    return x, idx, w


def _check(pool, x, idx, w, tokens=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _run(pool, x, idx, w, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    recs = oracle_pack_many(pool, idx[sel].ravel())
    want = O.moe_layer_grouped_by_expert(bits(x), idx, w, recs, pool.H, pool.I, pool.fmt,
                                         tokens=sel)
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    return O.rel_l2(got[sel], want[sel])


@pytest.fixture(scope="module")
def small_pool():
    return Pool(16, 256, 128, 0, workload=20)


@pytest.mark.parametrize("T,k", [(1, 1), (5, 4), (37, 4), (64, 10)])
def test_grouped_small_shapes(small_pool, T, k):
    x, idx, w = _route(T, 16, 256, k, seed=200 + T)
    err = _check(small_pool, x, idx, w)
    assert err <= TOL, err


def test_grouped_expert_with_many_token_tiles(small_pool):
    T = 300                                        # > 2 token tiles of 128 on one expert
    x = synth.activations(T, 256, 210)
    idx = np.stack([np.full(T, 3), (np.arange(T) % 15) + (np.arange(T) % 15 >= 3)], 1).astype(np.int32)
    w = np.tile(np.array([[0.7, 0.3]]), (T, 1))
    err = _check(small_pool, x, idx, w)
    assert err <= TOL, err


def test_grouped_mxfp4():
    pool = Pool(8, 256, 256, 1, workload=21)
    x, idx, w = _route(40, 8, 256, 3, seed=220)
    err = _check(pool, x, idx, w)
    assert err <= TOL, err


def test_grouped_qwen_shape_64_tokens():
    pool = Pool(64, 2560, 640, 0, workload=22)
    x, idx, w = _route(64, 64, 2560, 10, seed=230)
    err = _check(pool, x, idx, w, tokens=np.arange(0, 64, 9))
    assert err <= TOL, err


def test_grouped_matches_decode_path_within_tolerance(small_pool):
    x, idx, w = _route(24, 16, 256, 4, seed=240)
    yg = _run(small_pool, x, idx, w)
    yd = moe.moe_experts_decode(x.cuda(), torch.from_numpy(idx).cuda(),
                                torch.from_numpy(w.astype(np.float32)).cuda(), small_pool.ptrs,
                                small_pool.shape)
    assert O.rel_l2(yg.cpu().numpy(), yd.cpu().numpy()) <= TOL


def test_grouped_repeatable_within_tolerance(small_pool):
    x, idx, w = _route(50, 16, 256, 4, seed=250)
    ref = _run(small_pool, x, idx, w).cpu().numpy()
    for _ in range(5):
        got = _run(small_pool, x, idx, w).cpu().numpy()
        assert np.all(np.isfinite(got))
        assert O.rel_l2(got, ref) <= 1e-6


def test_grouped_bad_index_poisons_token(small_pool):
    x, idx, w = _route(6, 16, 256, 2, seed=260)
    idx = idx.copy()
    idx[2, 1] = 99
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _run(small_pool, x, idx, w, st).cpu().numpy()
    assert int(st.item()) & moe.DEV_BAD_INDEX
    assert np.all(np.isnan(y[2]))
    assert np.all(np.isfinite(np.delete(y, 2, axis=0)))
