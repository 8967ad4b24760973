"""moe_experts_decode vs the oracle: rel-L2 <= 1e-5 (FP32 accumulation path)."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def pool64():
    return Pool(64, 2560, 640, 0, workload=0)


def _route(T, E, H, k, seed):
    x = synth.activations(T, H, seed)
    wr = synth.router_weights(E, H, seed + 1)
    xb, wb = bits(x), bits(wr)
    idx, w = O.topk_softmax(O.router_logits(xb, wb), k)
    return x, xb, idx, w


def _decode_vs_oracle(pool, T, k, seed, idx=None, w=None):
    x, xb, ridx, rw = _route(T, pool.E, pool.H, k, seed)
    idx = ridx if idx is None else idx
    w = rw if w is None else w
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe.moe_experts_decode(x.cuda(), torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda(),
                               torch.from_numpy(w.astype(np.float32)).cuda(), pool.ptrs,
                               pool.shape, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = O.moe_layer_decode(xb, idx, w, pool.oracle_records(idx.ravel()), pool.H, pool.I,
                              pool.fmt)
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    return O.rel_l2(got, want), got


def test_decode_one_token_top10_of_64(pool64):
    err, _ = _decode_vs_oracle(pool64, 1, 10, seed=1)
    assert err <= TOL, err


@pytest.mark.parametrize("T", [2, 17, 32])
def test_decode_multi_token(pool64, T):
    err, _ = _decode_vs_oracle(pool64, T, 10, seed=100 + T)
    assert err <= TOL, err


def test_decode_k1_and_repeated_expert(pool64):
    idx = np.array([[5]], dtype=np.int32)
    err, _ = _decode_vs_oracle(pool64, 1, 1, seed=3, idx=idx, w=np.array([[1.0]]))
    assert err <= TOL
    idx = np.array([[9, 9, 2]], dtype=np.int32)       # same expert twice in one token
    err, _ = _decode_vs_oracle(pool64, 1, 3, seed=4, idx=idx, w=np.array([[0.5, 0.3, 0.2]]))
    assert err <= TOL


def test_decode_mxfp4_deepseek_shape():
    pool = Pool(12, 4096, 2880, 1, workload=3)
    err, _ = _decode_vs_oracle(pool, 1, 6, seed=30)
    assert err <= TOL, err


@pytest.mark.parametrize("T", [4, 6])
def test_decode_ring_multi_row_chunks(pool64, T):
    """Shapes the one-shot plan does not take but the ring kernel does (T*k
    <= 64): its chunks of several row pairs and blocks of several output rows
    are cut at pair and token boundaries and end ragged."""
    err, _ = _decode_vs_oracle(pool64, T, 10, seed=200 + T)
    assert err <= TOL, err


def test_decode_ring_mxfp4_two_tokens():
    pool = Pool(12, 4096, 2880, 1, workload=3)
    err, _ = _decode_vs_oracle(pool, 2, 6, seed=33)
    assert err <= TOL, err


@pytest.mark.parametrize("T,k", [(51, 10), (64, 8), (52, 10), (130, 4)])
def test_decode_ring_limit_and_two_kernel_path(pool64, T, k):
    """T*k = 510 and 512 take the ring kernel (its pair table holds at most 512
    pairs); 520 takes the two-kernel path on HBM records, with k = 10 and 4."""
    err, _ = _decode_vs_oracle(pool64, T, k, seed=300 + T)
    assert err <= TOL, err


def test_decode_small_shapes():
    pool = Pool(8, 128, 64, 0, workload=9)
    err, _ = _decode_vs_oracle(pool, 3, 4, seed=31)
    assert err <= TOL, err
    pool = Pool(8, 192, 128, 1, workload=9, layer=1)
    err, _ = _decode_vs_oracle(pool, 5, 3, seed=32)
    assert err <= TOL, err


def test_decode_repeatable_bitwise(pool64):
    x, xb, idx, w = _route(4, 64, 2560, 10, seed=40)
    args = (x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(),
            pool64.ptrs, pool64.shape)
    ref = moe.moe_experts_decode(*args)
    for _ in range(5):
        assert torch.equal(moe.moe_experts_decode(*args), ref)


def test_decode_bad_inputs_flag_status_and_poison_only_that_token(pool64):
    x, xb, idx, w = _route(3, 64, 2560, 4, seed=41)
    idx = idx.copy()
    idx[1, 2] = 64                                   # out of range
    ptrs = pool64.ptrs.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe.moe_experts_decode(x.cuda(), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w.astype(np.float32)).cuda(), ptrs, pool64.shape,
                               dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_INDEX
    yc = y.cpu().numpy()
    assert np.all(np.isnan(yc[1])) and np.all(np.isfinite(yc[0])) and np.all(np.isfinite(yc[2]))
    # NULL and misaligned records are reported, never dereferenced
    ptrs[int(idx[0, 0])] = 0
    ptrs[int(idx[2, 1])] += 8
    st.zero_()
    idx[1, 2] = 0
    y = moe.moe_experts_decode(x.cuda(), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w.astype(np.float32)).cuda(), ptrs, pool64.shape,
                               dev_status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & moe.DEV_NULL_EXPERT and s & moe.DEV_MISALIGNED
    yc = y.cpu().numpy()
    assert np.all(np.isnan(yc[0])) and np.all(np.isnan(yc[2])) and np.all(np.isfinite(yc[1]))


def test_decode_rejects_small_workspace(pool64):
    x = synth.activations(1, 2560, 1).cuda()
    idx = torch.zeros(1, 10, dtype=torch.int32, device="cuda")
    w = torch.zeros(1, 10, dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError, match="workspace too small"):
        moe.moe_experts_decode(x, idx, w, pool64.ptrs, pool64.shape, workspace=ws)
