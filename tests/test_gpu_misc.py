"""Bucketing (bit-exact), RMS chaining (bit-exact) and FP8 GEMV (rel-L2 1e-5)
vs the oracle."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _idx(T, k, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,k,E", [(1, 10, 64), (2451, 10, 512), (33, 6, 384), (300, 1, 1),
                                   (1024, 8, 16), (5, 3, 4096)])
def test_bucket_exact(T, k, E):
    idx = _idx(T, k, E, T + E) if k <= E else None
    counts, offsets, pairs = moe.moe_bucket_by_expert(torch.from_numpy(idx).cuda(), E)
    c, o, p = O.bucket_by_expert(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(pairs.cpu().numpy()[: T * k], p)


def test_bucket_skewed_and_empty_experts():
    rng = np.random.default_rng(3)
    T, k, E = 1500, 2, 300
    idx = np.zeros((T, k), dtype=np.int32)
    idx[:, 0] = 7                                   # one expert gets every token
    idx[:, 1] = rng.integers(100, 110, T)           # most experts get none
    counts, offsets, pairs = moe.moe_bucket_by_expert(torch.from_numpy(idx).cuda(), E)
    c, o, p = O.bucket_by_expert(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(pairs.cpu().numpy(), p)


def test_bucket_bad_index_flagged():
    idx = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts, offsets, pairs = moe.moe_bucket_by_expert(idx, 4, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_INDEX
    assert counts.cpu().tolist() == [1, 1, 1, 0]


@pytest.mark.parametrize("T,H", [(1, 2560), (32, 2560), (3, 4096), (2, 64)])
def test_rmsnorm_bitexact(T, H):
    g = torch.Generator().manual_seed(T * H)
    y = torch.randn(T, H, generator=g) * 0.05
    x = moe.moe_rmsnorm_bf16(y.cuda(), 1e-6)
    want = O.rmsnorm_bf16(y.numpy(), 1e-6)
    got = bits(x)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} differ"


# one or two rows per warp (odd M leaves a warp with one), one to eight
# 16-byte units per lane (every instance of the row kernel), ragged units per
# lane, and rows longer than 4096 elements (the chunked kernel)
@pytest.mark.parametrize("M,K", [(8192, 2560), (2560, 4096), (1000, 16), (37, 272), (4097, 2560), (65, 1040),
                                 (3, 8192), (33, 1024), (34, 2048), (35, 3072), (36, 3584)])
def test_fp8_gemv(M, K):
    rng = np.random.default_rng(M + K)
    W = synth.expert_matrix((M, K), seed=M * 7 + K)
    w8 = W.to(torch.float8_e4m3fn).view(torch.uint8)
    s = synth.uniform((M,), seed=M, lo=0.5, hi=2.0)
    x = synth.activations(1, K, seed=K)[0]
    y = moe.fp8_rowscale_gemv(w8.cuda(), s.cuda(), x.cuda())
    want = O.fp8_rowscale_gemv(w8.numpy(), s.numpy(), bits(x))
    err = O.rel_l2(y.cpu().numpy(), want)
    assert err <= 1e-5, err


def test_fp8_gemv_chained_after_the_kernel_that_writes_x():
    """The GEMV reads its weights before waiting on the previous kernel of the
    stream and x only after: x produced by the kernel right before it (the RMS
    normalisation, launched on the same stream) must be the x it uses, across
    a chain of back-to-back calls captured in a graph."""
    M, K = 4096, 2560
    W = synth.expert_matrix((M, K), seed=77)
    w8 = W.to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    s = synth.uniform((M,), seed=78, lo=0.5, hi=2.0).cuda()
    ys = [torch.randn(1, K, generator=torch.Generator().manual_seed(80 + i)) * 0.05 for i in range(4)]
    yd = [y.cuda() for y in ys]
    x = torch.empty(1, K, dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in ys]
    g = torch.cuda.CUDAGraph()
    moe.moe_rmsnorm_bf16(yd[0], 1e-6, x=x)
    moe.fp8_rowscale_gemv(w8, s, x[0], outs[0])
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(len(ys)):
            moe.moe_rmsnorm_bf16(yd[i], 1e-6, x=x)
            moe.fp8_rowscale_gemv(w8, s, x[0], outs[i])
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    w_np = w8.cpu().numpy()
    for i, y in enumerate(ys):
        xb = O.rmsnorm_bf16(y.numpy(), 1e-6)
        want = O.fp8_rowscale_gemv(w_np, s.cpu().numpy(), xb[0])
        err = O.rel_l2(outs[i].cpu().numpy(), want)
        assert err <= 1e-5, (i, err)

