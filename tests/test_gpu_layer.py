"""moe_decode_layer (router and expert pass in one launch) against the two
calls it fuses -- moe_router_topk / moe_rmsnorm_router_topk, then
moe_experts_decode -- which the other tests pin to the oracle: every output
must be identical bit for bit.  One case is also checked against the oracle
directly."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool64():
    return Pool(64, 2560, 640, 0, workload=0)


@pytest.fixture(scope="module")
def pool_small():
    return Pool(24, 256, 128, 1, workload=5)


def _two_calls(pool, k, x=None, y_prev=None, wr=None, bias=None, eps=1e-6):
    if x is not None:
        idx, w, logits = moe.moe_router_topk(x, wr, bias, k)
        x_out = x
    else:
        x_out, idx, w, logits = moe.moe_rmsnorm_router_topk(y_prev, wr, bias, k, eps)
    y = moe.moe_experts_decode(x_out, idx, w, pool.ptrs, pool.shape)
    return x_out, idx, w, logits, y


def _same(a, b):
    a, b = a.cpu(), b.cpu()
    if a.dtype.is_floating_point:
        return torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("mode", ["x", "y_prev"])
@pytest.mark.parametrize("with_bias", [False, True])
def test_layer_equals_two_calls(pool64, mode, with_bias):
    k, H, T = 10, pool64.H, 1
    wr = synth.router_weights(pool64.E, H, 700 + with_bias).cuda()
    bias = synth.zipf_bias(pool64.E, 71).cuda() if with_bias else None
    if mode == "x":
        x = synth.activations(T, H, 800 + T).cuda()
        ref = _two_calls(pool64, k, x=x, wr=wr, bias=bias)
        got = moe.moe_decode_layer(wr, bias, k, pool64.ptrs, pool64.shape, x=x)
        assert got[0] is None
        pairs = zip(ref[1:], got[1:])
    else:
        y_prev = torch.randn(T, H, device="cuda", generator=torch.Generator("cuda").manual_seed(7 + with_bias)) * 0.3
        ref = _two_calls(pool64, k, y_prev=y_prev, wr=wr, bias=bias)
        got = moe.moe_decode_layer(wr, bias, k, pool64.ptrs, pool64.shape, y_prev=y_prev)
        pairs = zip(ref, got)
    torch.cuda.synchronize()
    for r, g in pairs:
        assert _same(r, g)


@pytest.mark.parametrize("mode", ["x", "y_prev"])
def test_layer_mxfp4_several_tokens(pool_small, mode):
    k, H, T = 3, pool_small.H, 5
    wr = synth.router_weights(pool_small.E, H, 901).cuda()
    if mode == "x":
        x = synth.activations(T, H, 902).cuda()
        ref = _two_calls(pool_small, k, x=x, wr=wr)
        got = moe.moe_decode_layer(wr, None, k, pool_small.ptrs, pool_small.shape, x=x)
        pairs = zip(ref[1:], got[1:])
    else:
        y_prev = torch.randn(T, H, device="cuda", generator=torch.Generator("cuda").manual_seed(9)) * 2.0
        ref = _two_calls(pool_small, k, y_prev=y_prev, wr=wr)
        got = moe.moe_decode_layer(wr, None, k, pool_small.ptrs, pool_small.shape, y_prev=y_prev)
        pairs = zip(ref, got)
    torch.cuda.synchronize()
    for r, g in pairs:
        assert _same(r, g)


def test_layer_chain_in_place(pool64):
    """Three chained layers with y written over y_prev, as a decode stack runs."""
    k, H = 10, pool64.H
    wrs = [synth.router_weights(pool64.E, H, 910 + L).cuda() for L in range(3)]
    x0 = synth.activations(1, H, 920).cuda()
    # reference: separate calls
    x = x0.clone()
    y = None
    for L in range(3):
        if L == 0:
            idx, w, _ = moe.moe_router_topk(x, wrs[L], None, k)
        else:
            x, idx, w, _ = moe.moe_rmsnorm_router_topk(y, wrs[L], None, k, 1e-6)
        y = moe.moe_experts_decode(x, idx, w, pool64.ptrs, pool64.shape)
    want = y.clone()
    # fused, one buffer for y across layers
    ws = torch.zeros(moe.moe_experts_decode_workspace(1, k, pool64.shape), dtype=torch.uint8, device="cuda")
    yb = torch.empty(1, H, dtype=torch.float32, device="cuda")
    xb = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    for L in range(3):
        if L == 0:
            moe.moe_decode_layer(wrs[L], None, k, pool64.ptrs, pool64.shape, x=x0, y=yb, workspace=ws)
        else:
            moe.moe_decode_layer(wrs[L], None, k, pool64.ptrs, pool64.shape, y_prev=yb, x_out=xb, y=yb,
                                 workspace=ws)
    torch.cuda.synchronize()
    assert _same(yb, want)


def test_layer_vs_oracle(pool64):
    k, T, H = 10, 1, pool64.H
    x = synth.activations(T, H, 930)
    wr = synth.router_weights(pool64.E, H, 931)
    _, idx, w, logits, y = moe.moe_decode_layer(wr.cuda(), None, k, pool64.ptrs, pool64.shape, x=x.cuda())
    torch.cuda.synchronize()
    xb, wb = bits(x), bits(wr)
    ref_logits = O.router_logits(xb, wb)
    ridx, rw = O.topk_softmax(ref_logits, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    want = O.moe_layer_decode(xb, ridx, rw, pool64.oracle_records(ridx.ravel()), H, pool64.I, pool64.fmt)
    assert O.rel_l2(y.cpu().numpy(), want) <= 1e-5


def test_layer_rejects_shapes_outside_one_shot(pool64):
    k, H = 10, pool64.H
    wr = synth.router_weights(pool64.E, H, 940).cuda()
    x = synth.activations(8, H, 941).cuda()   # T*k = 80 > 64
    with pytest.raises(moe.MoeError):
        moe.moe_decode_layer(wr, None, k, pool64.ptrs, pool64.shape, x=x)


@pytest.fixture(scope="module")
def pool_wide():
    return Pool(1000, 256, 128, 0, workload=6)


def _tied_router(E, H, x, seed):
    """Random BF16 router rows plus rows aligned with sign(x), each copied to a
    second expert in another warp's candidate set, so that the top-k holds
    exactly equal logits (ties go to the lower expert index)."""
    wr = synth.router_weights(E, H, seed)
    sx = torch.sign(x[0].float())
    for scale, a, b in [(0.25, 3, 961), (0.125, 500, 998), (0.0625, 17, 480), (0.03125, 31, 992)]:
        wr[a] = (sx * scale).to(torch.bfloat16)
        wr[b] = wr[a]
    return wr


@pytest.mark.parametrize("k", [8, 24])
def test_layer_wide_router_with_ties(pool_wide, k):
    """E = 1000 needs three candidates per lane in the fused top-k (15 warps);
    k = 8 reads the router rows through L2, k = 24 stages them in shared
    memory.  Fused = two calls, bit for bit, and the picks are the oracle's."""
    E, H = pool_wide.E, pool_wide.H
    x = synth.activations(1, H, 960 + k)
    wr = _tied_router(E, H, x, 961 + k)
    ref = _two_calls(pool_wide, k, x=x.cuda(), wr=wr.cuda())
    got = moe.moe_decode_layer(wr.cuda(), None, k, pool_wide.ptrs, pool_wide.shape, x=x.cuda())
    torch.cuda.synchronize()
    for r, g in zip(ref[1:], got[1:]):
        assert _same(r, g)
    ridx, _ = O.topk_softmax(O.router_logits(bits(x), bits(wr)), k)
    assert np.array_equal(got[1].cpu().numpy(), ridx)
    picks = set(ridx[0].tolist())
    assert {3, 961, 500, 998} <= picks  # the tied pairs are both selected


@pytest.mark.parametrize("k", [8, 24])
def test_layer_wide_router_chained(pool_wide, k):
    E, H = pool_wide.E, pool_wide.H
    wr = synth.router_weights(E, H, 970 + k).cuda()
    y_prev = torch.randn(1, H, device="cuda", generator=torch.Generator("cuda").manual_seed(97 + k)) * 0.5
    ref = _two_calls(pool_wide, k, y_prev=y_prev, wr=wr)
    got = moe.moe_decode_layer(wr, None, k, pool_wide.ptrs, pool_wide.shape, y_prev=y_prev)
    torch.cuda.synchronize()
    for r, g in zip(ref, got):
        assert _same(r, g)
