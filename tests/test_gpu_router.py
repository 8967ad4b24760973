"""moe_router_topk vs the oracle: logits and indices bit for bit, weights to
1e-6 relative."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _run(T, E, H, k, seed, bias=None, dup=None):
    x = synth.activations(T, H, seed).cuda()
    wr = synth.router_weights(E, H, seed + 1)
    if dup:
        for a, b in dup:
            wr[a] = wr[b]
    wr = wr.cuda()
    b = None if bias is None else bias.cuda()
    idx, w, logits = moe.moe_router_topk(x, wr, b, k)
    torch.cuda.synchronize()
    return x, wr, bias, idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def _check(x, wr, bias, idx, w, logits, k, rows=None):
    xb, wb = bits(x), bits(wr)
    if rows is not None:
        xb = xb[rows]
        idx, w, logits = idx[rows], w[rows], logits[rows]
    want_l = O.router_logits(xb, wb, None if bias is None else bias.numpy())
    assert np.array_equal(logits.view(np.uint32), want_l.view(np.uint32)), \
        f"{np.count_nonzero(logits != want_l)} logits differ"
    want_i, want_w = O.topk_softmax(want_l, k)
    assert np.array_equal(idx, want_i)
    assert np.allclose(w, want_w, rtol=1e-6, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


@pytest.mark.parametrize("T,E,H,k", [
    (1, 64, 2560, 10),      # one layer, one token
    (1, 512, 2560, 10),     # decode-stack layer
    (32, 512, 2560, 10),    # batched decode
    (17, 65, 256, 7),       # ragged tokens and experts
    (1, 384, 4096, 6),      # DeepSeek-shaped
    (5, 8, 64, 8),          # k = E: full softmax
    (3, 33, 72, 1),         # k = 1, H not a multiple of 256
])
def test_router_exact(T, E, H, k):
    out = _run(T, E, H, k, seed=10 * T + E)
    _check(*out, k)


# Many-token shapes: T >= 64 with H a multiple of 256 take the shared-memory
# tiled kernel (32 tokens x 8 experts per CTA, K-steps of 256 through a
# three-buffer ring); just below either threshold the warp-per-logit kernel.
@pytest.mark.parametrize("T,E,H,k,biased", [
    (64, 8, 256, 4, False),       # the threshold; one K-step; one expert tile
    (97, 65, 512, 10, False),     # ragged token and expert tiles; two K-steps
    (130, 33, 768, 3, True),      # three K-steps (one full turn of the ring), bias
    (300, 512, 2560, 10, True),   # ten K-steps: the ring wraps three times
    (63, 64, 2560, 10, False),    # one token short of the tiled kernel
    (80, 64, 320, 10, False),     # H not a multiple of 256
])
def test_router_many_tokens_exact(T, E, H, k, biased):
    bias = synth.zipf_bias(E, seed=T + E) if biased else None
    out = _run(T, E, H, k, seed=7 * T + E, bias=bias)
    _check(*out, k)


def test_router_prompt_sampled_rows_with_zipf_bias():
    T, E, H, k = 2451, 512, 2560, 10
    bias = synth.zipf_bias(E, seed=2003)
    x, wr, b, idx, w, logits = _run(T, E, H, k, seed=2000, bias=bias)
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(T - 8, T),
                                     np.random.default_rng(0).choice(T, 48, replace=False)]))
    _check(x, wr, b, idx, w, logits, k, rows)


def test_router_exact_ties_go_to_lower_index():
    dup = [(20, 3), (7, 3), (31, 3)]
    x, wr, b, idx, w, logits = _run(4, 32, 512, 32, seed=5, dup=dup)
    _check(x, wr, b, idx, w, logits, 32)
    for t in range(4):
        order = list(idx[t])
        assert order.index(3) < order.index(7) < order.index(20) < order.index(31)


def test_router_nan_ranks_last():
    bias = torch.zeros(32)
    bias[5] = float("nan")
    bias[6] = float("-inf")
    x, wr, b, idx, w, logits = _run(3, 32, 128, 32, seed=6, bias=bias)
    assert np.all(idx[:, -1] == 5) and np.all(idx[:, -2] == 6)


def test_router_repeatable():
    x = synth.activations(32, 2560, 7).cuda()
    wr = synth.router_weights(512, 2560, 8).cuda()
    ref = moe.moe_router_topk(x, wr, None, 10)
    for _ in range(5):
        out = moe.moe_router_topk(x, wr, None, 10)
        for a, b in zip(ref, out):
            assert torch.equal(a, b)


@pytest.mark.parametrize("T,E,H,k", [(1, 512, 2560, 10), (1, 384, 4096, 6), (3, 64, 2560, 10),
                                     (6, 512, 2560, 10)])
def test_rmsnorm_router_fused_exact(T, E, H, k):
    g = torch.Generator().manual_seed(T * E)
    y = torch.randn(T, H, generator=g) * 0.05
    wr = synth.router_weights(E, H, seed=T + E)
    x, idx, w, logits = moe.moe_rmsnorm_router_topk(y.cuda(), wr.cuda(), None, k, eps=1e-6)
    torch.cuda.synchronize()
    want_x = O.rmsnorm_bf16(y.numpy(), 1e-6)
    assert np.array_equal(bits(x), want_x)
    want_l = O.router_logits(want_x, bits(wr))
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), want_l.view(np.uint32))
    want_i, want_w = O.topk_softmax(want_l, k)
    assert np.array_equal(idx.cpu().numpy(), want_i)
    assert np.allclose(w.cpu().numpy(), want_w, rtol=1e-6, atol=0)
