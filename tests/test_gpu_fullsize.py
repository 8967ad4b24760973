"""Parity at the workloads' full sizes, in the launch configuration bench.py
times, on outputs the oracle computes one by one.

* Qwen decode stack: 48 layers x 512 NVFP4 experts (68 GB resident).  The
  CUDA-graph replay bench.py times must equal the eager per-layer calls bit
  for bit; sampled layers are checked against the oracle with the oracle's own
  inputs (layer 0 from x0, deeper layers from independently seeded inputs).
* Qwen prompt layer: 2451 tokens, Zipf-skewed routing over 512 experts --
  every token against the oracle, and every token of the most-loaded expert
  on its own.
* DeepSeek-shaped MXFP4 layer: 384 experts of 18,800,640 bytes, top-6; ten of
  the forty seeded calls, with the L2 flushed before each.
* Batched decode: 32 tokens through all 48 layers of the stack, the router's
  RMS chaining included, teacher-forced layer by layer with the oracle's own
  chain (marked slow as well: it runs the oracle on ~11,000 expert pairs).

The oracle's layer functions run split over worker processes by expert
(helpers.oracle_layer_split); each pair's arithmetic is the oracle's own.
"""
import os
import sys

import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits, oracle_layer_split, oracle_pack_many
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


class _StackView:
    """Gives oracle_pack_many the FP32 inputs behind a decode-stack slot."""

    def __init__(self, stack, layer):
        self.stack, self.layer = stack, layer
        self.fmt = O.FMT_NVFP4
        self._oracle_records = {}

    def weights(self, e):
        u = int(self.stack.choice[self.layer][e])
        return synth.expert_weights(bench.H, bench.I, synth.expert_seed(bench.WORKLOAD_ID, 0, u),
                                    device="cuda")


@pytest.fixture(scope="module")
def stack():
    st = bench.DecodeStack(torch, moe, synth, torch.device("cuda"), 0, 4)
    yield st
    del st.slots
    torch.cuda.empty_cache()


def _layer_gpu(st, L, x):
    """One layer on the GPU with the bench's kernels for a given BF16 input."""
    st.x.copy_(x)
    moe.moe_router_topk(st.x, st.wr[L], None, bench.K_TOP, st.idx, st.w, st.logits)
    moe.moe_experts_decode(st.x, st.idx, st.w, st.ptrs[L], st.s, st.y, st.ws, st.st)
    torch.cuda.synchronize()
    return st.idx.cpu().numpy().copy(), st.y.cpu().numpy().copy()


def _layer_oracle(st, L, xb):
    idx, w = O.topk_softmax(O.router_logits(xb, bits(st.wr[L])), bench.K_TOP)
    recs = oracle_pack_many(_StackView(st, L), idx.ravel())
    y = O.moe_layer_decode(xb, idx, w, recs, bench.H, bench.I, O.FMT_NVFP4)
    return idx, y


def test_stack_graph_replay_equals_eager_calls(stack):
    st = stack
    g, _ = st.capture(with_events=False)
    st.x.copy_(st.x0[1:2])
    g.replay()
    torch.cuda.synchronize()
    y_graph = st.y.clone()
    st.x.copy_(st.x0[1:2])
    st.run_layers()
    torch.cuda.synchronize()
    assert int(st.st.item()) == 0
    assert torch.equal(st.y, y_graph)
    assert torch.isfinite(y_graph).all()


def test_persistent_stack_equals_graph_replay(stack):
    """moe_decode_stack runs all 48 layers of the bench's stack in one launch;
    it must give the bits of the per-layer launches bench.py times."""
    st = stack
    st.x.copy_(st.x0[2:3])
    st.run_layers()
    torch.cuda.synchronize()
    y_ref, idx_last = st.y.clone(), st.idx.clone()
    ptrs = torch.stack(st.ptrs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x_out, idx, w, lg, y = moe.moe_decode_stack(st.x0[2:3].contiguous(), st.wr, None, bench.K_TOP, ptrs, st.s,
                                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(idx[-1], idx_last)
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))


def test_stack_layers_against_oracle(stack):
    st = stack
    # layer 0 from the stack's own first token, then the oracle's chained x1
    xb0 = bits(st.x0[0:1])
    idx0, y0 = _layer_oracle(st, 0, xb0)
    gi, gy = _layer_gpu(st, 0, st.x0[0:1])
    assert np.array_equal(gi, idx0)
    assert O.rel_l2(gy, y0) <= 1e-5
    x1 = O.rmsnorm_bf16(y0, 1e-6)
    x1_t = torch.from_numpy(x1.view(np.int16)).view(torch.bfloat16).cuda()
    idx1, y1 = _layer_oracle(st, 1, x1)
    gi, gy = _layer_gpu(st, 1, x1_t)
    assert np.array_equal(gi, idx1)
    assert O.rel_l2(gy, y1) <= 1e-5
    # the fused RMS-chaining router on the oracle's y0 gives the oracle's x1 and routing
    xg, ig, wg, _ = moe.moe_rmsnorm_router_topk(torch.from_numpy(y0).cuda(), st.wr[1], None,
                                                bench.K_TOP, 1e-6)
    assert np.array_equal(bits(xg), x1)
    assert np.array_equal(ig.cpu().numpy(), idx1)
    # deep layers on independently seeded, RMS-normalised inputs
    for L in (23, 47):
        y_seed = synth.activations(1, bench.H, 7000 + L).float().numpy()
        xl = O.rmsnorm_bf16(y_seed, 1e-6)
        xl_t = torch.from_numpy(xl.view(np.int16)).view(torch.bfloat16).cuda()
        idx_l, y_l = _layer_oracle(st, L, xl)
        gi, gy = _layer_gpu(st, L, xl_t)
        assert np.array_equal(gi, idx_l)
        assert O.rel_l2(gy, y_l) <= 1e-5


class _UniqueView:
    """Oracle packing of the stack's distinct experts, keyed by distinct id."""

    def __init__(self, stack):
        self.stack = stack
        self.fmt = O.FMT_NVFP4
        self._oracle_records = {}

    def weights(self, u):
        return synth.expert_weights(bench.H, bench.I, synth.expert_seed(bench.WORKLOAD_ID, 0, int(u)),
                                    device="cuda")


@pytest.mark.slow
def test_batched_decode_32_tokens_48_chained_layers(stack):
    """The batched-decode workload as bench.py runs it (router or fused RMS
    chaining + router, then the expert pass for 32 tokens), layer by layer on
    the oracle's own chain: the GPU gets the oracle's x_L (and, for the
    chaining, the oracle's y_{L-1}); indices must be equal and y within the
    decode tolerance on every one of the 48 layers."""
    st = stack
    T = 32
    uv = _UniqueView(st)
    x0 = synth.activations(T, bench.H, synth.seed_of(4, 100, synth.T_X), device="cuda")
    xb = bits(x0)
    y_prev = None
    worst = 0.0
    for L in range(bench.LAYERS):
        wrb = bits(st.wr[L])
        idx_o, w_o = O.topk_softmax(O.router_logits(xb, wrb), bench.K_TOP)
        ch = st.choice[L]
        recs_u = oracle_pack_many(uv, [int(ch[e]) for e in idx_o.ravel()])
        recs = {int(e): recs_u[int(ch[e])] for e in idx_o.ravel()}
        y_o = oracle_layer_split("moe_layer_decode", xb, idx_o, w_o, recs, bench.H, bench.I, O.FMT_NVFP4)
        x_t = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        if y_prev is None:
            idx_g, w_g, _ = moe.moe_router_topk(x_t, st.wr[L], None, bench.K_TOP)
        else:
            xg, idx_g, w_g, _ = moe.moe_rmsnorm_router_topk(torch.from_numpy(y_prev).cuda(), st.wr[L], None,
                                                            bench.K_TOP, 1e-6)
            assert np.array_equal(bits(xg), xb), L
        y_g = moe.moe_experts_decode(x_t, idx_g, w_g, st.ptrs[L], st.s)
        torch.cuda.synchronize()
        assert np.array_equal(idx_g.cpu().numpy(), idx_o), L
        err = O.rel_l2(y_g.cpu().numpy(), y_o)
        worst = max(worst, err)
        assert err <= 1e-5, (L, err)
        y_prev = y_o
        xb = O.rmsnorm_bf16(y_o, 1e-6)
    print(f"worst rel-L2 over 48 layers x 32 tokens: {worst:.2e}")


def test_prompt_layer_full_size_all_tokens():
    pl = bench.PromptLayer(torch, moe, synth, torch.device("cuda"))
    pl.step()
    torch.cuda.synchronize()
    assert int(pl.st.item()) == 0
    counts = torch.bincount(pl.idx.flatten().long(), minlength=bench.E)
    assert int((counts > 0).sum()) >= 480            # Zipf bias: nearly every expert is hit
    xb = bits(pl.x)
    logits = O.router_logits(xb, bits(pl.wr), pl.bias.cpu().numpy())
    idx, w = O.topk_softmax(logits, bench.K_TOP)
    assert np.array_equal(pl.idx.cpu().numpy(), idx)

    class _View:
        fmt = O.FMT_NVFP4
        _oracle_records = {}

        def weights(self, e):
            return synth.expert_weights(bench.H, bench.I, synth.expert_seed(pl.WORKLOAD, 0, int(e)),
                                        device="cuda")

    recs = oracle_pack_many(_View(), idx.ravel())
    want = oracle_layer_split("moe_layer_grouped_by_expert", xb, idx, w, recs, bench.H, bench.I, O.FMT_NVFP4)
    got = pl.y.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert O.rel_l2(got, want) <= 2e-3
    # every token of the most-loaded expert (its token tiles span 13 tiles of 128)
    top = int(np.argmax(np.bincount(idx.ravel(), minlength=bench.E)))
    toks = np.nonzero((idx == top).any(axis=1))[0]
    assert len(toks) > 1000
    for t in toks:
        assert O.rel_l2(got[t], want[t]) <= 2e-3, t


def test_deepseek_shaped_mxfp4_calls():
    """Ten of the forty seeded DeepSeek-shaped calls exactly as bench.py runs
    them (router, then the expert pass on one 384-expert MXFP4 weight set),
    the L2 flushed before each."""
    dc = bench.DeepSeekCalls(torch, moe, synth, torch.device("cuda"))
    assert dc.rb == 18_800_640

    class _View:
        fmt = O.FMT_MXFP4
        _oracle_records = {}

        def weights(self, e):
            return synth.expert_weights(dc.HD, dc.ID, synth.expert_seed(dc.WORKLOAD, 0, int(e)), device="cuda")

    view = _View()
    for c in range(0, dc.CALLS, 4):
        dc.flush()
        dc.router(c)
        dc.experts(c)
        torch.cuda.synchronize()
        assert int(dc.st.item()) == 0
        xb = bits(dc.xs[c])
        want_i, want_w = O.topk_softmax(O.router_logits(xb, bits(dc.wr[c])), dc.KD)
        assert np.array_equal(dc.idx.cpu().numpy(), want_i), c
        recs = oracle_pack_many(view, want_i.ravel())
        want = oracle_layer_split("moe_layer_decode", xb, want_i, want_w, recs, dc.HD, dc.ID, O.FMT_MXFP4)
        assert O.rel_l2(dc.y.cpu().numpy(), want) <= 1e-5, c
