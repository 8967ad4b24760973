"""Parity at the workloads' full sizes, in the launch configuration bench.py
times, on outputs the oracle computes one by one.

* Qwen decode stack: 48 layers x 512 NVFP4 experts (68 GB resident).  The
  CUDA-graph replay bench.py times must equal the eager per-layer calls bit
  for bit; sampled layers are checked against the oracle with the oracle's own
  inputs (layer 0 from x0, deeper layers from independently seeded inputs).
* Qwen prompt layer: 2451 tokens, Zipf-skewed routing over 512 experts.
* DeepSeek-shaped MXFP4 layer: 384 experts of 18,800,640 bytes, top-6.
* Batched decode: 32 tokens over the 512-expert pool.
"""
import os
import sys

import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits, oracle_pack_many
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


def test_batched_decode_32_tokens(stack):
    st = stack
    L = 5
    x = synth.activations(32, bench.H, 4321)
    xb = bits(x)
    idx, w = O.topk_softmax(O.router_logits(xb, bits(st.wr[L])), bench.K_TOP)
    y = moe.moe_experts_decode(x.cuda(), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(w.astype(np.float32)).cuda(), st.ptrs[L], st.s)
    got = y.cpu().numpy()
    sample = [0, 7, 31]
    recs = oracle_pack_many(_StackView(st, L), idx[sample].ravel())
    want = O.moe_layer_decode(xb[sample], idx[sample], w[sample], recs, bench.H, bench.I,
                              O.FMT_NVFP4)
    assert O.rel_l2(got[sample], want) <= 1e-5


def test_prompt_layer_full_size_sampled_tokens():
    pl = bench.PromptLayer(torch, moe, synth, torch.device("cuda"))
    pl.step()
    torch.cuda.synchronize()
    assert int(pl.st.item()) == 0
    counts = torch.bincount(pl.idx.flatten().long(), minlength=bench.E)
    assert int((counts > 0).sum()) >= 480            # Zipf bias: nearly every expert is hit
    xb = bits(pl.x)
    tokens = np.array([0, 1, 1000, 2450])
    logits = O.router_logits(xb[tokens], bits(pl.wr), pl.bias.cpu().numpy())
    idx, w = O.topk_softmax(logits, bench.K_TOP)
    assert np.array_equal(pl.idx.cpu().numpy()[tokens], idx)

    class _View:
        fmt = O.FMT_NVFP4
        _oracle_records = {}

        def weights(self, e):
            return synth.expert_weights(bench.H, bench.I, synth.expert_seed(pl.WORKLOAD, 0, int(e)),
                                        device="cuda")

    recs = oracle_pack_many(_View(), idx.ravel())
    want = O.moe_layer_grouped(xb[tokens], idx, w, recs, bench.H, bench.I, O.FMT_NVFP4)
    got = pl.y.cpu().numpy()[tokens]
    assert np.all(np.isfinite(pl.y.cpu().numpy()))
    assert O.rel_l2(got, want) <= 2e-3


def test_deepseek_shaped_mxfp4_layer():
    pool = Pool(384, 4096, 2880, 1, workload=3)
    assert moe.moe_expert_record_bytes(pool.shape) == 18_800_640
    wr = synth.router_weights(384, 4096, synth.seed_of(3, 0, synth.T_ROUTER))
    for call in range(2):
        x = synth.activations(1, 4096, synth.seed_of(3, 10 + call, synth.T_X))
        xb = bits(x)
        idx, w, _ = moe.moe_router_topk(x.cuda(), wr.cuda(), None, 6)
        want_i, want_w = O.topk_softmax(O.router_logits(xb, bits(wr)), 6)
        assert np.array_equal(idx.cpu().numpy(), want_i)
        y = moe.moe_experts_decode(x.cuda(), idx, w, pool.ptrs, pool.shape)
        recs = oracle_pack_many(pool, want_i.ravel())
        want = O.moe_layer_decode(xb, want_i, want_w, recs, 4096, 2880, O.FMT_MXFP4)
        assert O.rel_l2(y.cpu().numpy(), want) <= 1e-5
