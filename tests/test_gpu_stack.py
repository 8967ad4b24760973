"""moe_decode_stack (all layers of a decode stack in one persistent launch)
against the per-layer launches it replaces -- moe_decode_layer from x for
layer 0, then from the previous y -- which the other tests pin to the oracle:
every output must be identical bit for bit."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool

pytestmark = pytest.mark.gpu


def _per_layer(x0, wr, ptrs, s, k, bias=None, eps=1e-6):
    L = wr.shape[0]
    T, H = x0.shape
    ws = torch.zeros(moe.moe_experts_decode_workspace(T, k, s), dtype=torch.uint8, device="cuda")
    y = torch.empty(T, H, dtype=torch.float32, device="cuda")
    x_out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    idx, w = [], []
    for l in range(L):
        b = bias[l] if bias is not None else None
        if l == 0:
            _, i, ww, lg, _ = moe.moe_decode_layer(wr[l], b, k, ptrs[l], s, x=x0, y=y, workspace=ws)
        else:
            _, i, ww, lg, _ = moe.moe_decode_layer(wr[l], b, k, ptrs[l], s, y_prev=y, eps=eps, x_out=x_out, y=y,
                                                   workspace=ws)
        idx.append(i.clone())
        w.append(ww.clone())
    return torch.stack(idx), torch.stack(w), lg, x_out, y


def _gave_up(ws):
    """The first wait that gave up, as recorded in the workspace header."""
    v = int(ws[192:200].cpu().numpy().view(np.uint64)[0])
    return {"site": v >> 56, "layer": ((v >> 32) & 0xFFFFFF) - 1, "block": v & 0xFFFFFFFF} if v else None


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


# the decode shape; two tokens with a router bias; MXFP4 with three tokens;
# 512 experts, whose router rows are read from global memory rather than
# staged in shared memory
@pytest.mark.parametrize("fmt,H,I,E,k,T,L", [(0, 2560, 640, 64, 10, 1, 6), (0, 1024, 512, 64, 8, 2, 3),
                                             (1, 512, 256, 32, 4, 3, 4), (0, 512, 256, 512, 4, 1, 3)])
def test_stack_equals_per_layer_launches(fmt, H, I, E, k, T, L):
    pools = [Pool(E, H, I, fmt, workload=60 + fmt, layer=l) for l in range(L)]
    s = pools[0].shape
    wr = torch.stack([synth.router_weights(E, H, 6000 + l) for l in range(L)]).cuda()
    ptrs = torch.stack([p.ptrs for p in pools])
    bias = synth.zipf_bias(E, 61).cuda().repeat(L, 1) if T == 2 else None
    x0 = synth.activations(T, H, 6100 + T).cuda()
    ref = _per_layer(x0, wr, ptrs, s, k, bias)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(moe.moe_experts_decode_workspace(T, k, s), dtype=torch.uint8, device="cuda")
    got = moe.moe_decode_stack(x0, wr, bias, k, ptrs, s, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, _gave_up(ws)
    x_out, idx, w, lg, y = got
    assert torch.equal(idx, ref[0])
    assert torch.equal(_bits(w), _bits(ref[1]))
    assert torch.equal(_bits(lg), _bits(ref[2]))
    assert torch.equal(_bits(x_out), _bits(ref[3]))
    assert torch.equal(_bits(y), _bits(ref[4]))
    assert torch.isfinite(y).all()
    # repeated launches on one workspace give the same bits
    got2 = moe.moe_decode_stack(x0, wr, bias, k, ptrs, s)
    assert torch.equal(_bits(got2[4]), _bits(y))


def test_stack_barrier_wait_runs_out_then_next_call_is_exact():
    E, H, I, k, T, L = 16, 256, 128, 4, 2, 5
    pools = [Pool(E, H, I, 0, workload=62, layer=l) for l in range(L)]
    s = pools[0].shape
    wr = torch.stack([synth.router_weights(E, H, 6200 + l) for l in range(L)]).cuda()
    ptrs = torch.stack([p.ptrs for p in pools])
    x0 = synth.activations(T, H, 6300).cuda()
    ref = _per_layer(x0, wr, ptrs, s, k)
    ws = torch.zeros(moe.moe_experts_decode_workspace(T, k, s), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_test_set_wait_limit(200_000, 1)
    try:
        bad = moe.moe_decode_stack(x0, wr, None, k, ptrs, s, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        moe.moe_test_set_wait_limit(0, 0)
    assert int(st.item()) & moe.DEV_TIMEOUT
    assert torch.isnan(bad[4]).all()
    # the extra arrival moves every grid-barrier target: the first to give up
    # is the router's barrier of layer 0
    assert _gave_up(ws) is not None and _gave_up(ws)["site"] == 5 and _gave_up(ws)["layer"] == 0
    ws.zero_()
    st.zero_()
    got = moe.moe_decode_stack(x0, wr, None, k, ptrs, s, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(_bits(got[4]), _bits(ref[4]))
