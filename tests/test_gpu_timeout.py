"""The bounded waits of the one-shot decode kernel run out cleanly.

A test hook shortens every wait to 200 us and makes each grid barrier expect
one arrival more than the grid makes, so the barriers cannot complete.  The
launch must end by itself, set MOE_DEV_TIMEOUT, write NaN outputs and leave
the GPU usable: the next call on a zeroed workspace, with the hook reset, must
give the normal result.  Nothing here traps, faults or waits without a limit.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    return Pool(16, 256, 128, 0, workload=41)


@pytest.mark.parametrize("fused", [True, False])
def test_barrier_wait_runs_out_then_next_call_is_correct(pool, fused):
    k, T, H = 4, 2, pool.H
    x = synth.activations(T, H, 4100).cuda()
    wr = synth.router_weights(pool.E, H, 4101).cuda()
    idx, w, _ = moe.moe_router_topk(x, wr, None, k)
    ref = moe.moe_experts_decode(x, idx, w, pool.ptrs, pool.shape)
    torch.cuda.synchronize()
    ws = torch.zeros(moe.moe_experts_decode_workspace(T, k, pool.shape), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        if fused:
            return moe.moe_decode_layer(wr, None, k, pool.ptrs, pool.shape, x=x, workspace=ws, dev_status=st)[4]
        return moe.moe_experts_decode(x, idx, w, pool.ptrs, pool.shape, workspace=ws, dev_status=st)

    moe.moe_test_set_wait_limit(200_000, 1)
    try:
        y_bad = run()
        torch.cuda.synchronize()
    finally:
        moe.moe_test_set_wait_limit(0, 0)
    assert int(st.item()) & moe.DEV_TIMEOUT
    assert torch.isnan(y_bad).all()

    ws.zero_()
    st.zero_()
    y = run()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))

