"""The host-memory expert tier: records in pinned host memory, read by the
device over its address space (NVLink-C2C on a Grace machine, PCIe elsewhere)
through moe_experts_decode_host.  The result must equal the same call on the
same records in HBM bit for bit, and the oracle within the decode
tolerance."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool, bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,H,I,E,k,T", [(0, 2560, 640, 24, 10, 1), (0, 2560, 640, 24, 10, 3),
                                           (1, 512, 256, 12, 4, 2)])
def test_host_records_equal_hbm_records_and_oracle(fmt, H, I, E, k, T):
    pool = Pool(E, H, I, fmt, workload=50 + fmt)
    nbytes = moe.moe_expert_record_bytes(pool.shape)
    host = torch.empty(E, nbytes, dtype=torch.uint8, pin_memory=True)
    for e in range(E):
        host[e].copy_(pool.record(e))
    torch.cuda.synchronize()
    host_ptrs = torch.tensor([host[e].data_ptr() for e in range(E)], dtype=torch.int64, device="cuda")
    x = synth.activations(T, H, 5000 + T)
    wr = synth.router_weights(E, H, 5001)
    idx, w = O.topk_softmax(O.router_logits(bits(x), bits(wr)), k)
    args = (x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w.astype(np.float32)).cuda())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_host = moe.moe_experts_decode_host(*args, host_ptrs, pool.shape, dev_status=st)
    y_hbm = moe.moe_experts_decode_host(*args, pool.ptrs, pool.shape, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y_host.view(torch.int32), y_hbm.view(torch.int32))
    want = O.moe_layer_decode(bits(x), idx, w, pool.oracle_records(idx.ravel()), H, I, fmt)
    assert O.rel_l2(y_host.cpu().numpy(), want) <= 1e-5
