"""fp4_pack_expert on the GPU vs the oracle packer: byte for byte."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from helpers import Pool
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _pack_both(gate, up, down, fmt):
    H = gate.shape[1]
    I = gate.shape[0]
    s = moe.shape(H, I, fmt)
    rec = moe.fp4_pack_expert(gate.cuda(), up.cuda(), down.cuda(), s)
    want = O.pack_expert(gate.numpy(), up.numpy(), down.numpy(), fmt)
    return rec.cpu().numpy(), want


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("H,I", [(64, 64), (128, 192), (2560, 640)])
def test_pack_byte_exact_random(fmt, H, I):
    g, u, d = synth.expert_weights(H, I, seed=1234 + H + I + fmt)
    got, want = _pack_both(g, u, d, fmt)
    assert got.shape == want.shape
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("fmt", [0, 1])
def test_pack_byte_exact_special_values(fmt):
    H, I = 128, 64
    g, u, d = (t.clone() for t in synth.expert_weights(H, I, seed=77))
    g[0, :] = 0.0                                   # zero blocks
    g[1, :32] = 1e-9                                # NVFP4 scale underflows to 0
    g[2, :32] = -1e-3                               # negative small values
    g[3, :32] = torch.linspace(-7, 7, 32)           # ties on the grid after scaling
    g[4, :] = 1e30                                  # huge (E4M3 scale saturates)
    g[5, :16] = torch.tensor([6.0, 3.0, 1.5, 0.75, 0.25, -0.25, -0.75, 5.0,
                              2.5, 1.25, 0.5, 3.5, -5.0, -2.5, 1.75, 4.0])
    u[0, :] = -0.0
    d[7, :] = torch.tensor(np.float32(2.0) ** -140)  # subnormal FP32 inputs
    got, want = _pack_both(g, u, d, fmt)
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}: " \
                           f"{got[diff[:8]]} vs {want[diff[:8]]}"


def test_pack_mxfp4_deepseek_shape():
    g, u, d = synth.expert_weights(4096, 2880, seed=99)
    got, want = _pack_both(g, u, d, 1)
    assert got.size == 18_800_640
    assert np.array_equal(got, want)


def test_pool_records_match_oracle():
    pool = Pool(4, 2560, 640, 0, workload=0)
    for e in range(4):
        assert np.array_equal(pool.record(e).cpu().numpy(), pool.oracle_record(e))
