"""The allocation-free decode entry point, called through the C ABI.

It serves callers that cannot allocate device memory on the decode path (a
plugin handed only its input/output buffers, a loop that must never enter an
allocator).  Its output must match moe_experts_decode's within the decode
tolerance, on consecutive calls that share the library's static scratch.
Collected last on purpose, so a failure here never hides another test."""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp4_softmax_gb300 import build, moe, synth
from helpers import Pool, bits
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _route(T, E, H, k, seed):
    x = synth.activations(T, H, seed)
    wr = synth.router_weights(E, H, seed + 1)
    idx, w = O.topk_softmax(O.router_logits(bits(x), bits(wr)), k)
    return (x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w.astype(np.float32)).cuda())


def _noalloc_c(lib, x, idx, w, pool, y, st):
    T, k = idx.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.moe_experts_decode_noalloc(p(x), p(idx), p(w), T, k, p(pool.ptrs), pool.E,
                                          pool.shape, p(y), p(st),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_decode_on_consecutive_calls():
    build.build()
    lib = moe.load()
    pool = Pool(24, 2560, 640, 0, workload=30)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a fused-path call (1 token) and a two-kernel call (8 tokens), twice each
    cases = [_route(1, 24, 2560, 10, 300), _route(8, 24, 2560, 10, 301)]
    for rnd in range(2):
        for x, idx, w in cases:
            y = torch.full((x.shape[0], 2560), float("nan"), dtype=torch.float32, device="cuda")
            assert _noalloc_c(lib, x, idx, w, pool, y, st) == 0
            ref = moe.moe_experts_decode(x, idx, w, pool.ptrs, pool.shape)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            got = y.cpu().numpy()
            assert np.all(np.isfinite(got))
            err = O.rel_l2(got, ref.cpu().numpy())
            assert err <= TOL, (rnd, x.shape[0], err)


def test_noalloc_rejects_sizes_beyond_its_limit():
    build.build()
    lib = moe.load()
    limit = int(lib.moe_experts_decode_noalloc_limit())
    assert limit == 2 << 20
    s = moe.shape(2560, 640, 0)
    T, k = 100, 10                                    # within decode's limits, 3.4 MB of scratch
    assert moe.moe_experts_decode_workspace(T, k, s) > limit
    one = ctypes.c_void_p(256)
    rc = lib.moe_experts_decode_noalloc(one, one, one, T, k, one, 64, s, one, None, None)
    assert rc == 4
    assert moe.moe_status_string(rc) == "workspace too small"
    # a shape moe_experts_decode rejects gets the same status here (checked
    # before the size, and before the shared array is touched)
    assert lib.moe_experts_decode_noalloc(one, one, one, 1024, 32, one, 64, s, one, None, None) == 3
