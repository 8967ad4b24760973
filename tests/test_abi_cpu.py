"""The C-ABI library builds, loads and exports what include/moe.h declares.

No GPU: only host-side functions (record geometry, status strings, argument
validation that returns before any CUDA call) are executed.
"""
import ctypes
import os
import re
import subprocess

import pytest

from block_scaled_fp4_softmax_gb300 import build, moe
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    skip = {"if", "for", "while", "return", "sizeof"}
    return sorted({n for n in names if n not in skip})


def test_header_declares_the_binding_names():
    assert set(_declared()) == set(moe.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_record_geometry_matches_oracle(lib):
    for H, I, fmt in ((2560, 640, 0), (4096, 2880, 1), (64, 64, 0), (128, 64, 1)):
        s = moe.shape(H, I, fmt)
        assert moe.moe_expert_record_bytes(s) == O.record_bytes(H, I, fmt)
        assert moe.moe_expert_record_offsets(s) == O.record_layout(H, I, fmt)


def test_unsupported_shapes_report_zero(lib):
    assert moe.moe_expert_record_bytes(moe.shape(100, 64, 0)) == 0
    assert moe.moe_expert_record_bytes(moe.shape(64, 64, 7)) == 0


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert moe.moe_status_string(4) == "workspace too small"
    assert moe.moe_status_string(99) == "unknown status"


def test_argument_validation_before_any_cuda_call(lib):
    s = moe.shape(2560, 640, 0)
    vp = ctypes.c_void_p
    # NULL outputs -> invalid argument
    assert lib.moe_router_topk(None, None, None, 1, 2560, 64, 10, None, None, None, None) == 1
    # k > E
    one = vp(16)
    assert lib.moe_router_topk(one, one, None, 1, 2560, 8, 10, one, one, one, None) == 1
    # misaligned x
    assert lib.moe_router_topk(vp(18), one, None, 1, 2560, 64, 10, one, one, one, None) == 2
    # decode: workspace too small
    assert lib.moe_experts_decode(one, one, one, 1, 10, one, 64, s, one, one, 16, None,
                                  None) == 4
    # decode: unsupported shape
    assert lib.moe_experts_decode(one, one, one, 1, 10, one, 64, moe.shape(100, 64, 0), one, one,
                                  1 << 20, None, None) == 3
    assert lib.fp8_rowscale_gemv(one, one, one, 4, 24, one, None) == 3
    assert lib.fp4_pack_expert(one, one, vp(20), s, one, None) == 2
    # counters header, then 1024 tagged 8-byte logits per token, then FP32 h
    # [T*k][I] (the other decode paths keep theirs right after the header)
    assert moe.moe_experts_decode_workspace(1, 10, s) == 16640 + 1024 * 8 + 10 * 640 * 4
    assert moe.moe_experts_decode_workspace(32, 10, s) == 16640 + 32 * 1024 * 8 + 32 * 10 * 640 * 4


def test_wait_limit_hook_rejects_bad_values(lib):
    # host-side checks only; (0, 0) restores the defaults
    assert lib.moe_test_set_wait_limit(10, 0) == 1            # below 1 us
    assert lib.moe_test_set_wait_limit(200_000, 2) == 1       # only 0 or 1 extra arrival
    assert lib.moe_test_set_wait_limit(0, 0) == 0
