"""Thin ctypes binding over the C ABI in include/moe.h.

Each function here carries the C entry point's name and does argument
marshalling only: it checks dtypes/devices, allocates outputs with torch when
the caller passes none, and hands raw device pointers plus the current CUDA
stream to the library.  Every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the compiled library is missing,
or no CUDA device is present, the calls raise.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

FMT_NVFP4 = 0
FMT_MXFP4 = 1

DEV_NULL_EXPERT = 1
DEV_MISALIGNED = 2
DEV_BAD_INDEX = 4
DEV_TIMEOUT = 8
DEV_FP16_RANGE = 16

EXPORTS = (
    "moe_expert_record_bytes",
    "moe_expert_record_offsets",
    "fp4_pack_expert",
    "moe_router_topk",
    "moe_rmsnorm_bf16",
    "moe_rmsnorm_router_topk",
    "moe_experts_decode_workspace",
    "moe_experts_decode",
    "moe_experts_decode_host",
    "moe_decode_layer",
    "moe_decode_stack",
    "moe_experts_decode_noalloc_limit",
    "moe_experts_decode_noalloc",
    "moe_bucket_workspace",
    "moe_bucket_by_expert",
    "moe_experts_grouped_workspace",
    "moe_experts_grouped",
    "fp8_rowscale_gemv",
    "moe_status_string",
    "moe_test_set_wait_limit",
)


class MoeError(RuntimeError):
    pass


class ExpertShape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("format", ctypes.c_int32)]

    def __repr__(self):
        return f"ExpertShape(H={self.hidden}, I={self.inter}, fmt={self.format})"


_LIB = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_SIGS = {
    "moe_expert_record_bytes": (_sz, [ExpertShape]),
    "moe_expert_record_offsets": (_i, [ExpertShape, ctypes.POINTER(ctypes.c_size_t)]),
    "fp4_pack_expert": (_i, [_vp, _vp, _vp, ExpertShape, _vp, _vp]),
    "moe_router_topk": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "moe_rmsnorm_bf16": (_i, [_vp, _i, _i, ctypes.c_double, _vp, _vp]),
    "moe_rmsnorm_router_topk": (_i, [_vp, _i, _i, ctypes.c_double, _vp, _vp, _vp, _i, _i, _vp, _vp,
                                     _vp, _vp]),
    "moe_experts_decode_workspace": (_sz, [_i, _i, ExpertShape]),
    "moe_experts_decode": (_i, [_vp, _vp, _vp, _i, _i, _vp, _i, ExpertShape, _vp, _vp, _sz,
                                _vp, _vp]),
    "moe_experts_decode_host": (_i, [_vp, _vp, _vp, _i, _i, _vp, _i, ExpertShape, _vp, _vp, _sz,
                                     _vp, _vp]),
    "moe_decode_layer": (_i, [_vp, _vp, _i, ctypes.c_double, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp,
                              ExpertShape, _vp, _vp, _sz, _vp, _vp]),
    "moe_decode_stack": (_i, [_vp, _i, ctypes.c_double, _i, _vp, _vp, _i, _i, _vp, ExpertShape, _vp, _vp, _vp,
                              _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_experts_decode_noalloc_limit": (_sz, []),
    "moe_experts_decode_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _vp, _i, ExpertShape, _vp, _vp, _vp]),
    "moe_bucket_workspace": (_sz, [_i, _i, _i]),
    "moe_bucket_by_expert": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_experts_grouped_workspace": (_sz, [_i, _i, _i, ExpertShape]),
    "moe_experts_grouped": (_i, [_vp, _vp, _vp, _i, _i, _vp, _i, ExpertShape, _vp, _vp, _sz,
                                 _vp, _vp]),
    "fp8_rowscale_gemv": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_i]),
    "moe_test_set_wait_limit": (_i, [ctypes.c_ulonglong, _i]),
}


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load (once) the compiled library; raise if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        raise MoeError(f"CUDA library not built: {path} is missing "
                       "(run block_scaled_fp4_softmax_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().moe_status_string(rc).decode()
        raise MoeError(f"{what} failed: status {rc} ({msg})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise MoeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise MoeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MoeError(f"{name} must be contiguous")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def shape(hidden: int, inter: int, fmt: int = FMT_NVFP4) -> ExpertShape:
    return ExpertShape(hidden, inter, fmt)


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def moe_expert_record_bytes(s: ExpertShape) -> int:
    return int(load().moe_expert_record_bytes(s))


def moe_expert_record_offsets(s: ExpertShape) -> dict:
    arr = (ctypes.c_size_t * 7)()
    _check(load().moe_expert_record_offsets(s, arr), "moe_expert_record_offsets")
    names = ("gate", "up", "down", "gate_s", "up_s", "down_s", "total")
    return {n: int(v) for n, v in zip(names, arr)}


def fp4_pack_expert(gate, up, down, s: ExpertShape, record=None, stream=None):
    """Quantise/pack one expert; returns the uint8 record tensor."""
    for n, t in (("gate", gate), ("up", up), ("down", down)):
        _cuda(t, n, torch.float32)
    if record is None:
        record = torch.empty(moe_expert_record_bytes(s), dtype=torch.uint8, device=gate.device)
    _cuda(record, "record", torch.uint8)
    _check(load().fp4_pack_expert(_ptr(gate), _ptr(up), _ptr(down), s, _ptr(record),
                                  _stream(stream)), "fp4_pack_expert")
    return record


def moe_router_topk(x, wr, bias, k: int, idx=None, weights=None, logits=None, stream=None):
    """Returns (idx int32 [T,k], weights fp32 [T,k], logits fp32 [T,E])."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(wr, "wr", torch.bfloat16)
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    T, H = x.shape
    E = wr.shape[0]
    dev = x.device
    if idx is None:
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(T, k, dtype=torch.float32, device=dev)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    _check(load().moe_router_topk(_ptr(x), _ptr(wr), _ptr(bias), T, H, E, k, _ptr(idx),
                                  _ptr(weights), _ptr(logits), _stream(stream)), "moe_router_topk")
    return idx, weights, logits


def moe_rmsnorm_bf16(y, eps: float = 1e-6, x=None, stream=None):
    _cuda(y, "y", torch.float32)
    T, H = y.shape
    if x is None:
        x = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check(load().moe_rmsnorm_bf16(_ptr(y), T, H, float(eps), _ptr(x), _stream(stream)),
           "moe_rmsnorm_bf16")
    return x


def moe_rmsnorm_router_topk(y_prev, wr, bias, k: int, eps: float = 1e-6, x_out=None, idx=None,
                            weights=None, logits=None, stream=None):
    """RMS chaining of y_prev fused with the router; returns (x, idx, weights, logits)."""
    _cuda(y_prev, "y_prev", torch.float32)
    _cuda(wr, "wr", torch.bfloat16)
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    T, H = y_prev.shape
    E = wr.shape[0]
    dev = y_prev.device
    if x_out is None:
        x_out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if idx is None:
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(T, k, dtype=torch.float32, device=dev)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    _check(load().moe_rmsnorm_router_topk(_ptr(y_prev), T, H, float(eps), _ptr(x_out), _ptr(wr),
                                          _ptr(bias), E, k, _ptr(idx), _ptr(weights), _ptr(logits),
                                          _stream(stream)), "moe_rmsnorm_router_topk")
    return x_out, idx, weights, logits


def moe_experts_decode_workspace(T: int, k: int, s: ExpertShape) -> int:
    return int(load().moe_experts_decode_workspace(T, k, s))


def pointer_table(records, device=None):
    """Device int64 array of record addresses (expert id -> record)."""
    addrs = [0 if r is None else r.data_ptr() for r in records]
    dev = device or next(r.device for r in records if r is not None)
    return torch.tensor(addrs, dtype=torch.int64, device=dev)


def moe_decode_layer(wr, bias, k: int, ptrs, s: ExpertShape, x=None, y_prev=None, eps: float = 1e-6,
                     x_out=None, idx=None, weights=None, logits=None, y=None, workspace=None,
                     dev_status=None, stream=None):
    """Router and expert pass of one decode layer in one launch; exactly one of
    x (BF16) and y_prev (FP32, RMS-chained into x_out) is given.  Returns
    (x_out, idx, weights, logits, y)."""
    if (x is None) == (y_prev is None):
        raise ValueError("give exactly one of x and y_prev")
    src = x if x is not None else y_prev
    if x is not None:
        _cuda(x, "x", torch.bfloat16)
    else:
        _cuda(y_prev, "y_prev", torch.float32)
    _cuda(wr, "wr", torch.bfloat16)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    T, H = src.shape
    E = wr.shape[0]
    dev = src.device
    if x_out is None and y_prev is not None:
        x_out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if idx is None:
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(T, k, dtype=torch.float32, device=dev)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty(T, H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(moe_experts_decode_workspace(T, k, s), 16), dtype=torch.uint8, device=dev)
    _check(load().moe_decode_layer(_ptr(x), _ptr(y_prev), T, float(eps), _ptr(x_out), _ptr(wr), _ptr(bias),
                                   E, k, _ptr(idx), _ptr(weights), _ptr(logits), _ptr(ptrs), s, _ptr(y),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(dev_status), _stream(stream)), "moe_decode_layer")
    return x_out, idx, weights, logits, y


def moe_decode_stack(x0, wr, bias, k: int, ptrs, s: ExpertShape, eps: float = 1e-6, idx=None, weights=None,
                     logits=None, x_out=None, y=None, workspace=None, dev_status=None, stream=None):
    """All layers of a decode stack in one launch.  wr [L, E, H] BF16, ptrs
    [L, E] int64 record addresses, bias [L, E] or None.  Returns
    (x_out, idx [L, T, k], weights [L, T, k], logits [T, E], y [T, H])."""
    _cuda(x0, "x0", torch.bfloat16)
    _cuda(wr, "wr", torch.bfloat16)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    T, H = x0.shape
    layers, E = wr.shape[0], wr.shape[1]
    dev = x0.device
    if idx is None:
        idx = torch.empty(layers, T, k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(layers, T, k, dtype=torch.float32, device=dev)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    if x_out is None:
        x_out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if y is None:
        y = torch.empty(T, H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(moe_experts_decode_workspace(T, k, s), 16), dtype=torch.uint8, device=dev)
    _check(load().moe_decode_stack(_ptr(x0), T, float(eps), layers, _ptr(wr), _ptr(bias), E, k, _ptr(ptrs), s,
                                   _ptr(idx), _ptr(weights), _ptr(logits), _ptr(x_out), _ptr(y), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                   _stream(stream)), "moe_decode_stack")
    return x_out, idx, weights, logits, y


def moe_experts_decode(x, idx, weights, ptrs, s: ExpertShape, y=None, workspace=None,
                       dev_status=None, stream=None):
    _cuda(x, "x", torch.bfloat16)
    _cuda(idx, "idx", torch.int32)
    _cuda(weights, "weights", torch.float32)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    T, k = idx.shape
    H = x.shape[1]
    if y is None:
        y = torch.empty(T, H, dtype=torch.float32, device=x.device)
    if workspace is None:
        nbytes = max(moe_experts_decode_workspace(T, k, s), 16)
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=x.device)
    _check(load().moe_experts_decode(_ptr(x), _ptr(idx), _ptr(weights), T, k, _ptr(ptrs),
                                     ptrs.numel(), s, _ptr(y), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(dev_status), _stream(stream)), "moe_experts_decode")
    return y


def moe_experts_decode_host(x, idx, weights, ptrs, s: ExpertShape, y=None, workspace=None,
                            dev_status=None, stream=None):
    """Expert pass over records that may sit in host memory the device can
    address (pinned, or Grace memory over NVLink-C2C); plain loads only."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(idx, "idx", torch.int32)
    _cuda(weights, "weights", torch.float32)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    T, k = idx.shape
    H = x.shape[1]
    if y is None:
        y = torch.empty(T, H, dtype=torch.float32, device=x.device)
    if workspace is None:
        nbytes = max(moe_experts_decode_workspace(T, k, s), 16)
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=x.device)
    _check(load().moe_experts_decode_host(_ptr(x), _ptr(idx), _ptr(weights), T, k, _ptr(ptrs),
                                          ptrs.numel(), s, _ptr(y), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _ptr(dev_status), _stream(stream)), "moe_experts_decode_host")
    return y


def moe_experts_decode_noalloc_limit() -> int:
    return int(load().moe_experts_decode_noalloc_limit())


def moe_experts_decode_noalloc(x, idx, weights, ptrs, s: ExpertShape, y, dev_status=None,
                               stream=None):
    """Decode with the library's static scratch: the caller passes the output
    buffer ``y`` too, and nothing is allocated on either side."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(idx, "idx", torch.int32)
    _cuda(weights, "weights", torch.float32)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    _cuda(y, "y", torch.float32)
    T, k = idx.shape
    _check(load().moe_experts_decode_noalloc(_ptr(x), _ptr(idx), _ptr(weights), T, k, _ptr(ptrs),
                                             ptrs.numel(), s, _ptr(y), _ptr(dev_status),
                                             _stream(stream)), "moe_experts_decode_noalloc")
    return y


def moe_bucket_workspace(T: int, k: int, E: int) -> int:
    return int(load().moe_bucket_workspace(T, k, E))


def moe_bucket_by_expert(idx, E: int, counts=None, offsets=None, pairs=None, workspace=None,
                         dev_status=None, stream=None):
    _cuda(idx, "idx", torch.int32)
    T, k = idx.shape
    dev = idx.device
    if counts is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
    if offsets is None:
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if pairs is None:
        pairs = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(moe_bucket_workspace(T, k, E), 16), dtype=torch.uint8,
                                device=dev)
    _check(load().moe_bucket_by_expert(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets),
                                       _ptr(pairs), _ptr(workspace), workspace.numel(),
                                       _ptr(dev_status), _stream(stream)), "moe_bucket_by_expert")
    return counts, offsets, pairs


def moe_experts_grouped_workspace(T: int, k: int, E: int, s: ExpertShape) -> int:
    return int(load().moe_experts_grouped_workspace(T, k, E, s))


def moe_experts_grouped(x, idx, weights, ptrs, s: ExpertShape, y=None, workspace=None,
                        dev_status=None, stream=None):
    _cuda(x, "x", torch.bfloat16)
    _cuda(idx, "idx", torch.int32)
    _cuda(weights, "weights", torch.float32)
    _cuda(ptrs, "expert_ptrs", torch.int64)
    T, k = idx.shape
    H = x.shape[1]
    E = ptrs.numel()
    if y is None:
        y = torch.empty(T, H, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(moe_experts_grouped_workspace(T, k, E, s), 16),
                                dtype=torch.uint8, device=x.device)
    _check(load().moe_experts_grouped(_ptr(x), _ptr(idx), _ptr(weights), T, k, _ptr(ptrs), E, s,
                                      _ptr(y), _ptr(workspace), workspace.numel(),
                                      _ptr(dev_status), _stream(stream)), "moe_experts_grouped")
    return y


def fp8_rowscale_gemv(w, row_scale, x, y=None, stream=None):
    _cuda(w, "w", torch.uint8)
    _cuda(row_scale, "row_scale", torch.float32)
    _cuda(x, "x", torch.bfloat16)
    M, K = w.shape
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=w.device)
    _check(load().fp8_rowscale_gemv(_ptr(w), _ptr(row_scale), _ptr(x), M, K, _ptr(y),
                                    _stream(stream)), "fp8_rowscale_gemv")
    return y


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_test_set_wait_limit(wait_ns: int = 0, barrier_extra_arrivals: int = 0) -> None:
    """Test hook: the limit of the decode kernels' bounded waits, and one extra
    arrival each grid barrier expects (which no CTA makes, so the barriers run
    out); (0, 0) restores the defaults."""
    _check(load().moe_test_set_wait_limit(int(wait_ns), int(barrier_extra_arrivals)),
           "moe_test_set_wait_limit")
