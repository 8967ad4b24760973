"""Plain CPU oracle for the routed-MoE FFN with block-scaled FP4 experts.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  The
library (the CUDA path) never imports it and shares no code with it.

Written from three pages on streaming MoE experts to a small GPU:

* "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
  experts from NVMe" (aiwithghost.com) -- called *Qwen page* below;
* "Running the 510 GB DeepSeek-V4.1-Flash on an 8 GB GPU, and three bugs that
  never raise an error" (dev.to) -- called *DeepSeek page*;
* the clawdbytes.com summary of the DeepSeek page.

Everything is computed in the plainest form: dense dequantised matrices in
float64, numpy matmul as the only library step, and explicit per-element
definitions for the encodings.  Where the pages leave a step open the reading
taken is stated at the function.

Pins (tests/test_oracle_*.py, CPU only) tie each function to something other
than itself: hand-worked code tables, byte counts printed on the pages, torch's
own float8/bfloat16 conversions, brute force on tiny inputs, and invariants.
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Formats
# ---------------------------------------------------------------------------

FMT_NVFP4 = 0  # e2m1 codes, one FP8 E4M3 scale per 16 elements
FMT_MXFP4 = 1  # e2m1 codes, one UE8M0 (power of two) scale per 32 elements


def block_size(fmt: int) -> int:
    return 16 if fmt == FMT_NVFP4 else 32


def e2m1_decode(codes) -> np.ndarray:
    """Value of 4-bit e2m1 codes (Qwen page, "The engine" item 4: the FP4
    e2m1 format the expert kernel converts with the hardware e2m1 cvt).

    Bit 3 is the sign, bits 2..1 the exponent (bias 1), bit 0 the mantissa.
    Exponent field 0 is subnormal: value = m * 0.5.  Otherwise
    value = 2**(e-1) * (1 + m/2).
    """
    c = np.asarray(codes, dtype=np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return sign * mag


def e4m3_decode(b) -> np.ndarray:
    """Value of OCP FP8 E4M3FN bytes (the per-16 block scale of NVFP4).

    Sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.  Exponent 0
    is subnormal: m/8 * 2**-6.  0x7F / 0xFF are NaN; there is no infinity, so
    the largest finite value is 0x7E = 448.
    """
    v = np.asarray(b, dtype=np.int64) & 0xFF
    sign = np.where(v & 0x80, -1.0, 1.0)
    e = (v >> 3) & 0xF
    m = v & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    out = sign * mag
    return np.where((v & 0x7F) == 0x7F, np.nan, out)


def ue8m0_decode(b) -> np.ndarray:
    """Value of UE8M0 scale bytes: 2**(s-127); 0xFF is NaN (the DeepSeek page,
    "Three bugs" item 2, names this ue8m0 scale format)."""
    v = np.asarray(b, dtype=np.int64) & 0xFF
    return np.where(v == 0xFF, np.nan, np.ldexp(1.0, v - 127))


def _rn_even_on_grid(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index into an ascending non-negative grid of the nearest point to
    ``mag`` (>= 0), ties going to the even index; values above the top of the
    grid saturate to the top (satfinite).

    With mid[m] = (grid[m] + grid[m+1]) / 2 (exact in binary), the nearest
    index is the number of midpoints strictly below ``mag``; when ``mag``
    equals a midpoint the two neighbours m and m+1 tie and the even one wins.
    """
    mids = (grid[:-1] + grid[1:]) / 2
    below = np.searchsorted(mids, mag, side="left")       # #mids < mag
    at = np.minimum(below, len(mids) - 1)
    tie = mids[at] == mag
    return np.where(tie & (below % 2 == 1), below + 1, below)


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E4M3_GRID = e4m3_decode(np.arange(0, 127))  # codes 0..126, ascending, finite


def e2m1_encode(v) -> np.ndarray:
    """Round float values to e2m1 codes: nearest, ties to even, |v| > 6
    saturates to 6.  The sign is kept, so a negative value that rounds to zero
    gives code 8 (-0)."""
    v = np.asarray(v)
    mag_code = _rn_even_on_grid(np.abs(v), _E2M1_GRID).astype(np.uint8)
    return mag_code | (np.signbit(v).astype(np.uint8) << 3)


def e4m3_encode(v) -> np.ndarray:
    """Round float values to E4M3FN bytes: nearest, ties to even, |v| > 448
    saturates to 448 (satfinite).  Sign kept."""
    v = np.asarray(v)
    mag_code = _rn_even_on_grid(np.abs(v), _E4M3_GRID).astype(np.uint8)
    return mag_code | (np.signbit(v).astype(np.uint8) << 7)


# ---------------------------------------------------------------------------
# BF16 helpers (bit patterns carried as uint16)
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest BF16 value (ties to even), in one
    rounding step; returned as float64 holding the BF16 value."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0) & np.isfinite(v)
    a = np.abs(v[nz])
    ex = np.floor(np.log2(a)).astype(np.int64)
    # correct floor(log2) at exact powers and rounding edges of log2 itself
    ex = np.where(np.ldexp(1.0, ex) > a, ex - 1, ex)
    ex = np.where(np.ldexp(1.0, ex + 1) <= a, ex + 1, ex)
    quantum_exp = np.maximum(ex - 7, -133)  # 8 significant bits; subnormal floor
    q = np.rint(np.ldexp(a, -quantum_exp))  # exact scaling, rint = ties-to-even
    r = np.ldexp(q, quantum_exp)
    r = np.where(r >= np.ldexp(2.0 - 2.0 ** -8, 127), np.inf, r)
    out[nz] = np.sign(v[nz]) * r
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    out[v == 0] = v[v == 0]
    return out


def bf16_round_bits(v) -> np.ndarray:
    r = bf16_round(v).astype(np.float32)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Expert record (Qwen page, "The engine" item 1; DeepSeek page, "The approach")
# ---------------------------------------------------------------------------

def record_layout(H: int, I: int, fmt: int) -> dict:
    """Byte offsets of one expert record: gate | up | down | gate_s | up_s |
    down_s, each part plain row-major with K (the input dimension) contiguous.

    gate and up are [I x H], down is [H x I].  Codes pack two elements per
    byte; scales take one byte per block of 16 (NVFP4) or 32 (MXFP4).
    """
    G = block_size(fmt)
    codes = I * H // 2
    scales = I * H // G
    off = {}
    off["gate"] = 0
    off["up"] = codes
    off["down"] = 2 * codes
    off["gate_s"] = 3 * codes
    off["up_s"] = 3 * codes + scales
    off["down_s"] = 3 * codes + 2 * scales
    off["total"] = 3 * codes + 3 * scales
    return off


def record_bytes(H: int, I: int, fmt: int) -> int:
    return record_layout(H, I, fmt)["total"]


def quantize_matrix(W, fmt: int):
    """Block-quantise one FP32 matrix [rows x K] along K.

    The pages never quantise (they repack vendor files), so the reading is:
    NVFP4, per block of 16: s = E4M3(amax / 6) in FP32 arithmetic; if the
    decoded s is 0 all codes are +0, else code = e2m1(x / s) with an FP32
    divide.  MXFP4, per block of 32: the smallest power of two 2**E with
    6 * 2**E >= amax, stored as s = clamp(E + 127, 0, 254) (amax = 0 gives
    s = 0), then code = e2m1(x * 2**(127 - s)) with an FP32 multiply.
    Returns (codes uint8 [rows x K/2], scales uint8 [rows x K/G]).
    Element 2i goes to the low nibble of byte i, element 2i+1 to the high one.
    """
    W = np.asarray(W, dtype=np.float32)
    rows, K = W.shape
    G = block_size(fmt)
    assert K % G == 0
    blocks = W.reshape(rows, K // G, G)
    amax = np.max(np.abs(blocks), axis=2)  # float32, exact
    if fmt == FMT_NVFP4:
        s_code = e4m3_encode(np.float32(amax) / np.float32(6.0))
        s_code = s_code & 0x7F  # amax >= 0: the sign bit is never set
        s_val = e4m3_decode(s_code).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = blocks / s_val[:, :, None]  # float32 / float32
        codes = e2m1_encode(q)
        codes = np.where(s_val[:, :, None] == 0, 0, codes).astype(np.uint8)
    else:
        amax64 = amax.astype(np.float64)
        E = np.zeros(amax.shape, dtype=np.int64)
        nz = amax64 > 0
        est = np.ceil(np.log2(np.where(nz, amax64, 1.0) / 6.0)).astype(np.int64)
        # exact correction: want the smallest E with 6 * 2**E >= amax
        est = np.where(np.ldexp(6.0, est) < amax64, est + 1, est)
        est = np.where(np.ldexp(6.0, est - 1) >= amax64, est - 1, est)
        E = np.where(nz, est, -1000)
        s_code = np.clip(E + 127, 0, 254).astype(np.uint8)
        mult = np.ldexp(np.float32(1.0), 127 - s_code.astype(np.int64)).astype(np.float32)
        q = blocks * mult[:, :, None]  # float32 * exact power of two
        codes = e2m1_encode(q)
    codes = codes.reshape(rows, K)
    packed = (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), s_code.astype(np.uint8)


def dequantize_matrix(codes, scales, K: int, fmt: int) -> np.ndarray:
    """Dense float64 matrix from packed codes [rows x K/2] and scales
    [rows x K/G]: value = e2m1(code) * scale (the product is exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows = codes.shape[0]
    G = block_size(fmt)
    el = np.empty((rows, K), dtype=np.uint8)
    el[:, 0::2] = codes & 0xF
    el[:, 1::2] = codes >> 4
    vals = e2m1_decode(el)
    sdec = e4m3_decode(scales) if fmt == FMT_NVFP4 else ue8m0_decode(scales)
    return vals * np.repeat(np.asarray(sdec, dtype=np.float64), G, axis=1)


def pack_expert(gate, up, down, fmt: int) -> np.ndarray:
    """One contiguous expert record (uint8) from FP32 gate [I,H], up [I,H],
    down [H,I]."""
    gate = np.asarray(gate, dtype=np.float32)
    up = np.asarray(up, dtype=np.float32)
    down = np.asarray(down, dtype=np.float32)
    I, H = gate.shape
    lay = record_layout(H, I, fmt)
    rec = np.zeros(lay["total"], dtype=np.uint8)
    for name, W in (("gate", gate), ("up", up), ("down", down)):
        c, s = quantize_matrix(W, fmt)
        rec[lay[name]: lay[name] + c.size] = c.ravel()
        rec[lay[name + "_s"]: lay[name + "_s"] + s.size] = s.ravel()
    return rec


def unpack_expert(record, H: int, I: int, fmt: int):
    """Dense float64 (gate [I,H], up [I,H], down [H,I]) from one record."""
    rec = np.asarray(record, dtype=np.uint8)
    lay = record_layout(H, I, fmt)
    G = block_size(fmt)
    out = []
    for name, rows, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        c = rec[lay[name]: lay[name] + rows * K // 2].reshape(rows, K // 2)
        s = rec[lay[name + "_s"]: lay[name + "_s"] + rows * K // G].reshape(rows, K // G)
        out.append(dequantize_matrix(c, s, K, fmt))
    return tuple(out)


# ---------------------------------------------------------------------------
# Router (Qwen page, "Why this model": top-10 of 512 per layer; DeepSeek page,
# "Bytes per token": 6 of 384)
# ---------------------------------------------------------------------------

def router_logits(x_bits, wr_bits, bias=None) -> np.ndarray:
    """FP32 router logits in the fixed summation order the library documents.

    logit[t,e] = sum_h x[t,h] * W_r[e,h] (+ bias[e]).  x and W_r are BF16, so
    each product is exact in FP32 and only the order of the FP32 additions
    matters.  Order: the K axis is cut into chunks of 8 elements; chunk c
    belongs to slot c mod 32.  Each of the 32 slots sums its chunks in
    ascending order, elements within a chunk ascending, starting from +0.
    Then five pairwise rounds combine slot i with slot i xor d for
    d = 16, 8, 4, 2, 1, and slot 0's value is the sum; the bias is added last.
    Fixing the order makes the top-k choice reproducible bit for bit.
    """
    x = bf16_bits_to_f32(x_bits)
    w = bf16_bits_to_f32(wr_bits)
    T, H = x.shape
    E = w.shape[0]
    assert H % 8 == 0
    nchunk = H // 8
    acc = np.zeros((T, E, 32), dtype=np.float32)
    for m in range((nchunk + 31) // 32):
        lanes = np.arange(32)
        c = 32 * m + lanes
        ok = c < nchunk
        lanes, c = lanes[ok], c[ok]
        for i in range(8):
            h = 8 * c + i
            prod = x[:, None, h] * w[None, :, h]  # exact in float32
            acc[:, :, lanes] = acc[:, :, lanes] + prod
    for d in (16, 8, 4, 2, 1):
        acc = acc + acc[:, :, np.arange(32) ^ d]
    out = acc[:, :, 0].copy()
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float32)[None, :]
    return out


def router_logits_f64(x_bits, wr_bits, bias=None) -> np.ndarray:
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    w = bf16_bits_to_f32(wr_bits).astype(np.float64)
    out = x @ w.T
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)[None, :]
    return out


def topk_softmax(logits, k: int):
    """Top-k experts per token and their renormalised softmax weights.

    Order: larger logit first, ties to the lower expert index, NaN last.
    Weights: w_j = exp(l_j - l_max) / sum over the k selected of
    exp(l_i - l_max) -- the softmax over all experts restricted to the top-k
    and renormalised to sum to one (the pages name only "router softmax /
    top-k"; renormalisation is the reading taken).  Returns idx int32 [T,k]
    and weights float64 [T,k].
    """
    L = np.asarray(logits, dtype=np.float32)
    T, E = L.shape
    idx = np.zeros((T, k), dtype=np.int32)
    wts = np.zeros((T, k), dtype=np.float64)
    ar = np.arange(E)
    for t in range(T):
        row = L[t].astype(np.float64)
        isn = np.isnan(row)
        key = np.where(isn, 0.0, -row)
        order = np.lexsort((ar, key, isn))
        sel = order[:k]
        idx[t] = sel
        ls = row[sel]
        ex = np.exp(ls - ls[0])
        wts[t] = ex / ex.sum()
    return idx, wts


# ---------------------------------------------------------------------------
# Bucketing (Qwen page, "The engine" item 5: the whole prompt goes through a
# layer at once; DeepSeek page, "v3": each expert's tokens are found by
# comparing the index tensor against the expert)
# ---------------------------------------------------------------------------

def bucket_by_expert(idx, E: int):
    """counts [E], offsets [E+1] (exclusive scan) and pairs [T*k]: the flat
    pair ids p = t*k + j grouped by expert, in ascending p inside a group."""
    flat = np.asarray(idx, dtype=np.int64).ravel()
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    pairs = np.argsort(flat, kind="stable").astype(np.int32)
    return counts, offsets, pairs


# ---------------------------------------------------------------------------
# Expert FFN (Qwen page, "The engine" item 4: NVFP4 SwiGLU expert kernel)
# ---------------------------------------------------------------------------

def silu(g):
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def moe_layer_decode(x_bits, idx, weights, records, H: int, I: int, fmt: int, experts=None) -> np.ndarray:
    """y[t] = sum_j w[t,j] * down_e (silu(gate_e x_t) * up_e x_t), e = idx[t,j].

    float64 throughout on the exactly dequantised weights; y returned as
    float32.  ``records`` maps expert id -> record bytes.  ``experts``, if
    given, restricts the sum to the pairs routed to those experts (the
    others contribute nothing), so that callers can split the work.
    """
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    T = x.shape[0]
    idx = np.asarray(idx)
    w = np.asarray(weights, dtype=np.float64)
    y = np.zeros((T, H), dtype=np.float64)
    keep = None if experts is None else {int(e) for e in experts}
    cache = {}
    for t in range(T):
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            if keep is not None and e not in keep:
                continue
            if e not in cache:
                cache[e] = unpack_expert(records[e], H, I, fmt)
            Wg, Wu, Wd = cache[e]
            g = Wg @ x[t]
            u = Wu @ x[t]
            h = silu(g) * u
            y[t] += w[t, j] * (Wd @ h)
    return y.astype(np.float32)


def moe_layer_grouped(x_bits, idx, weights, records, H: int, I: int, fmt: int) -> np.ndarray:
    """The prompt-path variant: gate and up results are rounded to FP32, the
    SwiGLU product silu(g)*u is rounded once to BF16 (the tensor-core path
    feeds it to the down projection as a BF16 operand), then down and the
    weighted sum follow in float64; y returned as float32."""
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    T = x.shape[0]
    idx = np.asarray(idx)
    w = np.asarray(weights, dtype=np.float64)
    y = np.zeros((T, H), dtype=np.float64)
    cache = {}
    for t in range(T):
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            if e not in cache:
                cache[e] = unpack_expert(records[e], H, I, fmt)
            Wg, Wu, Wd = cache[e]
            g = (Wg @ x[t]).astype(np.float32).astype(np.float64)
            u = (Wu @ x[t]).astype(np.float32).astype(np.float64)
            h = bf16_round(silu(g) * u)
            y[t] += w[t, j] * (Wd @ h)
    return y.astype(np.float32)


def moe_layer_grouped_by_expert(x_bits, idx, weights, records, H: int, I: int, fmt: int,
                                tokens=None, experts=None) -> np.ndarray:
    """Same result as ``moe_layer_grouped`` computed expert by expert with
    matrix products (for prompt-sized inputs).  ``tokens`` restricts the
    returned rows to a sample of tokens (the others are left zero);
    ``experts`` restricts the sum to the pairs routed to those experts."""
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    T = x.shape[0]
    idx = np.asarray(idx)
    w = np.asarray(weights, dtype=np.float64)
    want = np.ones(T, dtype=bool) if tokens is None else np.isin(np.arange(T), tokens)
    y = np.zeros((T, H), dtype=np.float64)
    chosen = np.unique(idx[want])
    if experts is not None:
        chosen = np.intersect1d(chosen, np.asarray(list(experts), dtype=chosen.dtype))
    for e in chosen:
        ts, js = np.nonzero((idx == e) & want[:, None])
        Wg, Wu, Wd = unpack_expert(records[int(e)], H, I, fmt)
        X = x[ts]
        g = (X @ Wg.T).astype(np.float32).astype(np.float64)
        u = (X @ Wu.T).astype(np.float32).astype(np.float64)
        h = bf16_round(silu(g) * u)
        o = h @ Wd.T
        np.add.at(y, ts, w[ts, js][:, None] * o)
    return y.astype(np.float32)


def rms_sumsq_fixed_order(y) -> np.ndarray:
    """The FP32 sum of squares of each row of y in the one fixed order of the
    RMS-chaining reading below: 256 strided partial sums (partial t adds
    y[t + 256 m]^2 for m ascending, each square rounded to FP32, then added),
    then a pairwise tree that adds partial t + w into partial t for
    w = 128, 64, ..., 1.  Returns float32 [T]."""
    y = np.asarray(y, dtype=np.float32)
    T, H = y.shape
    part = np.zeros((T, 256), dtype=np.float32)
    for m in range((H + 255) // 256):
        seg = y[:, 256 * m: 256 * (m + 1)]
        n = seg.shape[1]
        part[:, :n] = part[:, :n] + seg * seg
    w = 128
    while w >= 1:
        part[:, :w] = part[:, :w] + part[:, w: 2 * w]
        w //= 2
    return part[:, 0].copy()


def rms_inv_fixed_order(y, eps: float = 1e-6) -> np.ndarray:
    """The FP32 factor r = 1 / sqrt(mean(y^2) + eps) of each row of y: the
    fixed-order sum of squares, mean = sum / H, then IEEE sqrt and divide;
    eps is rounded to FP32.  Returns float32 [T]."""
    y = np.asarray(y, dtype=np.float32)
    mean = rms_sumsq_fixed_order(y) / np.float32(y.shape[1])
    return np.float32(1.0) / np.sqrt(mean + np.float32(eps))


def rmsnorm_bf16(y, eps: float = 1e-6) -> np.ndarray:
    """Layer-chaining glue for stacked decode: x_next = BF16(y * r) with
    r = 1 / sqrt(mean(y^2) + eps) and no learnable weight.

    The pages only say the next layer's input is the previous output,
    RMS-normalised (Qwen page, "Why this model": 48 layers in a row).  The
    reading taken is FP32 arithmetic in one fixed order (rms_inv_fixed_order),
    so that the BF16 x -- and with it the next layer's routing -- is
    reproducible bit for bit; x = y * r is rounded once to BF16 (ties to
    even).  rmsnorm_bf16_f64 is the plain definition it approximates, within
    one BF16 unit.  Returns BF16 bit patterns (uint16) [T, H]."""
    y = np.asarray(y, dtype=np.float32)
    r = rms_inv_fixed_order(y, eps)
    x = y * r[:, None]
    return bf16_round_bits(x.astype(np.float64))


def rmsnorm_bf16_f64(y, eps: float = 1e-6) -> np.ndarray:
    """The plain definition of the RMS chaining: x = BF16(y / sqrt(mean(y^2)
    + eps)) with the mean, the root and the quotient in float64 and a single
    rounding to BF16.  Returns BF16 bit patterns (uint16) [T, H]."""
    y = np.asarray(y, dtype=np.float64)
    ms = np.mean(y * y, axis=1, keepdims=True)
    return bf16_round_bits(y / np.sqrt(ms + float(eps)))


# ---------------------------------------------------------------------------
# FP8 row-scaled matrix-vector (Qwen page, "Why this model" and "The engine"
# item 4: FP8 matrices with one scale per row and their own GEMV kernel)
# ---------------------------------------------------------------------------

def fp8_rowscale_gemv(w_e4m3, row_scale, x_bits) -> np.ndarray:
    """y[m] = s[m] * sum_k e4m3(W[m,k]) * x[k], float64, returned as float32."""
    W = e4m3_decode(np.asarray(w_e4m3, dtype=np.uint8))
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    s = np.asarray(row_scale, dtype=np.float64)
    return (s * (W @ x)).astype(np.float32)


# ---------------------------------------------------------------------------
# Comparisons and byte model
# ---------------------------------------------------------------------------

def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = math.sqrt(float(np.sum(b * b)))
    num = math.sqrt(float(np.sum((a - b) ** 2)))
    return num / den if den > 0 else num


def expert_bytes_per_token(layers: int, k: int, H: int, I: int, fmt: int) -> int:
    """Expert bytes one decoded token reads (Qwen page, "Why this model";
    DeepSeek page, "Bytes per token decide everything")."""
    return layers * k * record_bytes(H, I, fmt)
