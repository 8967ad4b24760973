// Decode path: the selected experts of a few tokens, GEMV shaped and bound by
// the HBM stream of FP4 codes ("Running a 133 GB MoE model on an 8 GB GPU at
// 11 tokens/s by streaming experts from NVMe", section "The engine", item 4:
// the single-token NVFP4 SwiGLU expert kernel built on the hardware e2m1
// convert).
//
// Two kernels per call:
//  1. gate/up + SwiGLU: one warp per (pair, row i); lane j takes the 16-byte
//     code units j, j+32, ... of the gate row followed by the up row, so each
//     warp-wide load is 512 contiguous bytes.  h = silu(g) * u (FP32) goes to
//     the workspace.
//  2. down + weighted combine: one warp per (token, output row n); its lanes
//     walk the k experts' rows n and fold w_j in per unit, so y needs no
//     atomics and is bit-reproducible.
// Activations (x, then h) sit in shared memory as float2 pairs laid out
// [pair-of-elements][unit], so that 32 lanes reading 32 consecutive units
// touch 32 consecutive 8-byte words (no bank conflicts).
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnitBatch = 8;  // 16-byte units each lane keeps in flight

// Sum over one unit: 16 bytes of codes (32 elements) against the float2
// column `xcol` (pair pe of this unit at xcol[pe * stride]), times the block
// scale(s).
template <int FMT>
__device__ __forceinline__ float unit_dot_col(uint4 q, uint32_t sbits, const float2* xcol,
                                              int stride) {
  float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const uint32_t h2 = moe::e2m1x2_to_f16x2((w[wi] >> (8 * bi)) & 0xFFu);
      const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      const float2 xv = xcol[(4 * wi + bi) * stride];
      if (wi < 2) a = moe::ffma2(wf, xv, a);
      else b = moe::ffma2(wf, xv, b);
    }
  }
  if (FMT == MOE_FMT_NVFP4) {
    const float2 s = moe::e4m3x2_to_f32x2(sbits);
    return (a.x + a.y) * s.x + (b.x + b.y) * s.y;
  } else {
    return ((a.x + a.y) + (b.x + b.y)) * moe::ue8m0_to_f32(sbits);
  }
}

template <int FMT>
__device__ __forceinline__ uint32_t load_scale_bits(const uint8_t* sp) {
  if (FMT == MOE_FMT_NVFP4) return (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(sp));
  return (uint32_t)__ldg(sp);
}

// Checks one routed pair; returns the record or nullptr (and flags status).
__device__ __forceinline__ const uint8_t* checked_record(int e, int E, const void* const* ptrs,
                                                         int32_t* st) {
  if (e < 0 || e >= E) {
    moe::status_or(st, MOE_DEV_BAD_INDEX);
    return nullptr;
  }
  const uint8_t* r = reinterpret_cast<const uint8_t*>(ptrs[e]);
  if (!r) {
    moe::status_or(st, MOE_DEV_NULL_EXPERT);
    return nullptr;
  }
  if ((reinterpret_cast<uintptr_t>(r) & 15u) != 0) {
    moe::status_or(st, MOE_DEV_MISALIGNED);
    return nullptr;
  }
  return r;
}

// ---------------------------------------------------------------------------
// 1. gate/up + SwiGLU.  grid = (ceil(I / 8), T*k), 8 warps, warp w -> row
//    i = 8*blockIdx.x + w of pair p = blockIdx.y.
//    h workspace layout per pair: float2 [16][I/32] (same transposed layout
//    as the shared-memory activations of kernel 2).
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_gateup_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ idx, int k,
    const void* const* __restrict__ ptrs, int E, int H, int I, float* __restrict__ hws,
    int32_t* __restrict__ st) {
  extern __shared__ float2 xs2[];  // [16][H/32]
  const int p = blockIdx.y;
  const int t = p / k;
  const int upr = H >> 5;  // 16-byte units per row
  for (int h0 = threadIdx.x * 8; h0 < H; h0 += kThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + h0));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    const int c = h0 >> 5, pe0 = (h0 & 31) >> 1;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xs2[(pe0 + i) * upr + c] =
          make_float2(moe::bf16_bits_to_f32(wv[i] & 0xFFFFu), moe::bf16_bits_to_f32(wv[i] >> 16));
  }
  const uint8_t* rec = checked_record(idx[p], E, ptrs, threadIdx.x == 0 ? st : nullptr);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * (kThreads / 32) + warp;
  if (i >= I) return;
  const int updr = I >> 5;
  float* hp = hws + (size_t)p * I;
  const int hoff = 2 * (((i & 31) >> 1) * updr + (i >> 5)) + (i & 1);
  if (!rec) {
    if (lane == 0) hp[hoff] = __uint_as_float(0x7FC00000u);
    return;
  }
  const moe::RecordOffsets o = moe::record_offsets(H, I, FMT);
  const int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const uint8_t* gcode = rec + o.gate + (size_t)i * (H / 2);
  const uint8_t* ucode = rec + o.up + (size_t)i * (H / 2);
  const uint8_t* gsc = rec + o.gate_s + (size_t)i * (H / G);
  const uint8_t* usc = rec + o.up_s + (size_t)i * (H / G);
  const int sstep = 32 / G;  // scale bytes per unit

  float gacc = 0.f, uacc = 0.f;
  const int nunits = 2 * upr;
  for (int base = 0; base < nunits; base += 32 * kUnitBatch) {
    uint4 q[kUnitBatch];
    uint32_t sb[kUnitBatch];
#pragma unroll
    for (int m = 0; m < kUnitBatch; ++m) {
      const int u = base + lane + 32 * m;
      if (u < nunits) {
        const bool is_up = u >= upr;
        const int c = is_up ? u - upr : u;
        q[m] = moe::ldg_stream((is_up ? ucode : gcode) + 16 * c);
        sb[m] = load_scale_bits<FMT>((is_up ? usc : gsc) + sstep * c);
      }
    }
#pragma unroll
    for (int m = 0; m < kUnitBatch; ++m) {
      const int u = base + lane + 32 * m;
      if (u < nunits) {
        const bool is_up = u >= upr;
        const int c = is_up ? u - upr : u;
        const float d = unit_dot_col<FMT>(q[m], sb[m], xs2 + c, upr);
        if (is_up) uacc += d;
        else gacc += d;
      }
    }
  }
  gacc = moe::warp_sum(gacc);
  uacc = moe::warp_sum(uacc);
  if (lane == 0) {
    const float sg = gacc / (1.0f + expf(-gacc));
    hp[hoff] = sg * uacc;
  }
}

// ---------------------------------------------------------------------------
// 2. down + combine.  grid = (ceil(H / 16), T), 8 warps x 2 rows.
// ---------------------------------------------------------------------------
constexpr int kDownRowsPerWarp = 2;

template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_down_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, int k,
    const void* const* __restrict__ ptrs, int E, int H, int I, const float* __restrict__ hws,
    float* __restrict__ y, int32_t* __restrict__ st) {
  extern __shared__ float2 hs2[];  // [k][16][I/32]
  __shared__ const uint8_t* recs[32];
  __shared__ float wj[32];
  const int t = blockIdx.y;
  const int updr = I >> 5;
  {
    const uint4* src = reinterpret_cast<const uint4*>(hws + (size_t)t * k * I);
    uint4* dst = reinterpret_cast<uint4*>(hs2);
    const int n16 = k * I / 4;
    for (int i = threadIdx.x; i < n16; i += kThreads) dst[i] = src[i];
  }
  if (threadIdx.x < k) {
    recs[threadIdx.x] = checked_record(idx[(size_t)t * k + threadIdx.x], E, ptrs,
                                       blockIdx.x == 0 ? st : nullptr);
    wj[threadIdx.x] = wts[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const moe::RecordOffsets o = moe::record_offsets(H, I, FMT);
  const int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const int sstep = 32 / G;
  const int nunits = k * updr;
#pragma unroll
  for (int r = 0; r < kDownRowsPerWarp; ++r) {
    const int n = (blockIdx.x * (kThreads / 32) + warp) * kDownRowsPerWarp + r;
    if (n >= H) break;
    float acc = 0.f;
    bool bad = false;
    for (int base = 0; base < nunits; base += 32 * kUnitBatch) {
      uint4 q[kUnitBatch];
      uint32_t sb[kUnitBatch];
#pragma unroll
      for (int m = 0; m < kUnitBatch; ++m) {
        const int u = base + lane + 32 * m;
        if (u < nunits) {
          const int j = u / updr, c = u - j * updr;
          const uint8_t* rec = recs[j];
          if (rec) {
            q[m] = moe::ldg_stream(rec + o.down + (size_t)n * (I / 2) + 16 * c);
            sb[m] = load_scale_bits<FMT>(rec + o.down_s + (size_t)n * (I / G) + sstep * c);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kUnitBatch; ++m) {
        const int u = base + lane + 32 * m;
        if (u < nunits) {
          const int j = u / updr, c = u - j * updr;
          if (recs[j]) {
            acc += wj[j] * unit_dot_col<FMT>(q[m], sb[m], hs2 + (size_t)j * 16 * updr + c, updr);
          } else {
            bad = true;
          }
        }
      }
    }
    acc = moe::warp_sum(acc);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) y[(size_t)t * H + n] = bad ? __uint_as_float(0x7FC00000u) : acc;
  }
}

// Raises a kernel's dynamic shared-memory limit once (the attribute call is
// not repeated, so later launches can be captured in a CUDA graph).
// ---------------------------------------------------------------------------
// Streaming expert pass (T*k <= 64): one CTA per SM.  One producer thread
// walks this CTA's share of the selected records -- first the gate/up rows,
// then the down rows -- and moves it with 1-D TMA bulk copies into a ring of
// shared-memory slots, so every byte the CTA needs is requested at kernel
// entry and the HBM pipe stays full.  Fifteen consumer warps compute from
// shared memory: gate/up + SwiGLU rows -> h (global scratch), one grid
// barrier, then down rows against h and the weighted combine, accumulated per
// output row in a fixed order (bit-reproducible).  Slots that hold down rows
// are filled while the consumers still work on gate/up.
// ---------------------------------------------------------------------------
namespace st {

constexpr int kThreads = 512;      // warps 0-14 consume, warp 15 produces
constexpr int kCWarps = 15;
constexpr int kCThreads = kCWarps * 32;
constexpr int kSlots = 6;
constexpr int kSlotBytes = 24576;
constexpr int kMaxChunkUnits = 1536;  // per-chunk partial sums kept in shared memory
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
  const uint16_t* x;
  const int32_t* idx;
  const float* w;
  int T, k;
  const void* const* ptrs;
  int E, H, I;
  float* hws;      // [P][I] FP32, row-major
  unsigned* bar;   // grid barrier words
  float* y;
  int32_t* status;
};

struct Geo {
  int P, upr, updr, ch1, ch2;
  long long r0, r1, q0, q1;  // this CTA's gate/up row pairs and output rows
};

// Rows per chunk: bounded by the slot size, by the partial-sum buffer and (for
// gate/up) by one reduction warp per row pair.
__host__ __device__ inline void chunk_rows(int H, int I, int G, int& ch1, int& ch2) {
  const int b1 = 2 * (H / 2 + H / G);
  ch1 = (kSlotBytes - 64) / b1;
  ch1 = ch1 < kCWarps ? ch1 : kCWarps;
  const int u1 = 2 * (H / 32);
  ch1 = ch1 < kMaxChunkUnits / u1 ? ch1 : kMaxChunkUnits / u1;
  ch1 = ch1 < 1 ? 1 : ch1;
  ch2 = (kSlotBytes - 32) / (I / 2 + I / G);
  ch2 = ch2 < 64 ? ch2 : 64;
  ch2 = ch2 < kMaxChunkUnits / (I / 32) ? ch2 : kMaxChunkUnits / (I / 32);
  ch2 = ch2 < 1 ? 1 : ch2;
}

__device__ __forceinline__ Geo geometry(const Args& a, int fmt) {
  Geo g;
  g.P = a.T * a.k;
  g.upr = a.H >> 5;
  g.updr = a.I >> 5;
  chunk_rows(a.H, a.I, fmt == MOE_FMT_NVFP4 ? 16 : 32, g.ch1, g.ch2);
  const long long R1 = (long long)g.P * a.I, R2 = (long long)a.T * a.H;
  g.r0 = (long long)blockIdx.x * R1 / gridDim.x;
  g.r1 = (long long)(blockIdx.x + 1) * R1 / gridDim.x;
  g.q0 = (long long)blockIdx.x * R2 / gridDim.x;
  g.q1 = (long long)(blockIdx.x + 1) * R2 / gridDim.x;
  return g;
}

struct Win {  // 16-byte aligned window [lo, lo + bytes) around a byte range
  size_t lo;
  uint32_t bytes, delta;
};
__device__ __forceinline__ Win window(size_t start, size_t len) {
  Win w;
  w.lo = start & ~(size_t)15;
  const size_t hi = (start + len + 15) & ~(size_t)15;
  w.bytes = (uint32_t)(hi - w.lo);
  w.delta = (uint32_t)(start - w.lo);
  return w;
}

// One 16-byte unit of codes (32 elements) against activations held as float4
// quads: quad qq (elements 4qq..4qq+3 of the unit) at act[qq * stride].  Four
// independent accumulators (one per code word) keep the FMA chains short.
template <int FMT, int STRIDE>
__device__ __forceinline__ float unit_dot_q(uint4 q, uint32_t sbits, const float4* act, int stride_rt) {
  const int stride = STRIDE > 0 ? STRIDE : stride_rt;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float2 acc[4];
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    acc[wi] = make_float2(0.f, 0.f);
    const float4 x0 = act[(2 * wi) * stride];
    const float4 x1 = act[(2 * wi + 1) * stride];
    const float2 xp[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                          make_float2(x1.z, x1.w)};
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const uint32_t h2 = moe::e2m1x2_to_f16x2((w[wi] >> (8 * bi)) & 0xFFu);
      const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      acc[wi] = moe::ffma2(wf, xp[bi], acc[wi]);
    }
  }
  const float a = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
  const float b = (acc[2].x + acc[2].y) + (acc[3].x + acc[3].y);
  if (FMT == MOE_FMT_NVFP4) {
    const float2 s = moe::e4m3x2_to_f32x2(sbits);
    return a * s.x + b * s.y;
  } else {
    return (a + b) * moe::ue8m0_to_f32(sbits);
  }
}

// float element e of a unit-quad layout: quad (e%32)/4 at [quad][unit]
__device__ __forceinline__ int quad_index(int e, int stride) {
  return (((e & 31) >> 2) * stride + (e >> 5)) * 4 + (e & 3);
}

template <int FMT, int UPR, int UPDR>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(Args a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;                                          // kSlots x kSlotBytes
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSlots * kSlotBytes);
  uint64_t* empty = full + kSlots;
  const uint8_t** recs = reinterpret_cast<const uint8_t**>(empty + kSlots);  // [64]
  float* wts = reinterpret_cast<float*>(recs + 64);                          // [64]
  int* flags = reinterpret_cast<int*>(wts + 64);                             // [0] abort, [1] barrier ok
  float* part = reinterpret_cast<float*>(flags + 4);                         // [2][kMaxChunkUnits]
  float* yacc = part + 2 * kMaxChunkUnits;                                   // [rows/CTA + 1]
  moe::pdl_launch_dependents();

  const Geo g = geometry(a, FMT);
  const int upr = UPR > 0 ? UPR : g.upr;
  const int updr = UPDR > 0 ? UPDR : g.updr;
  const int rows_cta = (int)(g.q1 - g.q0);
  int* ybad = reinterpret_cast<int*>(yacc + rows_cta + 1);
  float4* act = reinterpret_cast<float4*>(
      (reinterpret_cast<uintptr_t>(ybad + rows_cta + 1) + 15) & ~(uintptr_t)15);
  const moe::RecordOffsets o = moe::record_offsets(a.H, a.I, FMT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      moe::tc::mbar_init(&full[s], 1);
      moe::tc::mbar_init(&empty[s], 1);
    }
    flags[0] = 0;
    moe::tc::mbar_fence_init();
  }
  for (int r = threadIdx.x; r <= rows_cta; r += kThreads) {
    yacc[r] = 0.f;
    ybad[r] = 0;
  }
  moe::pdl_wait();
  if (threadIdx.x < g.P) {
    recs[threadIdx.x] = checked_record(a.idx[threadIdx.x], a.E, a.ptrs,
                                       blockIdx.x == 0 ? a.status : nullptr);
    wts[threadIdx.x] = a.w[threadIdx.x];
  }
  // x of every token as float quads [t][8][H/32]
  for (int h0 = threadIdx.x * 4; h0 < a.T * a.H; h0 += kThreads * 4) {
    const int t = h0 / a.H, hh = h0 - t * a.H;
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.x + h0));
    act[(size_t)t * 8 * upr + ((hh & 31) >> 2) * upr + (hh >> 5)] =
        make_float4(moe::bf16_bits_to_f32(v.x & 0xFFFFu), moe::bf16_bits_to_f32(v.x >> 16),
                    moe::bf16_bits_to_f32(v.y & 0xFFFFu), moe::bf16_bits_to_f32(v.y >> 16));
  }
  __syncthreads();

  volatile int* abort_flag = flags;
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = 32 / G;

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int c = 0;
      bool ok = true;
      auto next_slot = [&](int& slot) -> bool {
        slot = c % kSlots;
        if (*abort_flag ||
            !moe::tc::mbar_wait(&empty[slot], ((c / kSlots) & 1) ^ 1,
                                moe::tc::globaltimer() + kWaitNs)) {
          *abort_flag = 1;
          moe::status_or(a.status, MOE_DEV_TIMEOUT);
          return false;
        }
        return true;
      };
      for (long long r = g.r0; r < g.r1 && ok;) {
        const int p = (int)(r / a.I), i0 = (int)(r - (long long)p * a.I);
        const int n = (int)min((long long)g.ch1, min(g.r1 - r, (long long)(a.I - i0)));
        int slot;
        if (!(ok = next_slot(slot))) break;
        const uint8_t* rec = recs[p];
        const uint32_t base = moe::tc::smem_u32(ring + slot * kSlotBytes);
        const uint32_t cb = (uint32_t)n * (a.H / 2);
        const Win gw = window(o.gate_s + (size_t)i0 * (a.H / G), (size_t)n * (a.H / G));
        const Win uw = window(o.up_s + (size_t)i0 * (a.H / G), (size_t)n * (a.H / G));
        moe::tc::mbar_arrive_expect_tx(&full[slot], rec ? 2 * cb + gw.bytes + uw.bytes : 0);
        if (rec) {
          moe::tc::bulk_g2s(base, rec + o.gate + (size_t)i0 * (a.H / 2), cb, &full[slot]);
          moe::tc::bulk_g2s(base + cb, rec + o.up + (size_t)i0 * (a.H / 2), cb, &full[slot]);
          moe::tc::bulk_g2s(base + 2 * cb, rec + gw.lo, gw.bytes, &full[slot]);
          moe::tc::bulk_g2s(base + 2 * cb + gw.bytes, rec + uw.lo, uw.bytes, &full[slot]);
        }
        ++c;
        r += n;
      }
      for (long long q = g.q0; q < g.q1 && ok;) {
        const int t = (int)(q / a.H), n0 = (int)(q - (long long)t * a.H);
        const int nr = (int)min((long long)g.ch2, min(g.q1 - q, (long long)(a.H - n0)));
        for (int j = 0; j < a.k && ok; ++j) {
          int slot;
          if (!(ok = next_slot(slot))) break;
          const uint8_t* rec = recs[t * a.k + j];
          const uint32_t base = moe::tc::smem_u32(ring + slot * kSlotBytes);
          const uint32_t cb = (uint32_t)nr * (a.I / 2);
          const Win dw = window(o.down_s + (size_t)n0 * (a.I / G), (size_t)nr * (a.I / G));
          moe::tc::mbar_arrive_expect_tx(&full[slot], rec ? cb + dw.bytes : 0);
          if (rec) {
            moe::tc::bulk_g2s(base, rec + o.down + (size_t)n0 * (a.I / 2), cb, &full[slot]);
            moe::tc::bulk_g2s(base + cb, rec + dw.lo, dw.bytes, &full[slot]);
          }
          ++c;
        }
        q += nr;
      }
      // every issued copy must land before this CTA may exit
      for (int cc = max(0, c - kSlots); cc < c; ++cc)
        moe::tc::mbar_wait(&full[cc % kSlots], (cc / kSlots) & 1, moe::tc::globaltimer() + kWaitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Control flow is the same for every consumer thread (fixed trip counts),
    // so the named barriers always match; after a timeout the work is skipped.
    const int ct = threadIdx.x;  // 0..479
    int c = 0;
    auto take = [&](int slot) -> bool {
      if (*abort_flag) return false;
      if (!moe::tc::mbar_wait(&full[slot], (c / kSlots) & 1, moe::tc::globaltimer() + kWaitNs)) {
        *abort_flag = 1;
        moe::status_or(a.status, MOE_DEV_TIMEOUT);
        return false;
      }
      return true;
    };
    // gate/up + SwiGLU: every consumer thread takes units of the chunk; one
    // warp per row pair then adds the partial sums in a fixed order.
    for (long long r = g.r0; r < g.r1;) {
      const int p = (int)(r / a.I), i0 = (int)(r - (long long)p * a.I);
      const int n = (int)min((long long)g.ch1, min(g.r1 - r, (long long)(a.I - i0)));
      const int slot = c % kSlots;
      float* pbuf = part + (c & 1) * kMaxChunkUnits;
      const bool live = take(slot);
      const uint8_t* base = ring + slot * kSlotBytes;
      const uint8_t* rec = recs[p];
      const uint32_t cb = (uint32_t)n * (a.H / 2);
      const Win gw = window(o.gate_s + (size_t)i0 * (a.H / G), (size_t)n * (a.H / G));
      const Win uw = window(o.up_s + (size_t)i0 * (a.H / G), (size_t)n * (a.H / G));
      const float4* xt = act + (size_t)(p / a.k) * 8 * upr;
      const int nunits = n * 2 * upr;
      if (live && rec) {
        for (int qf = ct; qf < nunits; qf += kCThreads) {
          const int rr = qf / (2 * upr), rem = qf - rr * 2 * upr;
          const bool is_up = rem >= upr;
          const int cix = is_up ? rem - upr : rem;
          const uint4 q = *reinterpret_cast<const uint4*>(base + (is_up ? cb : 0) + (size_t)rr * (a.H / 2) + 16 * cix);
          const uint8_t* sp = base + 2 * cb + (is_up ? gw.bytes + uw.delta : gw.delta) + (size_t)rr * (a.H / G) + sstep * cix;
          const uint32_t sb = FMT == MOE_FMT_NVFP4 ? (uint32_t)sp[0] | ((uint32_t)sp[1] << 8) : (uint32_t)sp[0];
          pbuf[qf] = unit_dot_q<FMT, UPR>(q, sb, xt + cix, upr);
        }
      }
      moe::tc::named_sync(1, kCThreads);
      if (ct == 0) moe::tc::mbar_arrive(&empty[slot]);
      if (warp < n) {
        float hv = __uint_as_float(0x7FC00000u);
        if (live && rec) {
          const float* pr = pbuf + warp * 2 * upr;
          float gs = 0.f, us = 0.f;
          for (int u = lane; u < upr; u += 32) {
            gs += pr[u];
            us += pr[upr + u];
          }
          gs = moe::warp_sum(gs);
          us = moe::warp_sum(us);
          hv = gs / (1.0f + expf(-gs)) * us;
        }
        if (lane == 0) a.hws[(size_t)p * a.I + i0 + warp] = hv;
      }
      ++c;
      r += n;
    }
    // grid barrier among the consumer threads of every CTA
    moe::tc::named_sync(1, kCThreads);
    if (ct == 0) {
      int good = !*abort_flag;
      if (good) {
        const unsigned e0 = moe::ld_acquire_gpu(a.bar + 1);
        __threadfence();
        const unsigned old = atomicAdd(a.bar, 1u);
        if (old == gridDim.x - 1) {
          atomicExch(a.bar, 0u);
          __threadfence();
          atomicAdd(a.bar + 1, 1u);
        } else {
          const uint64_t dl = moe::global_ns() + kWaitNs;
          while (moe::ld_acquire_gpu(a.bar + 1) == e0) {
            if (moe::global_ns() > dl) {
              good = 0;
              break;
            }
          }
        }
        __threadfence();
      }
      if (!good) {
        *abort_flag = 1;
        moe::status_or(a.status, MOE_DEV_TIMEOUT);
      }
      flags[1] = good;
    }
    moe::tc::named_sync(1, kCThreads);
    if (rows_cta > 0) {
      // stage h of the tokens this CTA's output rows belong to, float quads
      // [pair][8][I/32]
      const int t_lo = (int)(g.q0 / a.H), t_hi = (int)((g.q1 - 1) / a.H);
      const int n_q = (t_hi - t_lo + 1) * a.k * a.I / 4;
      const float4* src = reinterpret_cast<const float4*>(a.hws + (size_t)t_lo * a.k * a.I);
      if (flags[1]) {
        for (int e4 = ct; e4 < n_q; e4 += kCThreads) {
          const int e = 4 * e4;
          const int pj = e / a.I, i = e - pj * a.I;
          act[(size_t)pj * 8 * updr + ((i & 31) >> 2) * updr + (i >> 5)] = __ldcg(src + e4);
        }
      }
      moe::tc::named_sync(1, kCThreads);
      // down + weighted combine: units over all consumer threads, then one
      // thread per output row adds its partials in a fixed order
      for (long long q = g.q0; q < g.q1;) {
        const int t = (int)(q / a.H), n0 = (int)(q - (long long)t * a.H);
        const int nr = (int)min((long long)g.ch2, min(g.q1 - q, (long long)(a.H - n0)));
        for (int j = 0; j < a.k; ++j) {
          const int slot = c % kSlots;
          float* pbuf = part + (c & 1) * kMaxChunkUnits;
          const bool live = take(slot);
          const uint8_t* base = ring + slot * kSlotBytes;
          const int pj = t * a.k + j;
          const uint8_t* rec = recs[pj];
          const uint32_t cb = (uint32_t)nr * (a.I / 2);
          const Win dw = window(o.down_s + (size_t)n0 * (a.I / G), (size_t)nr * (a.I / G));
          const float4* hcol = act + (size_t)(pj - t_lo * a.k) * 8 * updr;
          const int nunits = nr * updr;
          if (live && rec) {
            for (int qf = ct; qf < nunits; qf += kCThreads) {
              const int rr = qf / updr, u = qf - rr * updr;
              const uint4 qv = *reinterpret_cast<const uint4*>(base + (size_t)rr * (a.I / 2) + 16 * u);
              const uint8_t* sp = base + cb + dw.delta + (size_t)rr * (a.I / G) + sstep * u;
              const uint32_t sb = FMT == MOE_FMT_NVFP4 ? (uint32_t)sp[0] | ((uint32_t)sp[1] << 8) : (uint32_t)sp[0];
              pbuf[qf] = unit_dot_q<FMT, UPDR>(qv, sb, hcol + u, updr);
            }
          }
          moe::tc::named_sync(1, kCThreads);
          if (ct == 0) moe::tc::mbar_arrive(&empty[slot]);
          if (ct < nr) {
            const int yi = (int)(q - g.q0) + ct;
            if (live && rec) {
              const float* pr = pbuf + ct * updr;
              float s = 0.f;
              for (int u = 0; u < updr; ++u) s += pr[u];
              yacc[yi] += wts[pj] * s;
            } else {
              ybad[yi] = 1;
            }
          }
          ++c;
        }
        q += nr;
      }
      moe::tc::named_sync(1, kCThreads);
      for (int r = ct; r < rows_cta; r += kCThreads)
        a.y[g.q0 + r] = (ybad[r] || *abort_flag) ? __uint_as_float(0x7FC00000u) : yacc[r];
    }
  }
  __syncthreads();
}

size_t smem_bytes(int T, int k, int H, int I, int sms) {
  const long long R2 = (long long)T * H;
  const long long rows = (R2 + sms - 1) / sms + 1;
  const long long ntok = std::min<long long>(T, rows / H + 2);
  const size_t act = std::max<size_t>((size_t)T * H * 4, (size_t)ntok * k * I * 4);
  return (size_t)kSlots * kSlotBytes + 2 * kSlots * 8 + 64 * 8 + 64 * 4 + 16 +
         2 * kMaxChunkUnits * 4 + (size_t)(rows + 1) * 8 + 16 + act;
}

}  // namespace st

template <typename K>
bool ensure_smem(K kernel, size_t bytes, size_t* granted) {
  if (bytes <= 48 * 1024 || bytes <= *granted) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  *granted = bytes;
  return true;
}

template <int FMT>
int launch_decode(const uint16_t* x, const int32_t* idx, const float* w, int T, int k,
                  const void* const* ptrs, int E, int H, int I, float* y, float* hws,
                  int32_t* st, cudaStream_t stream) {
  const size_t smem1 = (size_t)H * sizeof(float);
  const size_t smem2 = (size_t)k * I * sizeof(float);
  static size_t granted1 = 0, granted2 = 0;
  if (!ensure_smem(decode_gateup_kernel<FMT>, smem1, &granted1) ||
      !ensure_smem(decode_down_kernel<FMT>, smem2, &granted2))
    return MOE_ERR_CUDA;
  dim3 g1((I + 7) / 8, T * k);
  decode_gateup_kernel<FMT><<<g1, kThreads, smem1, stream>>>(x, idx, k, ptrs, E, H, I, hws, st);
  dim3 g2((H + 8 * kDownRowsPerWarp - 1) / (8 * kDownRowsPerWarp), T);
  decode_down_kernel<FMT><<<g2, kThreads, smem2, stream>>>(idx, w, k, ptrs, E, H, I, hws, y, st);
  return moe::launch_status();
}

int stream_smem_limit() {
  static int limit = 0;
  if (limit == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      limit = 0;
  }
  return limit;
}

int sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 0;
  }
  return sms;
}

// The streaming kernel takes T*k <= 64 pairs whose shared-memory plan fits.
bool stream_fits(int T, int k, int H, int I) {
  const int sms = sm_count();
  if (sms <= 0 || (long long)T * k > 64) return false;
  return st::smem_bytes(T, k, H, I, sms) + 1024 <= (size_t)stream_smem_limit();
}

template <int FMT, int UPR, int UPDR>
int launch_stream_shape(const st::Args& sa, size_t smem, int sms, cudaStream_t stream) {
  static size_t granted = 0;
  if (!ensure_smem(st::stream_kernel<FMT, UPR, UPDR>, smem, &granted)) return MOE_ERR_CUDA;
  return moe::launch_pdl(st::stream_kernel<FMT, UPR, UPDR>, dim3(sms), dim3(st::kThreads), smem,
                         stream, sa);
}

template <int FMT>
int launch_stream(const st::Args& sa, cudaStream_t stream) {
  const int sms = sm_count();
  const size_t smem = st::smem_bytes(sa.T, sa.k, sa.H, sa.I, sms);
  // one CTA per SM: all CTAs are resident together, as the grid barrier needs.
  // The row strides are compile-time constants for the two model shapes.
  const int upr = sa.H / 32, updr = sa.I / 32;
  if (upr == 80 && updr == 20) return launch_stream_shape<FMT, 80, 20>(sa, smem, sms, stream);
  if (upr == 128 && updr == 90) return launch_stream_shape<FMT, 128, 90>(sa, smem, sms, stream);
  return launch_stream_shape<FMT, 0, 0>(sa, smem, sms, stream);
}

}  // namespace

// h [T*k][I] FP32, then two barrier words (rounded up to 256 bytes).
extern "C" size_t moe_experts_decode_workspace(int T, int k, moe_expert_shape s) {
  if (T <= 0 || k <= 0 || !moe::shape_ok(s)) return 0;
  return (size_t)T * k * s.inter * sizeof(float) + 256;
}

extern "C" int moe_experts_decode(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                                  int T, int k, const void* const* expert_ptrs, int E,
                                  moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, void* stream) {
  if (!x_bf16 || !idx || !weights || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || k <= 0 || k > 32 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > 4096 || (long long)k * s.inter > 49152) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_experts_decode_workspace(T, k, s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(x_bf16) || !moe::aligned16(workspace)) return MOE_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  float* hws = reinterpret_cast<float*>(workspace);
  if (stream_fits(T, k, s.hidden, s.inter)) {
    st::Args sa;
    sa.x = x_bf16;
    sa.idx = idx;
    sa.w = weights;
    sa.T = T;
    sa.k = k;
    sa.ptrs = expert_ptrs;
    sa.E = E;
    sa.H = s.hidden;
    sa.I = s.inter;
    sa.hws = hws;
    sa.bar = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(workspace) +
                                         (size_t)T * k * s.inter * sizeof(float));
    sa.y = y;
    sa.status = dev_status;
    return s.format == MOE_FMT_NVFP4 ? launch_stream<MOE_FMT_NVFP4>(sa, st)
                                     : launch_stream<MOE_FMT_MXFP4>(sa, st);
  }
  if (s.format == MOE_FMT_NVFP4)
    return launch_decode<MOE_FMT_NVFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden,
                                        s.inter, y, hws, dev_status, st);
  return launch_decode<MOE_FMT_MXFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden,
                                      s.inter, y, hws, dev_status, st);
}

// ---------------------------------------------------------------------------
// Decode without any caller-side or library-side allocation.
//
// Some callers of this library cannot allocate device memory on the decode
// path: a plugin inside a host framework that is handed only its input and
// output buffers, or a latency-critical serving loop that must never enter an
// allocator.  For them the scratch of moe_experts_decode (the SwiGLU
// intermediate and the grid-barrier words) lives in the file-scope array
// below, which every GPU that loads this library holds until the process
// exits.  Host code must not use the array's name as a device address: the
// address is fetched once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The device address of g_decode_scratch on the current device (set up on
// the first call for that device).
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" size_t moe_experts_decode_noalloc_limit(void) { return kStaticScratchBytes; }

extern "C" int moe_experts_decode_noalloc(const uint16_t* x_bf16, const int32_t* idx,
                                          const float* weights, int T, int k,
                                          const void* const* expert_ptrs, int E,
                                          moe_expert_shape s, float* y, int32_t* dev_status,
                                          void* stream) {
  if (!x_bf16 || !idx || !weights || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || k <= 0 || k > 32 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  const size_t need = moe_experts_decode_workspace(T, k, s);
  if (need == 0 || need > kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = static_scratch(&scratch);
  if (rc != MOE_OK) return rc;
  // The array keeps whatever the previous call left; the barrier words sit
  // right after this call's h and must start at zero.
  const size_t bar_off = (size_t)T * k * s.inter * sizeof(float);
  if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + bar_off, 0, need - bar_off,
                      (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_experts_decode(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y, scratch,
                            kStaticScratchBytes, dev_status, stream);
}
