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
#include "decode_oneshot.h"
#include "decode_ring_plan.h"
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
// Streaming expert pass (T*k <= 512): one CTA per SM.  Producer lanes walk
// this CTA's share of the selected records -- first the gate/up rows, then
// the down rows -- and move it with 1-D TMA bulk copies of several rows each
// into a ring of shared-memory slots, refilled as soon as a slot's rows are
// done, so the HBM pipe stays full.  Fifteen consumer warps compute from
// shared memory: gate/up + SwiGLU rows -> h (global scratch), one grid
// barrier, then down rows against h and the weighted combine, accumulated per
// output row in a fixed order (bit-reproducible).  Slots that hold down rows
// are filled while the consumers still work on gate/up.
// ---------------------------------------------------------------------------
namespace st {

using namespace moe::ring;

constexpr int kThreads = 512;      // warps 0-14 consume, warp 15 lanes 0-15 produce
constexpr int kCWarps = 15;
constexpr int kCThreads = kCWarps * 32;
constexpr int kProdLanes = 16;  // copies issued by 16 lanes: measured faster than 4
constexpr int kMaxSlots = 64;
constexpr int kMaxPairs = 512;  // routed pairs (T*k) of one launch
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
  int slots;       // ring slots (<= kMaxSlots)
  int slot_bytes;  // bytes per slot (multiple of 128)
  int jn;          // experts per down-projection chunk
};

// FP16 x FP16 -> FP32 fused multiply-add (the product is exact in FP32).
__device__ __forceinline__ float fma_h(uint32_t a_lo16, uint32_t b_lo16, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;"
      : "=f"(d)
      : "h"((uint16_t)(a_lo16 & 0xFFFFu)), "h"((uint16_t)(b_lo16 & 0xFFFFu)), "f"(c));
  return d;
}

// 8 e2m1 codes (one word) -> 4 f16x2, element 2i in the low half of out[i].
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

template <int FMT>
__device__ __forceinline__ float apply_scale(float a, float b, uint32_t sbits) {
  if (FMT == MOE_FMT_NVFP4) {
    const float2 s = moe::e4m3x2_to_f32x2(sbits);
    return a * s.x + b * s.y;
  } else {
    return (a + b) * moe::ue8m0_to_f32(sbits);
  }
}

// One unit (16 bytes = 32 codes) against FP16 activations: quad qq of the
// unit (elements 8qq..8qq+7 as 4 f16x2) at xq[qq * stride].
template <int FMT, int STRIDE>
__device__ __forceinline__ float unit_dot_h(uint4 q, uint32_t sbits, const uint4* xq, int stride_rt) {
  const int stride = STRIDE > 0 ? STRIDE : stride_rt;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // two per scale block
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const uint4 xv4 = xq[wi * stride];
    const uint32_t xv[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
    uint32_t h[4];
    cvt_e2m1x8(w[wi], h);
    const int a0 = (wi >> 1) * 2;
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      acc[a0] = fma_h(h[bi], xv[bi], acc[a0]);
      acc[a0 + 1] = fma_h(h[bi] >> 16, xv[bi] >> 16, acc[a0 + 1]);
    }
  }
  return apply_scale<FMT>(acc[0] + acc[1], acc[2] + acc[3], sbits);
}

// The same against an FP32 operand carried as FP16 hi + lo parts.
template <int FMT, int STRIDE>
__device__ __forceinline__ float unit_dot_h2(uint4 q, uint32_t sbits, const uint4* hi, const uint4* lo,
                                             int stride_rt) {
  const int stride = STRIDE > 0 ? STRIDE : stride_rt;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const uint4 h4 = hi[wi * stride], l4 = lo[wi * stride];
    const uint32_t hv[4] = {h4.x, h4.y, h4.z, h4.w}, lv[4] = {l4.x, l4.y, l4.z, l4.w};
    uint32_t c[4];
    cvt_e2m1x8(w[wi], c);
    const int a0 = (wi >> 1) * 2;
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      acc[a0] = fma_h(c[bi], hv[bi], acc[a0]);
      acc[a0 + 1] = fma_h(c[bi] >> 16, hv[bi] >> 16, acc[a0 + 1]);
      acc[a0] = fma_h(c[bi], lv[bi], acc[a0]);
      acc[a0 + 1] = fma_h(c[bi] >> 16, lv[bi] >> 16, acc[a0 + 1]);
    }
  }
  return apply_scale<FMT>(acc[0] + acc[1], acc[2] + acc[3], sbits);
}

template <int FMT>
__device__ __forceinline__ uint32_t scale_bits(const uint8_t* sp) {
  return FMT == MOE_FMT_NVFP4 ? (uint32_t)sp[0] | ((uint32_t)sp[1] << 8) : (uint32_t)sp[0];
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int FMT, int UPR, int UPDR>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(Args a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = a.slots, SB = a.slot_bytes;
  uint8_t* ring = smem;                                                   // S x SB
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * SB);
  uint64_t* empty = full + kMaxSlots;
  const int P = a.T * a.k, Pr = (P + 15) & ~15;
  const uint8_t** recs = reinterpret_cast<const uint8_t**>(empty + kMaxSlots);  // [Pr]
  float* wts = reinterpret_cast<float*>(recs + Pr);                              // [Pr]
  int* flags = reinterpret_cast<int*>(wts + Pr);  // [0] abort, [1] barrier ok
  // slot_fill[s]: the last chunk a producer started in slot s.  A barrier's
  // parity is only meaningful once the slot is on the right fill: consumers
  // first wait for slot_fill == chunk, producers for slot_fill == chunk - S.
  volatile int* slot_fill = flags + 4;                                   // [kMaxSlots]
  uint4* act = reinterpret_cast<uint4*>(flags + 4 + kMaxSlots);
  moe::pdl_launch_dependents();

  const int upr = UPR > 0 ? UPR : a.H >> 5;
  const int updr = UPDR > 0 ? UPDR : a.I >> 5;
  const moe::RecordOffsets o = moe::record_offsets(a.H, a.I, FMT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = FMT == MOE_FMT_NVFP4 ? 2 : 1;
  const long long R1 = (long long)P * a.I, R2 = (long long)a.T * a.H;
  // row ranges of this CTA (32-bit: T*k*I and T*H stay below 2^23 here)
  const int r0 = share_at(blockIdx.x, gridDim.x, R1), r1 = share_at(blockIdx.x + 1, gridDim.x, R1);
  const int q0 = share_at(blockIdx.x, gridDim.x, R2), q1 = share_at(blockIdx.x + 1, gridDim.x, R2);
  const int jn = a.jn;
  const int cpr = (a.k + jn - 1) / jn;  // down chunks per output row
  const int n1 = gu_chunks(r0, r1);        // gate/up chunks of this CTA
  const int nb2 = dn_blocks(q0, q1, a.H);  // blocks of output rows
  const int n2 = nb2 * cpr;                // down chunks of this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxSlots; ++s) {
      moe::tc::mbar_init(&full[s], 1);
      moe::tc::mbar_init(&empty[s], kRG);  // one arrival per row of the chunk
      slot_fill[s] = -1;
    }
    flags[0] = 0;
    flags[1] = 0;
    moe::tc::mbar_fence_init();
  }
  moe::pdl_wait();
  for (int p = threadIdx.x; p < P; p += kThreads) {
    recs[p] = checked_record(a.idx[p], a.E, a.ptrs, blockIdx.x == 0 ? a.status : nullptr);
    wts[p] = a.w[p];
  }
  // x of the tokens of this CTA's gate/up rows, [xt0, xt1], as FP16 quads
  // [t - xt0][4][H/32] (8 values per uint4)
  const int xt0 = r1 > r0 ? (r0 / a.I) / a.k : 0;
  const int xt1 = r1 > r0 ? ((r1 - 1) / a.I) / a.k : -1;
  for (int h0 = threadIdx.x * 8; h0 < (xt1 - xt0 + 1) * a.H; h0 += kThreads * 8) {
    const int t = h0 / a.H, hh = h0 - t * a.H;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)xt0 * a.H + h0));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o4[i] = pack_h2(moe::bf16_bits_to_f32(wv[i] & 0xFFFFu), moe::bf16_bits_to_f32(wv[i] >> 16));
    act[(size_t)t * 4 * upr + ((hh & 31) >> 3) * upr + (hh >> 5)] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
  __syncthreads();
  volatile int* abort_flag = flags;

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producers
    if (lane < kProdLanes) {
      bool ok = true;
      auto claim = [&](int chunk) -> bool {
        const int slot = chunk % S;
        const uint64_t dl = moe::tc::globaltimer() + kWaitNs;
        bool good = !*abort_flag;
        if (good && chunk >= S) {
          while (slot_fill[slot] != chunk - S) {
            if (*abort_flag || moe::tc::globaltimer() > dl) {
              good = false;
              break;
            }
            __nanosleep(32);
          }
        }
        if (good) good = moe::tc::mbar_wait_backoff(&empty[slot], ((chunk / S) & 1) ^ 1, dl);
        if (!good) {
          *abort_flag = 1;
          moe::status_or(a.status, MOE_DEV_TIMEOUT);
          return false;
        }
        slot_fill[slot] = chunk;
        return true;
      };
      for (int c = lane; c < n1 + n2 && ok; c += kProdLanes) {
        if (!(ok = claim(c))) break;
        const int slot = c % S;
        const uint32_t base = moe::tc::smem_u32(ring + (size_t)slot * SB);
        if (c < n1) {  // gate/up: rows [rs, rs + nr), one or two pieces (one per pair)
          const GuChunk gc = gu_chunk(c, r0, r1, a.I);
          const uint32_t cb = (uint32_t)(a.H / 2), so = 2u * kRG * cb, room = (uint32_t)gu_scale_room(a.H, G);
          Win gw[2], uw[2];
          uint32_t total = 0;
#pragma unroll
          for (int pc = 0; pc < 2; ++pc) {
            const int n = pc == 0 ? gc.n0 : gc.nr - gc.n0, i = pc == 0 ? gc.i0 : 0;
            gw[pc] = window(o.gate_s + (size_t)i * (a.H / G), (size_t)n * (a.H / G));
            uw[pc] = window(o.up_s + (size_t)i * (a.H / G), (size_t)n * (a.H / G));
            if (n > 0 && recs[gc.p0 + pc]) total += 2u * n * cb + gw[pc].bytes + uw[pc].bytes;
          }
          moe::tc::mbar_arrive_expect_tx(&full[slot], total);
          uint32_t gso = 0, uso = 0;
#pragma unroll
          for (int pc = 0; pc < 2; ++pc) {
            const int n = pc == 0 ? gc.n0 : gc.nr - gc.n0, i = pc == 0 ? gc.i0 : 0, roff = pc == 0 ? 0 : gc.n0;
            const uint8_t* rec = n > 0 ? recs[gc.p0 + pc] : nullptr;
            if (rec) {
              const uint32_t gb = (uint32_t)n * cb;
              moe::tc::bulk_g2s(base + roff * cb, rec + o.gate + (size_t)i * cb, gb, &full[slot]);
              moe::tc::bulk_g2s(base + kRG * cb + roff * cb, rec + o.up + (size_t)i * cb, gb, &full[slot]);
              moe::tc::bulk_g2s(base + so + gso, rec + gw[pc].lo, gw[pc].bytes, &full[slot]);
              moe::tc::bulk_g2s(base + so + room + uso, rec + uw[pc].lo, uw[pc].bytes, &full[slot]);
            }
            gso += gw[pc].bytes;
            uso += uw[pc].bytes;
          }
        } else {  // down: output rows [n, n + nd) of token t, experts [j0, j1)
          const int c2 = c - n1;
          int qs = 0, nd = 0;
          dn_block(c2 / cpr, q0, q1, a.H, qs, nd);
          const int t = qs / a.H, n = qs - t * a.H;
          const int j0 = (c2 % cpr) * jn, j1 = min(a.k, j0 + jn);
          const uint32_t cb = (uint32_t)(a.I / 2), db = (uint32_t)nd * cb;
          const Win dw = window(o.down_s + (size_t)n * (a.I / G), (size_t)nd * (a.I / G));
          const uint32_t per = (uint32_t)dn_part_bytes(a.I, G);
          uint32_t total = 0;
          for (int j = j0; j < j1; ++j)
            if (recs[t * a.k + j]) total += db + dw.bytes;
          moe::tc::mbar_arrive_expect_tx(&full[slot], total);
          uint32_t off = 0;
          for (int j = j0; j < j1; ++j) {
            const uint8_t* rec = recs[t * a.k + j];
            if (rec) {
              moe::tc::bulk_g2s(base + off, rec + o.down + (size_t)n * cb, db, &full[slot]);
              moe::tc::bulk_g2s(base + off + kRD * cb, rec + dw.lo, dw.bytes, &full[slot]);
            }
            off += per;
          }
        }
      }
      // every copy this lane issued must land before the CTA may exit
      for (int c = lane; c < n1 + n2; c += kProdLanes)
        if (c >= n1 + n2 - S)
          moe::tc::mbar_wait_backoff(&full[c % S], (c / S) & 1, moe::tc::globaltimer() + kWaitNs);
    }
  } else {
    // ------------------------------------------------------------ consumers
    auto take = [&](int chunk) -> bool {
      if (*abort_flag) return false;
      const uint64_t dl = moe::tc::globaltimer() + kWaitNs;
      bool good = true;
      while (slot_fill[chunk % S] != chunk) {
        if (*abort_flag || moe::tc::globaltimer() > dl) {
          good = false;
          break;
        }
        __nanosleep(32);
      }
      if (good) good = moe::tc::mbar_wait_backoff(&full[chunk % S], (chunk / S) & 1, dl);
      if (!good) {
        *abort_flag = 1;
        moe::status_or(a.status, MOE_DEV_TIMEOUT);
        return false;
      }
      return true;
    };
    // a chunk's slot is free once every row of it is done: the warp of each
    // row arrives once, the warp of its last row also for the rows a ragged
    // chunk lacks
    auto release = [&](int chunk, int row, int rows) {
      __syncwarp();
      if (lane == 0) moe::tc::mbar_arrive_n(&empty[chunk % S], row == rows - 1 ? (uint32_t)(kRG - rows + 1) : 1u);
    };
    // gate/up + SwiGLU: task (chunk c, row ri) -> warp (c kRG + ri) % 15, so
    // the rows of one chunk (copied together) are computed by several warps
    // at once.  Lane l takes units l, l + 32, ... of the row, in that order.
    for (int task = warp; task < n1 * kRG; task += kCWarps) {
      const int c = task / kRG, ri = task - c * kRG;
      const GuChunk gc = gu_chunk(c, r0, r1, a.I);
      if (ri >= gc.nr) continue;
      const bool live = take(c);
      const int pc = ri < gc.n0 ? 0 : 1;
      const int p = gc.p0 + pc, i = pc == 0 ? gc.i0 + ri : ri - gc.n0;
      const uint8_t* rec = recs[p];
      const uint8_t* base = ring + (size_t)(c % S) * SB;
      const uint32_t cb = (uint32_t)(a.H / 2), so = 2u * kRG * cb, room = (uint32_t)gu_scale_room(a.H, G);
      // the row's scales: piece 0's windows first, then piece 1's
      const Win gw0 = window(o.gate_s + (size_t)gc.i0 * (a.H / G), (size_t)gc.n0 * (a.H / G));
      const Win uw0 = window(o.up_s + (size_t)gc.i0 * (a.H / G), (size_t)gc.n0 * (a.H / G));
      uint32_t gso = gw0.delta, uso = uw0.delta;
      if (pc == 1) {
        gso = gw0.bytes + window(o.gate_s, (size_t)(gc.nr - gc.n0) * (a.H / G)).delta;
        uso = uw0.bytes + window(o.up_s, (size_t)(gc.nr - gc.n0) * (a.H / G)).delta;
      }
      const int rr = pc == 0 ? ri : ri - gc.n0;  // row within its piece
      const uint8_t* crow = base + (size_t)ri * cb;
      const uint8_t* gsr = base + so + gso + (size_t)rr * (a.H / G);
      const uint8_t* usr = base + so + room + uso + (size_t)rr * (a.H / G);
      const uint4* xt = act + (size_t)(p / a.k - xt0) * 4 * upr;
      float gs = 0.f, us = 0.f;
      if (live && rec) {
        if constexpr (UPR > 0) {
#pragma unroll
          for (int m = 0; m < (2 * UPR + 31) / 32; ++m) {
            const int u = lane + 32 * m;
            if (u < 2 * UPR) {
              const bool is_up = u >= UPR;
              const int cix = is_up ? u - UPR : u;
              const uint4 q = *reinterpret_cast<const uint4*>(crow + (is_up ? kRG * cb : 0u) + 16 * cix);
              const float d = unit_dot_h<FMT, UPR>(q, scale_bits<FMT>((is_up ? usr : gsr) + sstep * cix), xt + cix, UPR);
              if (is_up) us += d;
              else gs += d;
            }
          }
        } else {
          for (int u = lane; u < 2 * upr; u += 32) {
            const bool is_up = u >= upr;
            const int cix = is_up ? u - upr : u;
            const uint4 q = *reinterpret_cast<const uint4*>(crow + (is_up ? kRG * cb : 0u) + 16 * cix);
            const float d = unit_dot_h<FMT, 0>(q, scale_bits<FMT>((is_up ? usr : gsr) + sstep * cix), xt + cix, upr);
            if (is_up) us += d;
            else gs += d;
          }
        }
      }
      release(c, ri, gc.nr);
      gs = moe::warp_sum(gs);
      us = moe::warp_sum(us);
      if (lane == 0)
        a.hws[(size_t)p * a.I + i] = (live && rec) ? gs / (1.0f + expf(-gs)) * us : __uint_as_float(0x7FC00000u);
    }
    // grid barrier among the consumer threads of every CTA
    moe::tc::named_sync(1, kCThreads);
    if (threadIdx.x == 0) {
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
            __nanosleep(32);
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
    if (q1 > q0) {
      // h of the tokens of this CTA's output rows as FP16 hi and lo quads:
      // hi [pair][4][I/32], then lo at +npairs*4*(I/32)
      const int t_lo = (int)(q0 / a.H), t_hi = (int)((q1 - 1) / a.H);
      const int npairs = (t_hi - t_lo + 1) * a.k;
      const int n8 = npairs * a.I / 8;
      uint4* hhi = act;
      uint4* hlo = act + (size_t)npairs * 4 * updr;
      const float4* src = reinterpret_cast<const float4*>(a.hws + (size_t)t_lo * a.k * a.I);
      if (flags[1]) {
        for (int e8 = threadIdx.x; e8 < n8; e8 += kCThreads) {
          const int e = 8 * e8;
          const int pj = e / a.I, i = e - pj * a.I;
          const float4 v0 = __ldcg(src + 2 * e8), v1 = __ldcg(src + 2 * e8 + 1);
          const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half h0 = __float2half_rn(v[2 * m]), h1 = __float2half_rn(v[2 * m + 1]);
            hv[m] = pack_h2(__half2float(h0), __half2float(h1));
            lv[m] = pack_h2(v[2 * m] - __half2float(h0), v[2 * m + 1] - __half2float(h1));
          }
          const size_t at = (size_t)pj * 4 * updr + ((i & 31) >> 3) * updr + (i >> 5);
          hhi[at] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          hlo[at] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
      }
      moe::tc::named_sync(1, kCThreads);
      // down + weighted combine: task (block bi of up to kRD output rows, kTR
      // of its rows from rb on) -> warp (task) % 15, which walks the block's
      // chunks (experts in ascending order).  Lane l takes the flattened
      // (expert, unit) items l, l + 32, ... of the task's rows, in that
      // order, each item's h loaded once for them.  One row per task: two
      // (h shared) measured slower, the fewer tasks leaving warps idle.
      constexpr int kTR = 1;  // rows per task
      static_assert(kRD % kTR == 0, "row tasks tile a block");
      for (int task = warp; task < nb2 * (kRD / kTR); task += kCWarps) {
        const int bi = task / (kRD / kTR), rb = (task - bi * (kRD / kTR)) * kTR;
        int qs = 0, nd = 0;
        dn_block(bi, q0, q1, a.H, qs, nd);
        if (rb >= nd) continue;
        const int nr = min(kTR, nd - rb);
        // this task's arrivals on each chunk: its rows, and, for the task of
        // the block's last row, the rows a ragged block lacks
        const uint32_t arrivals = rb + kTR >= nd ? (uint32_t)(kRD - rb) : (uint32_t)kTR;
        const int t = qs / a.H, n0 = qs - t * a.H;
        float acc[kTR];
#pragma unroll
        for (int r = 0; r < kTR; ++r) acc[r] = 0.f;
        bool bad = false;
        for (int cc = 0; cc < cpr; ++cc) {
          const int c = n1 + bi * cpr + cc;
          const bool live = take(c);
          const uint8_t* base = ring + (size_t)(c % S) * SB;
          const int j0 = cc * jn, j1 = min(a.k, j0 + jn);
          const uint32_t cb = (uint32_t)(a.I / 2);
          const Win dw = window(o.down_s + (size_t)n0 * (a.I / G), (size_t)nd * (a.I / G));
          const uint32_t per = (uint32_t)dn_part_bytes(a.I, G);
          for (int j = j0; j < j1; ++j)
            if (!(live && recs[t * a.k + j])) bad = true;
          if (!bad) {
            // units of experts j0..j1 flattened over the lanes
            const int nu = (j1 - j0) * updr;
            for (int f = lane; f < nu; f += 32) {
              const int jj = f / updr, u = f - jj * updr;
              const int pj = t * a.k + j0 + jj;
              const uint8_t* eb = base + (size_t)jj * per;
              const uint8_t* sp = eb + kRD * cb + dw.delta + (size_t)rb * (a.I / G) + sstep * u;
              const size_t col = (size_t)(pj - t_lo * a.k) * 4 * updr + u;
              uint4 hh[4], hl[4];
#pragma unroll
              for (int wi = 0; wi < 4; ++wi) {
                hh[wi] = hhi[col + (size_t)wi * updr];
                hl[wi] = hlo[col + (size_t)wi * updr];
              }
              const float wt = wts[pj];
#pragma unroll
              for (int r = 0; r < kTR; ++r) {
                if (r < nr)
                  acc[r] += wt * unit_dot_h2<FMT, 1>(
                                     *reinterpret_cast<const uint4*>(eb + (size_t)(rb + r) * cb + 16 * u),
                                     scale_bits<FMT>(sp + (size_t)r * (a.I / G)), hh, hl, 1);
              }
            }
          }
          __syncwarp();
          if (lane == 0) moe::tc::mbar_arrive_n(&empty[c % S], arrivals);
        }
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
          if (r < nr) {
            const float v = moe::warp_sum(acc[r]);
            if (lane == 0)
              a.y[(size_t)t * a.H + n0 + rb + r] = (bad || *abort_flag) ? __uint_as_float(0x7FC00000u) : v;
          }
        }
      }
    }
  }
  __syncthreads();
}

// Shared memory for `slots` ring slots plus the activation region: x as FP16
// quads (T*H halves) in phase 1, h as FP16 hi + lo quads in phase 2.
inline size_t smem_bytes(int T, int k, int H, int I, int sms, int slots, int slot_bytes) {
  // tokens of one CTA's gate/up rows (x) and of its output rows (h)
  const long long rows1 = (long long)T * k * I / sms + 1;
  const long long nx = std::min<long long>(T, (rows1 / I + 2) / k + 2);
  const long long rows2 = (long long)T * H / sms + 1;
  const long long ntok = std::min<long long>(T, rows2 / H + 2);
  const size_t act = std::max<size_t>((size_t)nx * H * 2, (size_t)ntok * k * I * 4);
  const size_t pr = ((size_t)T * k + 15) & ~(size_t)15;
  return (size_t)slots * slot_bytes + 2 * kMaxSlots * 8 + pr * 8 + pr * 4 + 16 + kMaxSlots * 4 + act;
}

}  // namespace st

template <int FMT>
int launch_decode(const uint16_t* x, const int32_t* idx, const float* w, int T, int k,
                  const void* const* ptrs, int E, int H, int I, float* y, float* hws,
                  int32_t* st, cudaStream_t stream) {
  const size_t smem1 = (size_t)H * sizeof(float);
  const size_t smem2 = (size_t)k * I * sizeof(float);
  static moe::SmemGrant granted1, granted2;
  if (!moe::grant_smem(decode_gateup_kernel<FMT>, smem1, granted1) ||
      !moe::grant_smem(decode_down_kernel<FMT>, smem2, granted2))
    return MOE_ERR_CUDA;
  dim3 g1((I + 7) / 8, T * k);
  decode_gateup_kernel<FMT><<<g1, kThreads, smem1, stream>>>(x, idx, k, ptrs, E, H, I, hws, st);
  dim3 g2((H + 8 * kDownRowsPerWarp - 1) / (8 * kDownRowsPerWarp), T);
  decode_down_kernel<FMT><<<g2, kThreads, smem2, stream>>>(idx, w, k, ptrs, E, H, I, hws, y, st);
  return moe::launch_status();
}

int stream_smem_limit() { return moe::device_info().smem_optin; }

int sm_count() { return moe::device_info().sms; }

// The streaming kernel takes T*k <= 512 pairs when at least 4 ring slots (of
// kRG row pairs each) fit next to the activations.
int stream_slots(int T, int k, int H, int I, int fmt, int* slot_bytes) {
  const int sms = sm_count();
  if (sms <= 0 || (long long)T * k > st::kMaxPairs) return 0;
  const int G = fmt == MOE_FMT_NVFP4 ? 16 : 32;
  *slot_bytes = st::plan_slot_bytes(H, I, G);
  const size_t limit = (size_t)stream_smem_limit();
  const size_t fixed = st::smem_bytes(T, k, H, I, sms, 0, *slot_bytes) + 1024;
  if (fixed >= limit) return 0;
  const int slots = (int)std::min<size_t>(st::kMaxSlots, (limit - fixed) / *slot_bytes);
  return slots >= 4 ? slots : 0;
}

template <int FMT, int UPR, int UPDR>
int launch_stream_shape(const st::Args& sa, size_t smem, int sms, cudaStream_t stream) {
  static moe::SmemGrant granted;
  if (!moe::grant_smem(st::stream_kernel<FMT, UPR, UPDR>, smem, granted, st::kThreads)) return MOE_ERR_CUDA;
  // the ring kernel's grid barrier needs every CTA resident: one CTA per SM,
  // checked by grant_smem above (see launch_shape of the one-shot kernel on
  // why the launch is not cooperative)
  return moe::launch_pdl(st::stream_kernel<FMT, UPR, UPDR>, dim3(sms), dim3(st::kThreads), smem, stream, sa);
}

template <int FMT>
int launch_stream(const st::Args& sa, cudaStream_t stream) {
  const int sms = sm_count();
  const size_t smem = st::smem_bytes(sa.T, sa.k, sa.H, sa.I, sms, sa.slots, sa.slot_bytes);
  // one CTA per SM: all CTAs are resident together, as the grid barrier needs.
  // The row strides are compile-time constants for the two model shapes.
  const int upr = sa.H / 32, updr = sa.I / 32;
  if (upr == 80 && updr == 20) return launch_stream_shape<FMT, 80, 20>(sa, smem, sms, stream);
  if (upr == 128 && updr == 90) return launch_stream_shape<FMT, 128, 90>(sa, smem, sms, stream);
  return launch_stream_shape<FMT, 0, 0>(sa, smem, sms, stream);
}

}  // namespace

// Workspace: a header (the one-shot kernel's 64-bit barrier counter at 0,
// the ring kernel's two barrier words at 128, the one-shot kernel's record
// of a wait that gave up at 192, the rest reserved), then the one-shot
// kernel's tagged logits and FP32 h (moe::os::oneshot_ws_bytes); the other
// paths keep their FP32 h [T*k][I] right after the header.  The header sits
// at a fixed place so that calls of any shape can share one workspace.
constexpr size_t kRingBarrierOffset = 128;
extern "C" size_t moe_experts_decode_workspace(int T, int k, moe_expert_shape s) {
  if (T <= 0 || k <= 0 || !moe::shape_ok(s)) return 0;
  const size_t fp32_h = moe::os::kHeaderBytes + (size_t)T * k * s.inter * sizeof(float);
  const size_t tagged = moe::os::oneshot_ws_bytes(T, k, s.inter);
  return tagged > fp32_h ? tagged : fp32_h;
}

// The argument checks of moe_experts_decode that do not involve the
// workspace (shared with the allocation-free entry point, which runs them
// before it touches its scratch).
static int decode_check_args(const uint16_t* x_bf16, const int32_t* idx, const float* weights, int T, int k,
                             const void* const* expert_ptrs, int E, const moe_expert_shape& s, const float* y) {
  if (!x_bf16 || !idx || !weights || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || k <= 0 || k > 32 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > 4096 || (long long)k * s.inter > 49152) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(x_bf16)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

static int decode_launch(const uint16_t* x_bf16, const int32_t* idx, const float* weights, int T, int k,
                         const void* const* expert_ptrs, int E, const moe_expert_shape& s, float* y,
                         void* workspace, int32_t* dev_status, void* stream);

extern "C" int moe_experts_decode(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                                  int T, int k, const void* const* expert_ptrs, int E,
                                  moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, void* stream) {
  const int rc = decode_check_args(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_experts_decode_workspace(T, k, s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(workspace)) return MOE_ERR_ALIGNMENT;
  return decode_launch(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y, workspace, dev_status, stream);
}

static int decode_launch(const uint16_t* x_bf16, const int32_t* idx, const float* weights, int T, int k,
                         const void* const* expert_ptrs, int E, const moe_expert_shape& s, float* y,
                         void* workspace, int32_t* dev_status, void* stream) {
  if (sm_count() <= 0) return MOE_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* hws = reinterpret_cast<float*>(ws + moe::os::kHeaderBytes);
  if (decode_oneshot_fits(T, k, s.hidden, s.inter, s.format, sm_count(), (size_t)stream_smem_limit())) {
    DecodeOneshotArgs oa = {};
    oa.x = x_bf16;
    oa.idx = idx;
    oa.w = weights;
    oa.T = T;
    oa.k = k;
    oa.ptrs = expert_ptrs;
    oa.E = E;
    oa.H = s.hidden;
    oa.I = s.inter;
    oneshot_set_workspace(oa, ws);
    oa.y = y;
    oa.status = dev_status;
    return launch_decode_oneshot(oa, s.format, sm_count(), stream);
  }
  int slot_bytes = 0;
  const int slots = stream_slots(T, k, s.hidden, s.inter, s.format, &slot_bytes);
  if (slots > 0) {
    st::Args sa;
    sa.slots = slots;
    sa.slot_bytes = slot_bytes;
    sa.jn = st::plan_jn(k, s.inter, s.format == MOE_FMT_NVFP4 ? 16 : 32, slot_bytes);
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
    sa.bar = reinterpret_cast<unsigned*>(ws + kRingBarrierOffset);
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

// Decode with records in host memory (the host tier): the same expert pass
// with plain 16-byte loads only, which read system memory through the
// device's address space (pinned host memory on a system with unified
// addressing, or any memory a Grace CPU and the GPU share over NVLink-C2C),
// so the records need not be in HBM.  The two-kernel path computes it.
extern "C" int moe_experts_decode_host(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                                       int T, int k, const void* const* expert_ptrs, int E,
                                       moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                                       int32_t* dev_status, void* stream) {
  const int rc = decode_check_args(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_experts_decode_workspace(T, k, s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(workspace)) return MOE_ERR_ALIGNMENT;
  if (sm_count() <= 0) return MOE_ERR_CUDA;
  float* hws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + moe::os::kHeaderBytes);
  cudaStream_t st = (cudaStream_t)stream;
  if (s.format == MOE_FMT_NVFP4)
    return launch_decode<MOE_FMT_NVFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden, s.inter, y, hws,
                                        dev_status, st);
  return launch_decode<MOE_FMT_MXFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden, s.inter, y, hws,
                                      dev_status, st);
}

// One decode layer in one launch: the router (RMS chaining of the previous
// layer's output or the given x, logits, top-k) and the expert pass of the
// one-shot kernel, with a grid barrier between them.
extern "C" int moe_decode_layer(const uint16_t* x_bf16, const float* y_prev, int T, double eps,
                                uint16_t* x_out, const uint16_t* wr_bf16, const float* bias, int E, int k,
                                int32_t* idx, float* weights, float* logits,
                                const void* const* expert_ptrs, moe_expert_shape s, float* y,
                                void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if ((x_bf16 == nullptr) == (y_prev == nullptr)) return MOE_ERR_INVALID_ARG;
  if (y_prev && !x_out) return MOE_ERR_INVALID_ARG;
  if (!wr_bf16 || !idx || !weights || !logits || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || E <= 0 || k <= 0 || k > E || k > 32 || !(eps >= 0.0)) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s) || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_experts_decode_workspace(T, k, s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((x_bf16 && !moe::aligned16(x_bf16)) || (x_out && !moe::aligned16(x_out)) || !moe::aligned16(wr_bf16) ||
      !moe::aligned16(workspace))
    return MOE_ERR_ALIGNMENT;
  if (!decode_oneshot_fits(T, k, s.hidden, s.inter, s.format, sm_count(), (size_t)stream_smem_limit(), true, E))
    return MOE_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeOneshotArgs oa = {};
  oa.x = x_bf16;
  oa.T = T;
  oa.k = k;
  oa.ptrs = expert_ptrs;
  oa.E = E;
  oa.H = s.hidden;
  oa.I = s.inter;
  oneshot_set_workspace(oa, ws);
  oa.y = y;
  oa.status = dev_status;
  oa.y_prev = y_prev;
  oa.eps = (float)eps;
  oa.x_out = x_out;
  oa.wr = wr_bf16;
  oa.bias = bias;
  oa.logits = logits;
  oa.idx_out = idx;
  oa.w_out = weights;
  return launch_decode_oneshot(oa, s.format, sm_count(), stream);
}

// A whole decode stack in one launch: layer 0 routes x0, every later layer
// RMS-chains the previous layer's y; the layers are separated by grid
// barriers inside one persistent kernel instead of launch boundaries.
extern "C" int moe_decode_stack(const uint16_t* x0, int T, double eps, int layers, const uint16_t* wr_bf16,
                                const float* bias, int E, int k, const void* const* expert_ptrs,
                                moe_expert_shape s, int32_t* idx, float* weights, float* logits, uint16_t* x_out,
                                float* y, void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!x0 || !wr_bf16 || !idx || !weights || !logits || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || layers <= 0 || layers > 4096 || E <= 0 || k <= 0 || k > E || k > 32 || !(eps >= 0.0))
    return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s) || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_experts_decode_workspace(T, k, s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(x0) || (x_out && !moe::aligned16(x_out)) || !moe::aligned16(wr_bf16) ||
      !moe::aligned16(workspace))
    return MOE_ERR_ALIGNMENT;
  if (sm_count() <= 0) return MOE_ERR_CUDA;
  if (!decode_oneshot_fits(T, k, s.hidden, s.inter, s.format, sm_count(), (size_t)stream_smem_limit(), true, E))
    return MOE_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeOneshotArgs oa = {};
  oa.x = x0;
  oa.T = T;
  oa.k = k;
  oa.ptrs = expert_ptrs;
  oa.E = E;
  oa.H = s.hidden;
  oa.I = s.inter;
  oneshot_set_workspace(oa, ws);
  oa.y = y;
  oa.status = dev_status;
  oa.y_prev = nullptr;
  oa.eps = (float)eps;
  oa.x_out = x_out;
  oa.wr = wr_bf16;
  oa.bias = bias;
  oa.logits = logits;
  oa.idx_out = idx;
  oa.w_out = weights;
  oa.layers = layers;
  return launch_decode_oneshot(oa, s.format, sm_count(), stream);
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

constexpr int kMaxDevices = moe::kMaxDevices;
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
  // every check that moe_experts_decode makes comes first, so a rejected
  // call leaves the shared array untouched and returns the same status
  int rc = decode_check_args(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  const size_t need = moe_experts_decode_workspace(T, k, s);
  if (need == 0 || need > kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  rc = static_scratch(&scratch);
  if (rc != MOE_OK) return rc;
  // The array keeps whatever the previous call left.  The part this call
  // uses starts at zero, as a fresh workspace would: the counters, and the
  // tagged exchange words, whose tags restart with the counter.
  if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  return decode_launch(x_bf16, idx, weights, T, k, expert_ptrs, E, s, y, scratch, dev_status, stream);
}
