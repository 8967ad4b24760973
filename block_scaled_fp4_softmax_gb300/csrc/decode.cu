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
#include "common.cuh"

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
// Fused expert pass for a handful of pairs (T*k <= 64): one persistent
// cooperative kernel runs gate/up + SwiGLU, a grid barrier, then down + the
// weighted combine.  Before waiting at the barrier every warp issues the loads
// of its first down row, so the down weights stream while the slowest gate/up
// rows finish.  Scratch: h [P][I] (transposed float2 layout per pair) and two
// barrier words.
// ---------------------------------------------------------------------------
struct FusedArgs {
  const uint16_t* x;
  const int32_t* idx;
  const float* w;
  int T, k;
  const void* const* ptrs;
  int E, H, I;
  float* hws;
  unsigned* bar;
  float* y;
  int32_t* st;
};

constexpr int kFusedMaxPairs = 64;

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) decode_fused_kernel(FusedArgs a) {
  extern __shared__ float2 act[];  // phase 1: x [T][16][H/32]; phase 2: h [P][16][I/32]
  __shared__ const uint8_t* recs[kFusedMaxPairs];
  __shared__ float wts[kFusedMaxPairs];
  __shared__ int bar_ok;
  moe::pdl_launch_dependents();
  moe::pdl_wait();

  const int P = a.T * a.k;
  const int H = a.H, I = a.I;
  const int upr = H >> 5, updr = I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kThreads / 32) + warp;
  const int NW = gridDim.x * (kThreads / 32);
  const moe::RecordOffsets o = moe::record_offsets(H, I, FMT);
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = 32 / G;

  // x of every token, transposed float2 layout per token
  for (int h0 = threadIdx.x * 8; h0 < a.T * H; h0 += kThreads * 8) {
    const int t = h0 / H, hh = h0 - t * H;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + h0));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    const int c = hh >> 5, pe0 = (hh & 31) >> 1;
    float2* xt = act + (size_t)t * 16 * upr;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xt[(pe0 + i) * upr + c] =
          make_float2(moe::bf16_bits_to_f32(wv[i] & 0xFFFFu), moe::bf16_bits_to_f32(wv[i] >> 16));
  }
  if (threadIdx.x < P) {
    recs[threadIdx.x] = checked_record(a.idx[threadIdx.x], a.E, a.ptrs,
                                       blockIdx.x == 0 ? a.st : nullptr);
    wts[threadIdx.x] = a.w[threadIdx.x];
  }
  __syncthreads();

  // ---- phase 1: one warp per (pair, intermediate row) ----
  const int tasks1 = P * I;
  for (int tau = gw; tau < tasks1; tau += NW) {
    const int p = tau / I, i = tau - p * I;
    const uint8_t* rec = recs[p];
    float* hp = a.hws + (size_t)p * I;
    const int hoff = 2 * (((i & 31) >> 1) * updr + (i >> 5)) + (i & 1);
    if (!rec) {
      if (lane == 0) hp[hoff] = __uint_as_float(0x7FC00000u);
      continue;
    }
    const float2* xt = act + (size_t)(p / a.k) * 16 * upr;
    const uint8_t* gcode = rec + o.gate + (size_t)i * (H / 2);
    const uint8_t* ucode = rec + o.up + (size_t)i * (H / 2);
    const uint8_t* gsc = rec + o.gate_s + (size_t)i * (H / G);
    const uint8_t* usc = rec + o.up_s + (size_t)i * (H / G);
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
          const float d = unit_dot_col<FMT>(q[m], sb[m], xt + c, upr);
          if (is_up) uacc += d;
          else gacc += d;
        }
      }
    }
    gacc = moe::warp_sum(gacc);
    uacc = moe::warp_sum(uacc);
    if (lane == 0) hp[hoff] = gacc / (1.0f + expf(-gacc)) * uacc;
  }

  // ---- prefetch the first unit batch of this warp's first down row ----
  const int tasks2 = a.T * H;
  const int nunits2 = a.k * updr;
  uint4 q0[kUnitBatch];
  uint32_t s0[kUnitBatch];
  if (gw < tasks2) {
    const int t = gw / H, n = gw - t * H;
#pragma unroll
    for (int m = 0; m < kUnitBatch; ++m) {
      const int u = lane + 32 * m;
      if (u < nunits2) {
        const int j = u / updr, c = u - j * updr;
        const uint8_t* rec = recs[t * a.k + j];
        if (rec) {
          q0[m] = moe::ldg_stream(rec + o.down + (size_t)n * (I / 2) + 16 * c);
          s0[m] = load_scale_bits<FMT>(rec + o.down_s + (size_t)n * (I / G) + sstep * c);
        }
      }
    }
  }

  if (!moe::grid_barrier(a.bar, gridDim.x, moe::global_ns() + 2000000000ull, &bar_ok)) {
    if (threadIdx.x == 0) moe::status_or(a.st, MOE_DEV_TIMEOUT);
    return;
  }

  // ---- stage h of every pair (L2 reads; written by other CTAs) ----
  {
    const float4* src = reinterpret_cast<const float4*>(a.hws);
    float4* dst = reinterpret_cast<float4*>(act);
    const int n16 = P * I / 4;
    for (int i = threadIdx.x; i < n16; i += kThreads) dst[i] = __ldcg(src + i);
  }
  __syncthreads();

  // ---- phase 2: one warp per (token, output row) ----
  for (int tau = gw; tau < tasks2; tau += NW) {
    const int t = tau / H, n = tau - t * H;
    float acc = 0.f;
    bool bad = false;
    for (int base = 0; base < nunits2; base += 32 * kUnitBatch) {
      uint4 q[kUnitBatch];
      uint32_t sb[kUnitBatch];
      const bool first = (tau == gw) && (base == 0);
#pragma unroll
      for (int m = 0; m < kUnitBatch; ++m) {
        const int u = base + lane + 32 * m;
        if (u < nunits2) {
          const int j = u / updr, c = u - j * updr;
          const uint8_t* rec = recs[t * a.k + j];
          if (first) {
            q[m] = q0[m];
            sb[m] = s0[m];
          } else if (rec) {
            q[m] = moe::ldg_stream(rec + o.down + (size_t)n * (I / 2) + 16 * c);
            sb[m] = load_scale_bits<FMT>(rec + o.down_s + (size_t)n * (I / G) + sstep * c);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kUnitBatch; ++m) {
        const int u = base + lane + 32 * m;
        if (u < nunits2) {
          const int j = u / updr, c = u - j * updr;
          const int pj = t * a.k + j;
          if (recs[pj]) {
            acc += wts[pj] * unit_dot_col<FMT>(q[m], sb[m], act + (size_t)pj * 16 * updr + c, updr);
          } else {
            bad = true;
          }
        }
      }
    }
    acc = moe::warp_sum(acc);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) a.y[(size_t)t * H + n] = bad ? __uint_as_float(0x7FC00000u) : acc;
  }
}

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

bool fused_fits(int T, int k, int H, int I) {
  const long long P = (long long)T * k;
  return P <= kFusedMaxPairs && (long long)T * H * 4 <= 96 * 1024 &&
         P * I * 4 <= 96 * 1024;
}

size_t fused_smem(int T, int k, int H, int I) {
  const size_t a = (size_t)T * H * 4, b = (size_t)T * k * I * 4;
  return a > b ? a : b;
}

template <int FMT>
int launch_fused(const FusedArgs& fa, cudaStream_t stream) {
  const size_t smem = fused_smem(fa.T, fa.k, fa.H, fa.I);
  static size_t granted = 0;
  if (!ensure_smem(decode_fused_kernel<FMT>, smem, &granted)) return MOE_ERR_CUDA;
  int dev = 0, sms = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_fused_kernel<FMT>, kThreads, smem) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  occ = occ < 1 ? 1 : (occ > 3 ? 3 : occ);
  // Grid = resident capacity, so every CTA is on an SM together (the grid
  // barrier needs that); its waits are bounded in any case.
  return moe::launch_pdl(decode_fused_kernel<FMT>, dim3(sms * occ), dim3(kThreads), smem, stream, fa);
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
  if (fused_fits(T, k, s.hidden, s.inter)) {
    FusedArgs fa;
    fa.x = x_bf16;
    fa.idx = idx;
    fa.w = weights;
    fa.T = T;
    fa.k = k;
    fa.ptrs = expert_ptrs;
    fa.E = E;
    fa.H = s.hidden;
    fa.I = s.inter;
    fa.hws = hws;
    fa.bar = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(workspace) +
                                         (size_t)T * k * s.inter * sizeof(float));
    fa.y = y;
    fa.st = dev_status;
    return s.format == MOE_FMT_NVFP4 ? launch_fused<MOE_FMT_NVFP4>(fa, st)
                                     : launch_fused<MOE_FMT_MXFP4>(fa, st);
  }
  if (s.format == MOE_FMT_NVFP4)
    return launch_decode<MOE_FMT_NVFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden,
                                        s.inter, y, hws, dev_status, st);
  return launch_decode<MOE_FMT_MXFP4>(x_bf16, idx, weights, T, k, expert_ptrs, E, s.hidden,
                                      s.inter, y, hws, dev_status, st);
}
