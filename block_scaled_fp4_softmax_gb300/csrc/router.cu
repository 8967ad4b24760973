// Router: FP32 logits in a fixed summation order, top-k with renormalised
// softmax weights, and the RMS chaining step between stacked decode layers.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": top-10 of 512 experts per
// layer; section "Where the time actually goes": the expert work of a layer
// waits on the router's answer, so routing stays on the device here and no
// index ever travels to the host.
#include "common.cuh"
#include "router_math.cuh"
#include "tcgen05.cuh"

namespace {

// ---------------------------------------------------------------------------
// Logits.  A warp owns TT tokens x EW experts.  Lane j walks the chunks of 8
// elements c = j, j+32, j+64, ... (ascending), elements inside a chunk in
// order, one FMA each (the BF16 x BF16 product is exact, so the FMA is the
// FP32 add of the exact product).  The 32 lane sums are then combined with an
// xor butterfly d = 16, 8, 4, 2, 1 and the bias is added last.  This is the
// order moe.h documents; it makes the logits, and so the top-k choice,
// reproducible bit for bit.
// ---------------------------------------------------------------------------
template <int TT, int EW>
__global__ void __launch_bounds__(256) router_logits_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ bias,
    int T, int H, int E, float* __restrict__ logits) {
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int e_tiles = (E + EW - 1) / EW;
  const int t0 = (warp / e_tiles) * TT;
  const int e0 = (warp % e_tiles) * EW;
  if (t0 >= T) return;

  float acc[TT][EW];
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < EW; ++b) acc[a][b] = 0.0f;

  const uint16_t* xr[TT];
  const uint16_t* wrr[EW];
#pragma unroll
  for (int a = 0; a < TT; ++a) xr[a] = x + (size_t)min(t0 + a, T - 1) * H;
#pragma unroll
  for (int b = 0; b < EW; ++b) wrr[b] = wr + (size_t)min(e0 + b, E - 1) * H;

  const int nchunk = H >> 3;
#pragma unroll 2
  for (int c = lane; c < nchunk; c += 32) {
    uint4 xv[TT], wv[EW];
#pragma unroll
    for (int a = 0; a < TT; ++a) xv[a] = __ldg(reinterpret_cast<const uint4*>(xr[a] + 8 * c));
#pragma unroll
    for (int b = 0; b < EW; ++b) wv[b] = __ldg(reinterpret_cast<const uint4*>(wrr[b] + 8 * c));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int a = 0; a < TT; ++a) {
        const uint32_t xw = (&xv[a].x)[i >> 1] >> (16 * (i & 1));
#pragma unroll
        for (int b = 0; b < EW; ++b) acc[a][b] = moe::fma_bf16(xw, (&wv[b].x)[i >> 1] >> (16 * (i & 1)), acc[a][b]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < EW; ++b) {
      float v = acc[a][b];
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
      acc[a][b] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int b = 0; b < EW; ++b) {
        const int t = t0 + a, e = e0 + b;
        if (t < T && e < E) {
          float v = acc[a][b];
          if (bias) v = __fadd_rn(v, bias[e]);
          logits[(size_t)t * E + e] = v;
        }
      }
  }
}

// ---------------------------------------------------------------------------
// Logits for many tokens, the same order as router_logits_kernel: a CTA owns
// 32 tokens x 2 WE experts and walks H in K-steps of 256 elements (32 chunks
// of 8), staging both BF16 tiles in shared memory with cp.async, three
// buffers deep.  Warp w owns tokens 8 (w >> 1) .. +8 and experts WE (w & 1) ..
// +WE; in K-step ks its lane j takes chunk 32 ks + j of every row, so lane j
// still walks chunks j, j + 32, ... in ascending order with one FMA per
// element, and the 32 lane sums meet in the same xor butterfly.  The FMAs take
// the BF16 halves as they are (fma.rn.f32.bf16: both factors are exact in
// FP32, so this is the FP32 FMA of the converted values).  Needs H % 256 == 0.
// ---------------------------------------------------------------------------
constexpr int kRtTok = 32, kRtK = 256, kRtWTok = 8, kRtStages = 3;
template <int WE>
constexpr int rt_stage_bytes() { return (kRtTok + 2 * WE) * kRtK * 2; }

template <int WE>
__global__ void __launch_bounds__(256) router_logits_tiled_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ bias,
    int T, int H, int E, float* __restrict__ logits) {
  constexpr int kExp = 2 * WE, kStage = rt_stage_bytes<WE>();
  extern __shared__ __align__(128) uint8_t rsm[];
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t_cta = blockIdx.x * kRtTok, e_cta = blockIdx.y * kExp;
  const int ta = (warp >> 1) * kRtWTok, ea = (warp & 1) * WE;  // the warp's rows in the tile
  const int nks = H / kRtK;
  // staging: lane j copies the 16-byte piece j of tile rows warp, warp + 8,
  // ...: x rows 0..31 (clamped to T - 1), then W_r rows (clamped to E - 1)
  constexpr int kRows = kRtTok + kExp, kPer = kRows / 8;
  const uint16_t* src[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int r = warp + 8 * j;
    src[j] = (r < kRtTok ? x + (size_t)min(t_cta + r, T - 1) * H : wr + (size_t)min(e_cta + r - kRtTok, E - 1) * H) +
             8 * lane;
  }
  const uint32_t dst0 = moe::tc::smem_u32(rsm) + (uint32_t)(warp * kRtK + 8 * lane) * 2u;
  auto stage = [&](int ks, int buf) {
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      moe::tc::cp_async16(dst0 + (uint32_t)(buf * kStage + j * 8 * kRtK * 2), src[j] + (size_t)ks * kRtK, 16u);
    moe::tc::cp_async_commit();
  };
  float acc[kRtWTok][WE];
#pragma unroll
  for (int a = 0; a < kRtWTok; ++a)
#pragma unroll
    for (int b = 0; b < WE; ++b) acc[a][b] = 0.0f;
  // three buffers: K-steps ks + 1 and ks + 2 are in flight while ks is
  // summed; one barrier per K-step both publishes buffer ks and retires the
  // buffer that K-step ks + 2 then refills (last read in K-step ks - 1)
  stage(0, 0);
  if (nks > 1) stage(1, 1);
  for (int ks = 0; ks < nks; ++ks) {
    if (ks + 1 < nks) moe::tc::cp_async_wait<1>();
    else moe::tc::cp_async_wait<0>();
    __syncthreads();
    if (ks + 2 < nks) stage(ks + 2, (ks + 2) % kRtStages);
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(rsm + (ks % kRtStages) * kStage);
    const uint16_t* ws = xs + kRtTok * kRtK;
    uint4 wv[WE];
#pragma unroll
    for (int b = 0; b < WE; ++b) wv[b] = *reinterpret_cast<const uint4*>(ws + (ea + b) * kRtK + 8 * lane);
#pragma unroll
    for (int a = 0; a < kRtWTok; ++a) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xs + (ta + a) * kRtK + 8 * lane);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t xw = (&xv.x)[i >> 1] >> (16 * (i & 1));
#pragma unroll
        for (int b = 0; b < WE; ++b) acc[a][b] = moe::fma_bf16(xw, (&wv[b].x)[i >> 1] >> (16 * (i & 1)), acc[a][b]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < kRtWTok; ++a)
#pragma unroll
    for (int b = 0; b < WE; ++b) {
      float v = acc[a][b];
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
      acc[a][b] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int a = 0; a < kRtWTok; ++a)
#pragma unroll
      for (int b = 0; b < WE; ++b) {
        const int t = t_cta + ta + a, e = e_cta + ea + b;
        if (t < T && e < E) {
          float v = acc[a][b];
          if (bias) v = __fadd_rn(v, bias[e]);
          logits[(size_t)t * E + e] = v;
        }
      }
  }
}

// ---------------------------------------------------------------------------
// Top-k.  One block of kTopkThreads per token, candidates keyed by (ordered
// logit, ~expert): every warp picks the k best of its share, warp 0 merges
// those sorted lists (moe::rt::topk_block, behind the filter of
// moe::rt::topk_block_fast); weights renormalised over the
// picks.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 512;
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                            int k, int32_t* __restrict__ idx,
                                                            float* __restrict__ weights) {
  __shared__ unsigned long long fin[kTopkThreads];
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int lane = threadIdx.x & 31, t = blockIdx.x;
  int my_e = 0;
  float my_l = 0.0f;
  moe::rt::topk_block_fast<kTopkThreads / 32>(logits + (size_t)t * E, E, k, fin, my_e, my_l);
  if (threadIdx.x < 32) {
    const float w = moe::rt::topk_weight(lane, k, my_l);
    if (lane < k) {
      idx[(size_t)t * k + lane] = my_e;
      weights[(size_t)t * k + lane] = w;
    }
  }
}

// ---------------------------------------------------------------------------
// RMS chaining in FP32 in one fixed order (moe::rt::rms_inv_fixed_order),
// x = BF16_rn(y * r).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ y, int H,
                                                           float eps,
                                                           uint16_t* __restrict__ x) {
  __shared__ float part[256];
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int t = blockIdx.x;
  const float* yr = y + (size_t)t * H;
  const float r = moe::rt::rms_inv_fixed_order(yr, H, eps, part);
  for (int i = threadIdx.x; i < H; i += 256) x[(size_t)t * H + i] = moe::rt::f32_to_bf16_bits(__fmul_rn(yr[i], r));
}

// ---------------------------------------------------------------------------
// Small-T router logits over the whole GPU.  CTA b owns experts
// [b*epc, (b+1)*epc).  Before it waits on the previous kernel it pulls its
// W_r rows into L2 (the weights never depend on that kernel); then it builds
// x (from x_bf16, or as RMS chaining of the previous layer's y -- every CTA
// computes the same fixed-order result, CTA 0 writes it out) and one warp
// per (token, expert) computes the logit in the fixed order of
// router_logits_kernel.  The top-k follows in topk_kernel.  The kernel needs
// a few KB of shared memory, so its CTAs fit beside a running expert pass.
// ---------------------------------------------------------------------------
constexpr int kGridThreads = 256;
constexpr int kGridMaxXBytes = 40 * 1024;

struct GridArgs {
  const uint16_t* x;    // [T, H] BF16, or NULL when y_prev is given
  const float* y_prev;  // [T, H] FP32 to RMS-normalise, or NULL
  float eps;
  uint16_t* x_out;      // written by CTA 0 when y_prev is given
  const uint16_t* wr;
  const float* bias;
  int T, H, E, epc;     // experts per CTA
  float* logits;
};

__global__ void __launch_bounds__(kGridThreads) router_grid_kernel(GridArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  float* part = reinterpret_cast<float*>(sm);             // [256]
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm + 1024);  // [T][H] BF16
  const int e0 = blockIdx.x * a.epc;
  const int ne = max(0, min(a.epc, a.E - e0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    const char* wb = reinterpret_cast<const char*>(a.wr + (size_t)e0 * a.H);
    const size_t bytes = (size_t)ne * a.H * 2;
    for (size_t off = (size_t)threadIdx.x * 128; off < bytes; off += (size_t)kGridThreads * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(wb + off));
  }
  moe::pdl_launch_dependents();
  moe::pdl_wait();

  for (int t = 0; t < a.T; ++t) {
    if (a.y_prev) {
      const float* yr = a.y_prev + (size_t)t * a.H;
      const float r = moe::rt::rms_inv_fixed_order(yr, a.H, a.eps, part);
      constexpr int kBatch = 8;
      for (int i0 = threadIdx.x; i0 < a.H; i0 += kGridThreads * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) v[b] = i0 + kGridThreads * b < a.H ? yr[i0 + kGridThreads * b] : 0.0f;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int i = i0 + kGridThreads * b;
          if (i < a.H) {
            const uint16_t x16 = moe::rt::f32_to_bf16_bits(__fmul_rn(v[b], r));
            xs[(size_t)t * a.H + i] = x16;
            if (blockIdx.x == 0 && a.x_out) a.x_out[(size_t)t * a.H + i] = x16;
          }
        }
      }
    } else {
      for (int i = threadIdx.x * 8; i < a.H; i += kGridThreads * 8)
        *reinterpret_cast<uint4*>(xs + (size_t)t * a.H + i) =
            __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H + i));
    }
  }
  __syncthreads();

  // logits: task (token t, expert q) -> warp, in the fixed order
  for (int task = warp; task < a.T * ne; task += kGridThreads / 32) {
    const int t = task / ne, q = task - t * ne;
    const float acc = moe::rt::logit_dot(xs + (size_t)t * a.H, a.wr + (size_t)(e0 + q) * a.H, a.H, lane);
    if (lane == 0) {
      const int e = e0 + q;
      a.logits[(size_t)t * a.E + e] = a.bias ? __fadd_rn(acc, a.bias[e]) : acc;
    }
  }
}

int sm_count_router() { return moe::device_info().sms; }

bool grid_fits(int T, int H, int E) {
  return T >= 1 && (size_t)T * H * 2 <= kGridMaxXBytes && E <= 1024 && H % 8 == 0 &&
         sm_count_router() > 0;
}

int launch_topk(const float* logits, int T, int E, int k, int32_t* idx, float* weights, cudaStream_t st) {
  return moe::launch_pdl(topk_kernel, dim3(T), dim3(kTopkThreads), 0, st, logits, T, E, k, idx, weights);
}

// Logits on the whole GPU, then the top-k.
int launch_grid_router(const GridArgs& a0, int k, int32_t* idx, float* weights, cudaStream_t st) {
  GridArgs a = a0;
  const int sms = sm_count_router();
  a.epc = (a.E + sms - 1) / sms;
  const int grid = (a.E + a.epc - 1) / a.epc;
  const size_t smem = 1024 + (size_t)a.T * a.H * 2;
  static moe::SmemGrant granted;
  if (!moe::grant_smem(router_grid_kernel, smem, granted)) return MOE_ERR_CUDA;
  const int rc = moe::launch_pdl(router_grid_kernel, dim3(grid), dim3(kGridThreads), smem, st, a);
  if (rc != MOE_OK) return rc;
  return launch_topk(a.logits, a.T, a.E, k, idx, weights, st);
}

}  // namespace

extern "C" int moe_router_topk(const uint16_t* x_bf16, const uint16_t* wr_bf16, const float* bias,
                               int T, int H, int E, int k, int32_t* idx, float* weights,
                               float* logits, void* stream) {
  if (!x_bf16 || !wr_bf16 || !idx || !weights || !logits) return MOE_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(x_bf16) || !moe::aligned16(wr_bf16)) return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (grid_fits(T, H, E)) {
    GridArgs a = {};
    a.x = x_bf16;
    a.wr = wr_bf16;
    a.bias = bias;
    a.T = T;
    a.H = H;
    a.E = E;
    a.logits = logits;
    return launch_grid_router(a, k, idx, weights, st);
  }
  const int threads = 256;
  int rc;
  if (T < 4) {
    const long long warps = (long long)T * E;
    rc = moe::launch_pdl(router_logits_kernel<1, 1>, dim3((unsigned)((warps * 32 + threads - 1) / threads)),
                         dim3(threads), 0, st, x_bf16, wr_bf16, bias, T, H, E, logits);
  } else if (T < 64 || H % kRtK != 0) {
    const long long warps = (long long)((T + 3) / 4) * ((E + 3) / 4);
    rc = moe::launch_pdl(router_logits_kernel<4, 4>, dim3((unsigned)((warps * 32 + threads - 1) / threads)),
                         dim3(threads), 0, st, x_bf16, wr_bf16, bias, T, H, E, logits);
  } else {
    // many tokens: shared-memory tiles of 32 tokens x 8 experts, 3 x 20 KB
    constexpr int WE = 4;
    static moe::SmemGrant granted;
    if (!moe::grant_smem(router_logits_tiled_kernel<WE>, kRtStages * rt_stage_bytes<WE>(), granted))
      return MOE_ERR_CUDA;
    rc = moe::launch_pdl(router_logits_tiled_kernel<WE>, dim3((unsigned)((T + kRtTok - 1) / kRtTok),
                                                              (unsigned)((E + 2 * WE - 1) / (2 * WE))),
                         dim3(256), kRtStages * rt_stage_bytes<WE>(), st, x_bf16, wr_bf16, bias, T, H, E, logits);
  }
  if (rc != MOE_OK) return rc;
  return launch_topk(logits, T, E, k, idx, weights, st);
}

extern "C" int moe_rmsnorm_bf16(const float* y, int T, int H, double eps, uint16_t* x_bf16,
                                void* stream) {
  if (!y || !x_bf16 || T < 0 || H <= 0 || !(eps >= 0.0)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  return moe::launch_pdl(rmsnorm_bf16_kernel, dim3(T), dim3(256), 0, (cudaStream_t)stream, y, H,
                         (float)eps, x_bf16);
}

extern "C" int moe_rmsnorm_router_topk(const float* y_prev, int T, int H, double eps,
                                       uint16_t* x_out, const uint16_t* wr_bf16, const float* bias,
                                       int E, int k, int32_t* idx, float* weights, float* logits,
                                       void* stream) {
  if (!y_prev || !x_out || !wr_bf16 || !idx || !weights || !logits) return MOE_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || k > 32 || !(eps >= 0.0))
    return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(wr_bf16) || !moe::aligned16(x_out)) return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (grid_fits(T, H, E)) {
    GridArgs a = {};
    a.y_prev = y_prev;
    a.eps = (float)eps;
    a.x_out = x_out;
    a.wr = wr_bf16;
    a.bias = bias;
    a.T = T;
    a.H = H;
    a.E = E;
    a.logits = logits;
    return launch_grid_router(a, k, idx, weights, st);
  }
  int rc = moe_rmsnorm_bf16(y_prev, T, H, eps, x_out, stream);
  if (rc != MOE_OK) return rc;
  return moe_router_topk(x_out, wr_bf16, bias, T, H, E, k, idx, weights, logits, stream);
}
