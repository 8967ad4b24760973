// Router: FP32 logits in a fixed summation order, top-k with renormalised
// softmax weights, and the RMS chaining step between stacked decode layers.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": top-10 of 512 experts per
// layer; section "Where the time actually goes": the expert work of a layer
// waits on the router's answer, so routing stays on the device here and no
// index ever travels to the host.
#include "common.cuh"
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
        const uint32_t xw = (&xv[a].x)[i >> 1];
        const float xf = moe::bf16_bits_to_f32((i & 1) ? (xw >> 16) : (xw & 0xFFFFu));
#pragma unroll
        for (int b = 0; b < EW; ++b) {
          const uint32_t ww = (&wv[b].x)[i >> 1];
          const float wf = moe::bf16_bits_to_f32((i & 1) ? (ww >> 16) : (ww & 0xFFFFu));
          acc[a][b] = __fmaf_rn(xf, wf, acc[a][b]);
        }
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
// Top-k.  One warp per token.  Each candidate gets a 64-bit key
// (ordered logit bits << 32 | ~expert) so that the maximum is the larger logit
// and, on equal logits, the lower expert index.  NaN ranks below -inf, -0
// counts as +0.  k rounds of warp arg-max pick the experts in order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_key(float v) {
  if (v != v) return 1u;
  if (v == 0.0f) v = 0.0f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  if (k == 1u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Selects the k best of the lanes' candidates (composite keys, unique): round
// r takes the largest key below round r-1's winner, so nothing is ever
// removed and the candidate array stays in registers.  Lane r ends with
// expert r and its logit.
template <int EPL>
__device__ __forceinline__ void warp_select_topk(const unsigned long long (&cand)[EPL], int k,
                                                 int lane, int& my_e, float& my_l) {
  unsigned long long prev = ~0ull;
  my_e = 0;
  my_l = 0.0f;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (cand[i] < prev && cand[i] > best) best = cand[i];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, d);
      best = o > best ? o : best;
    }
    prev = best;
    if (lane == r) {
      my_e = (int)(~(uint32_t)(best & 0xFFFFFFFFull));
      my_l = key_to_float((uint32_t)(best >> 32));
    }
  }
}

// Writes idx/weights of one token from the selection above.
__device__ __forceinline__ void write_topk(int lane, int k, int my_e, float my_l, int32_t* idx,
                                           float* weights) {
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.0f;
  const float sum = moe::warp_sum(ex);
  if (lane < k) {
    idx[lane] = my_e;
    weights[lane] = __fdiv_rn(ex, sum);
  }
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                   int k, int32_t* __restrict__ idx,
                                                   float* __restrict__ weights) {
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  unsigned long long cand[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    cand[i] = 0ull;
    if (e < E) {
      const uint32_t key = ordered_key(logits[(size_t)t * E + e]);
      cand[i] = ((unsigned long long)key << 32) | (unsigned long long)(~(uint32_t)e);
    }
  }
  int my_e;
  float my_l;
  warp_select_topk<EPL>(cand, k, lane, my_e, my_l);
  write_topk(lane, k, my_e, my_l, idx + (size_t)t * k, weights + (size_t)t * k);
}

// ---------------------------------------------------------------------------
// RMS chaining in FP32, one fixed order (so the BF16 result is reproducible):
// thread t of 256 sums y[t + 256 m]^2 for m ascending (square rounded, then
// added), a pairwise tree combines the 256 partial sums, mean = sum / H,
// r = 1 / sqrt(mean + eps) with IEEE sqrt and divide, x = BF16_rn(y * r).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float rms_inv_fixed_order(const float* __restrict__ yr, int H, float eps,
                                                     float* part) {
  float acc = 0.0f;
  for (int i = threadIdx.x; i < H; i += 256) {
    const float v = yr[i];
    acc = __fadd_rn(acc, __fmul_rn(v, v));
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] = __fadd_rn(part[threadIdx.x], part[threadIdx.x + w]);
    __syncthreads();
  }
  const float mean = __fdiv_rn(part[0], (float)H);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
  __syncthreads();  // part[] may be reused by the caller
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ y, int H,
                                                           float eps,
                                                           uint16_t* __restrict__ x) {
  __shared__ float part[256];
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int t = blockIdx.x;
  const float* yr = y + (size_t)t * H;
  const float r = rms_inv_fixed_order(yr, H, eps, part);
  for (int i = threadIdx.x; i < H; i += 256) x[(size_t)t * H + i] = f32_to_bf16_bits(__fmul_rn(yr[i], r));
}

// ---------------------------------------------------------------------------
// Small-T router in one launch: a cluster of kCl CTAs.  Each CTA pulls its
// contiguous slice of W_r rows into shared memory with one bulk copy issued
// before it waits on the previous kernel (the weights never depend on it),
// builds x (from x_bf16, or as RMS chaining of the previous layer's y), and
// computes its experts' logits in the fixed order.  After a cluster barrier,
// CTA 0 reads every CTA's logits through distributed shared memory and runs
// the top-k + softmax per token.
// ---------------------------------------------------------------------------
constexpr int kCl = 16;
constexpr int kClThreads = 256;
constexpr int kClMaxT = 4;

struct ClusterArgs {
  const uint16_t* x;    // [T, H] BF16, or NULL when y_prev is given
  const float* y_prev;  // [T, H] FP32 to RMS-normalise, or NULL
  float eps;
  uint16_t* x_out;      // written by CTA 0 when y_prev is given (may be NULL otherwise)
  const uint16_t* wr;
  const float* bias;
  int T, H, E, k, epc;  // experts per CTA
  int32_t* idx;
  float* weights;
  float* logits;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float dsmem_ld_f32(const float* local_addr, uint32_t rank) {
  uint32_t a = moe::tc::smem_u32(local_addr), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

template <int EPL>
__device__ __forceinline__ void cluster_topk(const ClusterArgs& a, const float* lg, int t, int lane) {
  unsigned long long cand[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    cand[i] = 0ull;
    const int e = lane + 32 * i;
    if (e < a.E) {
      const uint32_t owner = (uint32_t)(e / a.epc);
      const float v = dsmem_ld_f32(lg + t * a.epc + (e - (int)owner * a.epc), owner);
      cand[i] = ((unsigned long long)ordered_key(v) << 32) | (unsigned long long)(~(uint32_t)e);
    }
  }
  int my_e;
  float my_l;
  warp_select_topk<EPL>(cand, a.k, lane, my_e, my_l);
  write_topk(lane, a.k, my_e, my_l, a.idx + (size_t)t * a.k, a.weights + (size_t)t * a.k);
}

__global__ void __launch_bounds__(kClThreads) router_cluster_kernel(ClusterArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* wbar = reinterpret_cast<uint64_t*>(sm);
  float* part = reinterpret_cast<float*>(sm + 16);                   // [256]
  float* lg = reinterpret_cast<float*>(sm + 16 + 256 * 8);           // [kClMaxT][epc]
  uint16_t* xs = reinterpret_cast<uint16_t*>(lg + kClMaxT * a.epc);  // [T][H] BF16
  uint16_t* ws = reinterpret_cast<uint16_t*>(
      (reinterpret_cast<uintptr_t>(xs + (size_t)a.T * a.H) + 127) & ~(uintptr_t)127);  // [epc][H]
  const uint32_t rank = cluster_ctarank();
  const int e0 = (int)rank * a.epc;
  const int ne = max(0, min(a.epc, a.E - e0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool wok = true;

  if (threadIdx.x == 0) {
    moe::tc::mbar_init(wbar, 1);
    moe::tc::mbar_fence_init();
  }
  __syncthreads();
  if (warp == 0) {
    // one bulk copy per W_r row, spread over the lanes of warp 0
    const uint32_t row_bytes = (uint32_t)a.H * 2;
    if (lane == 0) moe::tc::mbar_arrive_expect_tx(wbar, (uint32_t)ne * row_bytes);
    __syncwarp();
    for (int q = lane; q < ne; q += 32)
      moe::tc::bulk_g2s(moe::tc::smem_u32(ws + (size_t)q * a.H), a.wr + (size_t)(e0 + q) * a.H,
                        row_bytes, wbar);
  }
  moe::pdl_launch_dependents();
  moe::pdl_wait();

  // x for every token
  for (int t = 0; t < a.T; ++t) {
    if (a.y_prev) {
      const float* yr = a.y_prev + (size_t)t * a.H;
      const float r = rms_inv_fixed_order(yr, a.H, a.eps, part);
      for (int i = threadIdx.x; i < a.H; i += kClThreads) {
        const uint16_t b = f32_to_bf16_bits(__fmul_rn(yr[i], r));
        xs[(size_t)t * a.H + i] = b;
        if (rank == 0 && a.x_out) a.x_out[(size_t)t * a.H + i] = b;
      }
    } else {
      for (int i = threadIdx.x * 8; i < a.H; i += kClThreads * 8)
        *reinterpret_cast<uint4*>(xs + (size_t)t * a.H + i) =
            __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H + i));
    }
  }
  __syncthreads();
  if (!moe::tc::mbar_wait(wbar, 0, moe::global_ns() + 2000000000ull)) wok = false;

  // logits: warp -> expert, lane j -> chunks j, j+32, ... (fixed order)
  const int nchunk = a.H >> 3;
  for (int q = warp; q < ne; q += kClThreads / 32) {
    float acc[kClMaxT];
#pragma unroll
    for (int t = 0; t < kClMaxT; ++t) acc[t] = 0.0f;
    const uint16_t* wrow = ws + (size_t)q * a.H;
    for (int c = lane; c < nchunk; c += 32) {
      const uint4 wv = *reinterpret_cast<const uint4*>(wrow + 8 * c);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int t = 0; t < kClMaxT; ++t) {
        if (t < a.T) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)t * a.H + 8 * c);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float xf = moe::bf16_bits_to_f32((i & 1) ? (xw[i >> 1] >> 16) : (xw[i >> 1] & 0xFFFFu));
            const float wf = moe::bf16_bits_to_f32((i & 1) ? (ww[i >> 1] >> 16) : (ww[i >> 1] & 0xFFFFu));
            acc[t] = __fmaf_rn(xf, wf, acc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kClMaxT; ++t) {
      float v = acc[t];
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
      if (t < a.T && lane == 0) {
        const int e = e0 + q;
        if (a.bias) v = __fadd_rn(v, a.bias[e]);
        if (!wok) v = __uint_as_float(0x7FC00000u);
        lg[t * a.epc + q] = v;
        a.logits[(size_t)t * a.E + e] = v;
      }
    }
  }
  cluster_sync_all();

  // top-k in CTA 0, one warp per token, candidates read over DSMEM
  if (rank == 0 && warp < a.T) {
    const int epl = (a.E + 31) / 32;
    if (epl <= 1) cluster_topk<1>(a, lg, warp, lane);
    else if (epl <= 2) cluster_topk<2>(a, lg, warp, lane);
    else if (epl <= 4) cluster_topk<4>(a, lg, warp, lane);
    else if (epl <= 8) cluster_topk<8>(a, lg, warp, lane);
    else if (epl <= 16) cluster_topk<16>(a, lg, warp, lane);
    else cluster_topk<32>(a, lg, warp, lane);
  }
  cluster_sync_all();  // keep every CTA's shared memory alive until CTA 0 is done
}

size_t cluster_smem(int T, int H, int epc) {
  return 16 + 256 * 8 + (size_t)kClMaxT * epc * 4 + (size_t)T * H * 2 + 128 + (size_t)epc * H * 2;
}

int cluster_smem_limit() {
  static int limit = -1;
  if (limit < 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      limit = 0;
  }
  return limit;
}

bool cluster_fits(int T, int H, int E) {
  const int epc = (E + kCl - 1) / kCl;
  return T >= 1 && T <= kClMaxT && E <= 1024 && H % 8 == 0 &&
         cluster_smem(T, H, epc) <= (size_t)cluster_smem_limit();
}

int launch_cluster_router(const ClusterArgs& a0, cudaStream_t st) {
  ClusterArgs a = a0;
  a.epc = (a.E + kCl - 1) / kCl;
  const size_t smem = cluster_smem(a.T, a.H, a.epc);
  static size_t granted = 0;
  static bool nonportable = false;
  if (!nonportable) {
    if (cudaFuncSetAttribute(router_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    nonportable = true;
  }
  if (smem > granted) {
    if (cudaFuncSetAttribute(router_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    granted = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCl);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_cluster_kernel, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
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
  if (cluster_fits(T, H, E)) {
    ClusterArgs a = {};
    a.x = x_bf16;
    a.wr = wr_bf16;
    a.bias = bias;
    a.T = T;
    a.H = H;
    a.E = E;
    a.k = k;
    a.idx = idx;
    a.weights = weights;
    a.logits = logits;
    return launch_cluster_router(a, st);
  }
  const int threads = 256;
  int rc;
  if (T < 4) {
    const long long warps = (long long)T * E;
    rc = moe::launch_pdl(router_logits_kernel<1, 1>, dim3((unsigned)((warps * 32 + threads - 1) / threads)),
                         dim3(threads), 0, st, x_bf16, wr_bf16, bias, T, H, E, logits);
  } else {
    const long long warps = (long long)((T + 3) / 4) * ((E + 3) / 4);
    rc = moe::launch_pdl(router_logits_kernel<4, 4>, dim3((unsigned)((warps * 32 + threads - 1) / threads)),
                         dim3(threads), 0, st, x_bf16, wr_bf16, bias, T, H, E, logits);
  }
  if (rc != MOE_OK) return rc;
  const dim3 grid((unsigned)(((long long)T * 32 + threads - 1) / threads));
  const int epl = (E + 31) / 32;
  if (epl <= 1) rc = moe::launch_pdl(topk_kernel<1>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  else if (epl <= 2) rc = moe::launch_pdl(topk_kernel<2>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  else if (epl <= 4) rc = moe::launch_pdl(topk_kernel<4>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  else if (epl <= 8) rc = moe::launch_pdl(topk_kernel<8>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  else if (epl <= 16) rc = moe::launch_pdl(topk_kernel<16>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  else rc = moe::launch_pdl(topk_kernel<32>, grid, dim3(threads), 0, st, logits, T, E, k, idx, weights);
  return rc;
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
  if (cluster_fits(T, H, E)) {
    ClusterArgs a = {};
    a.y_prev = y_prev;
    a.eps = (float)eps;
    a.x_out = x_out;
    a.wr = wr_bf16;
    a.bias = bias;
    a.T = T;
    a.H = H;
    a.E = E;
    a.k = k;
    a.idx = idx;
    a.weights = weights;
    a.logits = logits;
    return launch_cluster_router(a, st);
  }
  int rc = moe_rmsnorm_bf16(y_prev, T, H, eps, x_out, stream);
  if (rc != MOE_OK) return rc;
  return moe_router_topk(x_out, wr_bf16, bias, T, H, E, k, idx, weights, logits, stream);
}
