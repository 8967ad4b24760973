// Router: FP32 logits in a fixed summation order, top-k with renormalised
// softmax weights, and the RMS chaining step between stacked decode layers.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": top-10 of 512 experts per
// layer; section "Where the time actually goes": the expert work of a layer
// waits on the router's answer, so routing stays on the device here and no
// index ever travels to the host.
#include "common.cuh"

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
  int my_e = 0;
  float my_l = 0.0f;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < EPL; ++i) best = cand[i] > best ? cand[i] : best;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, d);
      best = o > best ? o : best;
    }
    const int e = (int)(~(uint32_t)(best & 0xFFFFFFFFull));
    if ((e & 31) == lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == (e >> 5)) cand[i] = 0ull;
    }
    if (lane == r) {
      my_e = e;
      my_l = key_to_float((uint32_t)(best >> 32));
    }
  }
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.0f;
  const float sum = moe::warp_sum(ex);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    weights[(size_t)t * k + lane] = __fdiv_rn(ex, sum);
  }
}

// ---------------------------------------------------------------------------
// RMS chaining: one CTA per token, FP64 mean of squares in a fixed tree, one
// rounding to BF16 (ties to even) from FP64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t f64_to_bf16_rn(double v) {
  if (v == 0.0 || !isfinite(v)) {
    const float f = (float)v;  // zero, inf and NaN convert exactly enough
    uint32_t b = __float_as_uint(f);
    if (f != f) b = 0x7FC00000u;
    return (uint16_t)(b >> 16);
  }
  const double a = fabs(v);
  const int e = ilogb(a);
  const int qe = max(e - 7, -133);
  const double q = rint(scalbn(a, -qe));
  double r = scalbn(q, qe);
  uint32_t bits;
  if (r >= 0x1.ffp127) {
    bits = 0x7F800000u;
  } else {
    bits = __float_as_uint((float)r);  // exact: r has at most 8 significant bits
  }
  if (v < 0) bits |= 0x80000000u;
  return (uint16_t)(bits >> 16);
}

__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ y, int H,
                                                           double eps,
                                                           uint16_t* __restrict__ x) {
  __shared__ double part[256];
  moe::pdl_launch_dependents();
  moe::pdl_wait();
  const int t = blockIdx.x;
  const float* yr = y + (size_t)t * H;
  double s = 0.0;
  for (int i = threadIdx.x; i < H; i += 256) {
    const double v = (double)yr[i];
    s = fma(v, v, s);
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  const double inv = 1.0 / sqrt(part[0] / (double)H + eps);
  for (int i = threadIdx.x; i < H; i += 256) x[(size_t)t * H + i] = f64_to_bf16_rn((double)yr[i] * inv);
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
                         eps, x_bf16);
}
