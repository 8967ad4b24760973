// FP8 (E4M3) row-scaled matrix-vector product.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": the large dense matrices are
// stored in FP8 with one scale per row; section "The engine", item 4: an FP8
// row-scaled matrix-vector kernel replaced a generic unpack path.
//
// HBM bound.  For K <= 4096 a warp owns one or two rows and issues every
// 16-byte load of them before it touches anything else, so the whole grid is
// one wave (the 8192 x 2560 matrix: 4096 warps, 64 rows per SM) and each SM
// keeps tens of KB of weights in flight from the first instruction on.  The
// weight loads are issued before the wait on the previous kernel of the stream
// (programmatic dependent launch), so they overlap its tail; x and the row
// scales are read after it.  x (BF16, a few KB) is read through L1, where the
// first warp of an SM leaves it for the others.  E4M3 pairs go through the
// hardware convert to f16x2 and are accumulated in FP32 with packed FMAs.
// Longer rows take a loop over 4 KB chunks of the row.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUPL = 8;  // 16-byte units per lane in flight (4 KB per warp)

// One 16-element unit: 16 E4M3 weights against x[16 c .. 16 c + 15], into the
// lane's two FP32 partial sums.
__device__ __forceinline__ void fp8_unit(const uint4 q, const uint16_t* __restrict__ x, int c, float2& acc) {
  const uint4 xa = __ldg(reinterpret_cast<const uint4*>(x + 16 * c));
  const uint4 xb = __ldg(reinterpret_cast<const uint4*>(x + 16 * c + 8));
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const float2 wf = moe::e4m3x2_to_f32x2(wd[wi] >> (16 * hi));
      const uint32_t xv = xw[2 * wi + hi];  // elements 4 wi + 2 hi, + 1
      const float2 xf = make_float2(moe::bf16_bits_to_f32(xv & 0xFFFFu), moe::bf16_bits_to_f32(xv >> 16));
      acc = moe::ffma2(wf, xf, acc);
    }
  }
}

__global__ void __launch_bounds__(kThreads) fp8_gemv_kernel(const uint8_t* __restrict__ w,
                                                           const float* __restrict__ rs,
                                                           const uint16_t* __restrict__ x,
                                                           int M, int K, float* __restrict__ y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kThreads / 32) + warp;
  if (m >= M) return;
  const uint8_t* row = w + (size_t)m * K;
  const int upr = K >> 4;  // 16-element units per row
  float2 acc = make_float2(0.f, 0.f);
  for (int base = 0; base < upr; base += 32 * kUPL) {
    uint4 q[kUPL];
#pragma unroll
    for (int i = 0; i < kUPL; ++i) {
      const int c = base + lane + 32 * i;
      q[i] = c < upr ? moe::ldg_stream(row + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kUPL; ++i) {
      const int c = base + lane + 32 * i;
      if (c < upr) fp8_unit(q[i], x, c, acc);
    }
  }
  const float s = moe::warp_sum(acc.x + acc.y);
  if (lane == 0) y[m] = rs[m] * s;
}

// Rows of at most 32 UPL units (K <= 512 UPL): warp g owns rows RPW g ..
// RPW g + RPW - 1, lane j units j, j + 32, ... of each, in the order of
// fp8_gemv_kernel (so the same sums, bit for bit).
template <int UPL, int RPW>
__global__ void __launch_bounds__(kThreads) fp8_gemv_rows_kernel(const uint8_t* __restrict__ w,
                                                                 const float* __restrict__ rs,
                                                                 const uint16_t* __restrict__ x,
                                                                 int M, int K, float* __restrict__ y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = (blockIdx.x * (kThreads / 32) + warp) * RPW;
  const int upr = K >> 4;
  uint4 q[RPW][UPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const uint8_t* row = w + (size_t)(m0 + r) * K;
#pragma unroll
    for (int i = 0; i < UPL; ++i) {
      const int c = lane + 32 * i;
      q[r][i] = (m0 + r < M && c < upr) ? moe::ldg_stream(row + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  moe::pdl_wait();  // x and the row scales may come from the previous kernel
  // the next kernel may start its own weight loads now; triggering earlier
  // would let a chain of such kernels pile up, each waiting on the one before
  moe::pdl_launch_dependents();
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    if (m0 + r >= M) break;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < UPL; ++i) {
      const int c = lane + 32 * i;
      if (c < upr) fp8_unit(q[r][i], x, c, acc);
    }
    const float s = moe::warp_sum(acc.x + acc.y);
    if (lane == 0) y[m0 + r] = rs[m0 + r] * s;
  }
}

template <int UPL>
int launch_rows(const uint8_t* w, const float* rs, const uint16_t* x, int M, int K, float* y, cudaStream_t st) {
  constexpr int RPW = UPL <= 5 ? 2 : 1;  // at most 10 units (160 B) per lane in flight
  const long long warps = ((long long)M + RPW - 1) / RPW;
  const unsigned grid = (unsigned)((warps + kThreads / 32 - 1) / (kThreads / 32));
  return moe::launch_pdl(fp8_gemv_rows_kernel<UPL, RPW>, dim3(grid), dim3(kThreads), 0, st, w, rs, x, M, K, y);
}

}  // namespace

extern "C" int fp8_rowscale_gemv(const uint8_t* w_e4m3, const float* row_scale,
                                 const uint16_t* x_bf16, int M, int K, float* y, void* stream) {
  if (!w_e4m3 || !row_scale || !x_bf16 || !y || M < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 32768) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(w_e4m3) || !moe::aligned16(x_bf16)) return MOE_ERR_ALIGNMENT;
  if (M == 0) return MOE_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  switch ((K / 16 + 31) / 32) {  // 16-element units per lane
    case 1: return launch_rows<1>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 2: return launch_rows<2>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 3: return launch_rows<3>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 4: return launch_rows<4>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 5: return launch_rows<5>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 6: return launch_rows<6>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 7: return launch_rows<7>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    case 8: return launch_rows<8>(w_e4m3, row_scale, x_bf16, M, K, y, st);
    default: break;
  }
  const int grid = (M + kThreads / 32 - 1) / (kThreads / 32);
  fp8_gemv_kernel<<<grid, kThreads, 0, st>>>(w_e4m3, row_scale, x_bf16, M, K, y);
  return moe::launch_status();
}
