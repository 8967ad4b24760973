// FP8 (E4M3) row-scaled matrix-vector product.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": the large dense matrices are
// stored in FP8 with one scale per row; section "The engine", item 4: an FP8
// row-scaled matrix-vector kernel replaced a generic unpack path.
//
// HBM bound: one warp per row, and the warp issues every 16-byte load of its
// row chunk (up to 4 KB) before it touches x, so each SM keeps tens of KB of
// weights in flight from the first instruction on.  x (BF16, a few KB) is read
// through L1, where the first warp of an SM leaves it for the others.  E4M3
// pairs go through the hardware convert to f16x2 and are accumulated in FP32
// with packed FMAs.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUPL = 8;  // 16-byte units per lane in flight (4 KB per warp)

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
      if (c < upr) {
        const uint4 xa = __ldg(reinterpret_cast<const uint4*>(x + 16 * c));
        const uint4 xb = __ldg(reinterpret_cast<const uint4*>(x + 16 * c + 8));
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const uint32_t wd[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
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
    }
  }
  const float s = moe::warp_sum(acc.x + acc.y);
  if (lane == 0) y[m] = rs[m] * s;
}

}  // namespace

extern "C" int fp8_rowscale_gemv(const uint8_t* w_e4m3, const float* row_scale,
                                 const uint16_t* x_bf16, int M, int K, float* y, void* stream) {
  if (!w_e4m3 || !row_scale || !x_bf16 || !y || M < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 32768) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(w_e4m3) || !moe::aligned16(x_bf16)) return MOE_ERR_ALIGNMENT;
  if (M == 0) return MOE_OK;
  const int grid = (M + kThreads / 32 - 1) / (kThreads / 32);
  fp8_gemv_kernel<<<grid, kThreads, 0, (cudaStream_t)stream>>>(w_e4m3, row_scale, x_bf16, M, K, y);
  return moe::launch_status();
}
