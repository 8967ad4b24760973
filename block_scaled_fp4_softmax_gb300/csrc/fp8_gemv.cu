// FP8 (E4M3) row-scaled matrix-vector product.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "Why this model": the large dense matrices are
// stored in FP8 with one scale per row; section "The engine", item 4: an FP8
// row-scaled matrix-vector kernel replaced a generic unpack path.
// One warp per row; lane j reads the 16-byte units j, j+32, ... (512
// contiguous bytes per warp-wide load); E4M3 pairs go through the hardware
// convert to f16x2 and are accumulated in FP32 against x from shared memory.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) fp8_gemv_kernel(const uint8_t* __restrict__ w,
                                                           const float* __restrict__ rs,
                                                           const uint16_t* __restrict__ x,
                                                           int M, int K, float* __restrict__ y) {
  extern __shared__ float2 xs2[];  // [8][K/16]: pair pe of unit c at xs2[pe * (K/16) + c]
  const int upr = K >> 4;
  for (int h0 = threadIdx.x * 8; h0 < K; h0 += kThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + h0));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    const int c = h0 >> 4, pe0 = (h0 & 15) >> 1;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xs2[(pe0 + i) * upr + c] =
          make_float2(moe::bf16_bits_to_f32(wv[i] & 0xFFFFu), moe::bf16_bits_to_f32(wv[i] >> 16));
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kThreads / 32) + warp;
  if (m >= M) return;
  const uint8_t* row = w + (size_t)m * K;
  float2 acc = make_float2(0.f, 0.f);
  for (int base = 0; base < upr; base += 32 * 4) {
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = base + lane + 32 * i;
      if (c < upr) q[i] = moe::ldg_stream(row + 16 * c);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = base + lane + 32 * i;
      if (c < upr) {
        const uint32_t wd[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const float2 wf = moe::e4m3x2_to_f32x2(wd[wi] >> (16 * hi));
            acc = moe::ffma2(wf, xs2[(2 * wi + hi) * upr + c], acc);
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
  const size_t smem = (size_t)K * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fp8_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = (M + 7) / 8;
  fp8_gemv_kernel<<<grid, kThreads, smem, (cudaStream_t)stream>>>(w_e4m3, row_scale, x_bf16, M, K,
                                                                  y);
  return moe::launch_status();
}
