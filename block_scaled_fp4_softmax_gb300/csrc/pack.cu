// fp4_pack_expert: FP32 expert matrices -> one block-scaled FP4 record.
//
// The record is the one-block-per-expert layout of "Running a 133 GB MoE model
// on an 8 GB GPU at 11 tokens/s by streaming experts from NVMe", section "The
// engine", item 1 (gate | up | down | gate_scale | up_scale | down_scale).
// The pages repack vendor files and never quantise, so the quantiser follows
// the rule stated in moe.h: amax/6 rounded to the scale format, then each
// element rounded to the nearest e2m1 value (ties to even, saturating).
#include "common.cuh"

namespace {

__device__ __forceinline__ uint32_t f32_to_e4m3_rn_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;  // second source lands in the low byte
}

// Two floats -> one byte of e2m1 codes: `lo` to the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

template <int G>
__device__ __forceinline__ void quantize_block(const float* __restrict__ src, uint8_t* codes,
                                               uint8_t* scale, int fmt) {
  float v[G];
#pragma unroll
  for (int i = 0; i < G; i += 4) {
    float4 f = *reinterpret_cast<const float4*>(src + i);
    v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < G; ++i) amax = fmaxf(amax, fabsf(v[i]));

  uint32_t s_code;
  float q[G];
  if (fmt == MOE_FMT_NVFP4) {
    s_code = f32_to_e4m3_rn_sat(__fdiv_rn(amax, 6.0f));
    float s = moe::e4m3x2_to_f32x2(s_code).x;
    if (s == 0.0f) {
#pragma unroll
      for (int i = 0; i < G; ++i) q[i] = 0.0f;
    } else {
#pragma unroll
      for (int i = 0; i < G; ++i) q[i] = __fdiv_rn(v[i], s);
    }
  } else {
    int s;
    if (amax == 0.0f) {
      s = 0;
    } else {
      int E = ilogbf(amax) - 3;  // 6 * 2^E < amax here
      while (ldexpf(6.0f, E) < amax) ++E;
      s = min(max(E + 127, 0), 254);
    }
    s_code = (uint32_t)s;
    const int pe = 127 - s;  // multiplier 2^(127 - s), exact
    const float mult = pe >= -126 ? __uint_as_float((uint32_t)(pe + 127) << 23)
                                  : __uint_as_float(0x00400000u);
#pragma unroll
    for (int i = 0; i < G; ++i) q[i] = __fmul_rn(v[i], mult);
  }

  uint32_t words[G / 8];
#pragma unroll
  for (int w = 0; w < G / 8; ++w) {
    uint32_t acc = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) acc |= f32x2_to_e2m1x2(q[8 * w + 2 * b], q[8 * w + 2 * b + 1]) << (8 * b);
    words[w] = acc;
  }
  if constexpr (G == 16) {
    *reinterpret_cast<uint2*>(codes) = make_uint2(words[0], words[1]);
  } else {
    *reinterpret_cast<uint4*>(codes) = make_uint4(words[0], words[1], words[2], words[3]);
  }
  *scale = (uint8_t)s_code;
}

template <int G>
__global__ void pack_kernel(const float* __restrict__ gate, const float* __restrict__ up,
                            const float* __restrict__ down, int H, int I, int fmt,
                            uint8_t* __restrict__ rec) {
  const moe::RecordOffsets o = moe::record_offsets(H, I, fmt);
  const long long per_gu = (long long)I * H / G;  // blocks in gate (and in up)
  const long long total = 3 * per_gu;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < total;
       b += (long long)gridDim.x * blockDim.x) {
    int m = (int)(b / per_gu);
    long long r = b - (long long)m * per_gu;
    const float* src;
    size_t code_off, scale_off;
    if (m == 0) { src = gate; code_off = o.gate; scale_off = o.gate_s; }
    else if (m == 1) { src = up; code_off = o.up; scale_off = o.up_s; }
    else { src = down; code_off = o.down; scale_off = o.down_s; }
    // block r covers elements [r*G, r*G + G) of the row-major matrix
    quantize_block<G>(src + r * G, rec + code_off + r * (G / 2), rec + scale_off + r, fmt);
  }
}

}  // namespace

extern "C" int fp4_pack_expert(const float* gate, const float* up, const float* down,
                               moe_expert_shape s, void* record, void* stream) {
  if (!gate || !up || !down || !record) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(gate) || !moe::aligned16(up) || !moe::aligned16(down) ||
      !moe::aligned16(record))
    return MOE_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  const int G = moe::block_elems(s.format);
  const long long blocks = 3LL * s.inter * s.hidden / G;
  const int threads = 256;
  const int grid = (int)((blocks + threads - 1) / threads);
  if (G == 16)
    pack_kernel<16><<<grid, threads, 0, st>>>(gate, up, down, s.hidden, s.inter, s.format,
                                              (uint8_t*)record);
  else
    pack_kernel<32><<<grid, threads, 0, st>>>(gate, up, down, s.hidden, s.inter, s.format,
                                              (uint8_t*)record);
  return moe::launch_status();
}
