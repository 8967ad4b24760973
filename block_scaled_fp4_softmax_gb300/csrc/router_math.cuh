// Router arithmetic shared by the router kernels and the fused decode layer:
// the fixed summation orders that make logits, the top-k choice and the RMS
// chaining reproducible bit for bit ("Running a 133 GB MoE model on an 8 GB
// GPU at 11 tokens/s by streaming experts from NVMe", section "Why this
// model": top-10 of 512 experts per layer, weights renormalised over the
// chosen ones).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace rt {

// Barrier among the threads that run a router step: the whole block
// (BAR < 0), or named barrier BAR over the first N threads.
template <int BAR, int N>
__device__ __forceinline__ void step_sync() {
  if constexpr (BAR < 0) __syncthreads();
  else asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(N) : "memory");
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// RMS chaining in FP32, one fixed order: thread t of 256 sums y[t + 256 m]^2
// for m ascending (square rounded, then added), a pairwise tree combines the
// 256 partial sums, mean = sum / H, r = 1 / sqrt(mean + eps) with IEEE sqrt
// and divide.  Every thread of the block (BAR < 0), or the first N >= 256
// threads (named barrier BAR), calls it; threads from 256 on only take part
// in the barriers.  part: 256 floats of shared memory.  L2_ONLY: y is read
// through L2 only (a persistent kernel reads a new y at the same address
// every layer; L1 is not coherent across SMs).
template <int BAR = -1, int N = 0, bool L2_ONLY = false>
__device__ __forceinline__ float rms_inv_fixed_order(const float* __restrict__ yr, int H, float eps,
                                                     float* part) {
  if (threadIdx.x < 256) {
    float acc = 0.0f;
    constexpr int kBatch = 16;  // loads in flight (all of them up to H = 4096); the adds keep the order above
    for (int i0 = threadIdx.x; i0 < H; i0 += 256 * kBatch) {
      float v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        v[b] = i0 + 256 * b >= H ? 0.0f : L2_ONLY ? __ldcg(yr + i0 + 256 * b) : yr[i0 + 256 * b];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (i0 + 256 * b < H) acc = __fadd_rn(acc, __fmul_rn(v[b], v[b]));
    }
    part[threadIdx.x] = acc;
  }
  step_sync<BAR, N>();
  for (int w = 128; w >= 32; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] = __fadd_rn(part[threadIdx.x], part[threadIdx.x + w]);
    step_sync<BAR, N>();
  }
  if (threadIdx.x < 32) {  // the levels w = 16 .. 1 inside warp 0: lane t adds lane t + w
    float v = part[threadIdx.x];
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, w));
    if (threadIdx.x == 0) part[0] = v;
  }
  step_sync<BAR, N>();
  const float mean = __fdiv_rn(part[0], (float)H);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
  step_sync<BAR, N>();  // part[] may be reused by the caller
  return r;
}

// One logit without bias, by one warp: lane j walks the chunks of 8 elements
// c = j, j+32, j+64, ... (ascending), elements inside a chunk in order, one
// FMA each (the BF16 x BF16 product is exact, so the FMA is the FP32 add of
// the exact product); the 32 lane sums are combined with an xor butterfly
// d = 16, 8, 4, 2, 1.  x_row may be in shared or global memory; w_row is in
// shared memory (W_SHARED) or read through the read-only path.  Every lane
// returns the logit.
template <bool W_SHARED = false>
__device__ __forceinline__ float logit_dot(const uint16_t* x_row, const uint16_t* __restrict__ w_row, int H,
                                           int lane) {
  const int nchunk = H >> 3;
  float acc = 0.0f;
  constexpr int kBatch = 10;  // chunks of a lane in flight; accumulated in chunk order
  for (int c0 = lane; c0 < nchunk; c0 += 32 * kBatch) {
    uint4 wv[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int c = c0 + 32 * b;
      const uint4* wp = reinterpret_cast<const uint4*>(w_row + 8 * c);
      wv[b] = c < nchunk ? (W_SHARED ? *wp : __ldg(wp)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int c = c0 + 32 * b;
      if (c < nchunk) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x_row + 8 * c);
        const uint32_t ww[4] = {wv[b].x, wv[b].y, wv[b].z, wv[b].w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = fma_bf16(xw[i >> 1] >> (16 * (i & 1)), ww[i >> 1] >> (16 * (i & 1)), acc);
        }
      }
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
  return acc;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Top-k keys: (ordered logit bits << 32 | ~expert), so the maximum is the
// larger logit and, on equal logits, the lower expert index.  NaN ranks below
// -inf, -0 counts as +0.
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

// Renormalised softmax weight of lane r's pick (lanes >= k get 0).
__device__ __forceinline__ float topk_weight(int lane, int k, float my_l) {
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.0f;
  const float sum = warp_sum(ex);
  return lane < k ? __fdiv_rn(ex, sum) : 0.0f;
}

// Top-k of one token's E <= 1024 logits by a whole block of NW <= 32 warps:
// every warp selects the k best of its candidates (expert e = warp * 32 +
// lane + 32 * NW * m) in descending order, then warp 0 merges those NW
// sorted lists -- lane i holds the head of list i, each round takes the
// largest head and the list it came from advances.  The k best of a union
// are the k best of the parts' k best (keys are unique), so the picks and
// their order are exactly those of a single-warp selection.  fin: NW * 32
// keys of shared memory.  Every thread of the block (BAR < 0; the block
// has NW warps), or of the first NW warps (named barrier BAR), calls it;
// warp 0, lane r < k, ends with pick r.  lrow is in global memory, read
// through L2 (written by other CTAs), or in shared memory (SHARED).
template <int NW, int BAR = -1, bool SHARED = false>
__device__ __forceinline__ void topk_block(const float* lrow, int E, int k, unsigned long long* fin, int& my_e,
                                           float& my_l) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kPer = (1024 + 32 * NW - 1) / (32 * NW);  // candidates per lane
  unsigned long long cand[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = warp * 32 + lane + 32 * NW * m;
    cand[m] = 0ull;
    if (e < E)
      cand[m] = ((unsigned long long)ordered_key(SHARED ? lrow[e] : __ldcg(lrow + e)) << 32) |
                (unsigned long long)(~(uint32_t)e);
  }
  if (warp < NW) {
    unsigned long long prev = ~0ull;
    for (int r = 0; r < k; ++r) {  // the warp's r-th best key, kept by lane r
      unsigned long long best = 0ull;
#pragma unroll
      for (int m = 0; m < kPer; ++m)
        if (cand[m] < prev && cand[m] > best) best = cand[m];
      const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
      const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
      best = ((unsigned long long)hi << 32) | lo;
      prev = best;
      if (lane == r) fin[warp * 32 + r] = best;
    }
    if (lane >= k) fin[warp * 32 + lane] = 0ull;
  }
  step_sync<BAR, NW * 32>();
  if (warp == 0) {
    int pos = 0;
    unsigned long long head = lane < NW ? fin[lane * 32] : 0ull;
    my_e = 0;
    my_l = 0.0f;
    for (int r = 0; r < k; ++r) {
      const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(head >> 32));
      const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(head >> 32) == hi ? (uint32_t)head : 0u);
      const unsigned long long best = ((unsigned long long)hi << 32) | lo;
      if (lane == r) {
        my_e = (int)(~lo);
        my_l = key_to_float(hi);
      }
      if (lane < NW && head == best) {  // real keys are nonzero, so one lane matches
        ++pos;
        head = pos < k ? fin[lane * 32 + pos] : 0ull;
      }
    }
  }
  step_sync<BAR, NW * 32>();  // fin[] may be reused by the caller
}

// The same top-k as topk_block, usually in a fraction of its time: every
// warp's largest key goes to shared memory, and tau = the k-th largest of
// those NW maxima bounds the answer from below -- at least k keys (the k
// largest maxima) are >= tau, so the k-th largest key of all is >= tau and
// every pick is a key >= tau.  Those survivors (typically a few more than k
// for continuous logits) are gathered in shared memory and warp 0 ranks them
// exactly; when more than 32 survive (few warps hold all the large keys) or
// NW < k, it falls back to topk_block.  Keys are unique, so both routes give
// the same picks in the same order.  fin: NW * 32 keys of shared memory
// (at least 128); same calling rules as topk_block.
template <int NW, int BAR = -1, bool SHARED = false>
__device__ __forceinline__ void topk_block_fast(const float* lrow, int E, int k, unsigned long long* fin,
                                                int& my_e, float& my_l) {
  static_assert(NW * 32 >= 128, "scratch");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (NW < k) {
    topk_block<NW, BAR, SHARED>(lrow, E, k, fin, my_e, my_l);
    return;
  }
  constexpr int kPer = (1024 + 32 * NW - 1) / (32 * NW);
  unsigned long long cand[kPer];
  unsigned long long best = 0ull;
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = warp * 32 + lane + 32 * NW * m;
    cand[m] = 0ull;
    if (e < E)
      cand[m] = ((unsigned long long)ordered_key(SHARED ? lrow[e] : __ldcg(lrow + e)) << 32) |
                (unsigned long long)(~(uint32_t)e);
    best = cand[m] > best ? cand[m] : best;
  }
  unsigned* cnt = reinterpret_cast<unsigned*>(fin + 96);
  if (warp < NW) {
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
    if (lane == 0) fin[warp] = ((unsigned long long)hi << 32) | lo;
    if (warp == 0 && lane == 0) *cnt = 0u;
  }
  step_sync<BAR, NW * 32>();
  // tau: lane i < NW ranks warp maximum i among the NW maxima
  unsigned long long tau = 0ull;
  {
    const unsigned long long mine = lane < NW ? fin[lane] : 0ull;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < NW; ++j) rank += fin[j] > mine;
    const unsigned sel = __ballot_sync(0xffffffffu, lane < NW && rank == k - 1);
    const int src = sel ? __ffs(sel) - 1 : 0;
    tau = __shfl_sync(0xffffffffu, mine, src);
    if (!sel) tau = 0ull;  // maxima tied at zero (fewer than k warps hold keys): no filter
  }
  // survivors: real keys >= tau, gathered at fin[32 .. 64) (unordered)
  if (warp < NW) {
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const bool keep = cand[m] != 0ull && cand[m] >= tau;
      const unsigned b = __ballot_sync(0xffffffffu, keep);
      unsigned base = 0u;
      if (lane == 0 && b) base = atomicAdd(cnt, (unsigned)__popc(b));
      base = __shfl_sync(0xffffffffu, base, 0);
      const unsigned pos = base + __popc(b & ((1u << lane) - 1u));
      if (keep && pos < 32u) fin[32 + pos] = cand[m];
    }
  }
  step_sync<BAR, NW * 32>();
  const unsigned total = *cnt;
  if (total > 32u || tau == 0ull) {
    step_sync<BAR, NW * 32>();  // every thread has read the count before topk_block reuses fin
    topk_block<NW, BAR, SHARED>(lrow, E, k, fin, my_e, my_l);
    return;
  }
  if (warp == 0) {
    const unsigned long long mine = lane < (int)total ? fin[32 + lane] : 0ull;
    int rank = 0;
    for (unsigned j = 0; j < total; ++j) rank += fin[32 + j] > mine;
    if (lane < (int)total && rank < k) fin[64 + rank] = mine;
    __syncwarp();
    my_e = 0;
    my_l = 0.0f;
    if (lane < k) {
      const unsigned long long key = fin[64 + lane];
      my_e = (int)(~(uint32_t)key);
      my_l = key_to_float((uint32_t)(key >> 32));
    }
  }
  step_sync<BAR, NW * 32>();  // fin[] may be reused by the caller
}

}  // namespace rt
}  // namespace moe
