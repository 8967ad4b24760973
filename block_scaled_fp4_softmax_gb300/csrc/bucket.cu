// Bucketing of routed (token, slot) pairs by expert.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "The engine", item 5: the whole prompt goes
// through a layer at once, so each expert is read once per layer; "Running
// the 510 GB DeepSeek-V4.1-Flash on an 8 GB GPU ...", section "Making it
// faster: v1 to v4", v3: each expert's tokens are found by comparing the index
// tensor with the expert.  Here that search is one stable counting sort on
// the device: per-segment histograms, one scan, and a stable scatter, all
// integer work and therefore bit-reproducible.
#include "common.cuh"

namespace {

constexpr int kSeg = 1024;  // pairs per segment

// 1. per-segment histogram: seg_counts[s][e]
__global__ void __launch_bounds__(256) seg_hist_kernel(const int32_t* __restrict__ idx, int P,
                                                       int E, int32_t* __restrict__ seg_counts,
                                                       int32_t* __restrict__ st) {
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += 256) h[e] = 0;
  __syncthreads();
  const int s = blockIdx.x;
  const int end = min(P, (s + 1) * kSeg);
  bool bad = false;
  for (int p = s * kSeg + threadIdx.x; p < end; p += 256) {
    const int e = idx[p];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
    else bad = true;
  }
  if (bad) moe::status_or(st, MOE_DEV_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) seg_counts[(size_t)s * E + e] = h[e];
}

// 2. one CTA: counts[e] = sum_s, offsets = exclusive scan over e,
//    seg_base[s][e] = offsets[e] + sum_{s' < s} seg_counts[s'][e]
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ seg_counts,
                                                    int S, int E, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ seg_base) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int c = 0;
    if (e < E)
      for (int s = 0; s < S; ++s) c += seg_counts[(size_t)s * E + e];
    // block-wide exclusive scan of c
    int v = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += o;
      }
      warp_tot[lane] = w;
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + v - c;
    if (e < E) {
      counts[e] = c;
      offsets[e] = excl;
      int run = excl;
      for (int s = 0; s < S; ++s) {
        seg_base[(size_t)s * E + e] = run;
        run += seg_counts[(size_t)s * E + e];
      }
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + c;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

// 3. stable scatter: one warp walks its segment 32 pairs at a time; pairs of
//    the same expert inside a step are ranked by lane.
__global__ void __launch_bounds__(32) scatter_kernel(const int32_t* __restrict__ idx, int P, int E,
                                                     const int32_t* __restrict__ seg_base,
                                                     int32_t* __restrict__ pairs) {
  extern __shared__ int32_t run[];
  const int s = blockIdx.x, lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) run[e] = seg_base[(size_t)s * E + e];
  __syncwarp();
  const int end = min(P, (s + 1) * kSeg);
  for (int p0 = s * kSeg; p0 < end; p0 += 32) {
    const int p = p0 + lane;
    const int e = p < end ? idx[p] : -1;
    const bool ok = e >= 0 && e < E;
    const unsigned same = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int rank = __popc(same & ((1u << lane) - 1u));
    const int leader = __ffs(same) - 1;
    int pos = 0;
    if (ok) pos = run[e] + rank;
    __syncwarp();
    if (ok && lane == leader) run[e] += __popc(same);
    __syncwarp();
    if (ok) pairs[pos] = p;
  }
}

}  // namespace

extern "C" size_t moe_bucket_workspace(int T, int k, int E) {
  if (T < 0 || k <= 0 || E <= 0) return 0;
  const long long P = (long long)T * k;
  const long long S = (P + kSeg - 1) / kSeg;
  return (size_t)(2 * S * E) * sizeof(int32_t);
}

extern "C" int moe_bucket_by_expert(const int32_t* idx, int T, int k, int E, int32_t* counts,
                                    int32_t* offsets, int32_t* pairs, void* workspace,
                                    size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!idx || !counts || !offsets || !pairs) return MOE_ERR_INVALID_ARG;
  if (T < 0 || k <= 0 || E <= 0 || E > 65536) return MOE_ERR_INVALID_ARG;
  const long long P = (long long)T * k;
  if (P > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  if (P == 0) {
    if (cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), st) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_bucket_workspace(T, k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int S = (int)((P + kSeg - 1) / kSeg);
  int32_t* seg_counts = reinterpret_cast<int32_t*>(workspace);
  int32_t* seg_base = seg_counts + (size_t)S * E;
  const size_t hsmem = (size_t)E * sizeof(int32_t);
  static moe::SmemGrant g_hist, g_scatter;
  if (!moe::grant_smem(seg_hist_kernel, hsmem, g_hist) || !moe::grant_smem(scatter_kernel, hsmem, g_scatter))
    return MOE_ERR_CUDA;
  seg_hist_kernel<<<S, 256, hsmem, st>>>(idx, (int)P, E, seg_counts, dev_status);
  scan_kernel<<<1, 1024, 0, st>>>(seg_counts, S, E, counts, offsets, seg_base);
  scatter_kernel<<<S, 32, hsmem, st>>>(idx, (int)P, E, seg_base, pairs);
  return moe::launch_status();
}
