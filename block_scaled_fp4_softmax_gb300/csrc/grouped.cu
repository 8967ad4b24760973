// Prompt path: the routed-MoE layer for many tokens as a grouped contraction
// on the 5th-generation tensor cores.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "The engine", item 5: the whole prompt runs
// through a layer at once, so each expert's weights are read once per layer
// (not once per prompt chunk).  Here the routed (token, slot) pairs are
// bucketed by expert on the device, and each expert's tokens form the N side
// of a BF16 MMA whose M side is 128 weight rows dequantised from the FP4
// record on the fly:
//
//   phase 0  (gate/up):  Dg = Wg[128 x H] . X^T,  Du = Wu[128 x H] . X^T  (TMEM)
//                        h  = BF16(silu(Dg) * Du)  -> workspace, rows sorted by expert
//   phase 1  (down):     D  = Wd[128 x I] . h^T                            (TMEM)
//                        y[t] += w * D  (FP32 atomic add)
//
// One persistent CTA per SM walks a static list of tiles (expert, token tile,
// weight-row tile).  Warp roles:
//   warp 0          TMEM allocation; lane 0 issues tcgen05.mma and commits
//   warps 1-2       gather B rows (tokens' x or h) with cp.async into
//                   128-byte-swizzled shared memory; each thread owns two rows
//                   and resolves their source addresses once per tile
//   warps 3-10      load FP4 codes + block scales, convert e2m1 x scale to BF16
//                   (exact) and store the A tile, 128-byte swizzled
//   warps 11-14     epilogue: tcgen05.ld from TMEM, SwiGLU or weighted combine
// Every mbarrier wait is bounded by the global timer; a wait that runs out sets
// MOE_DEV_TIMEOUT and the CTA drains and exits.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace {

using namespace moe::tc;

constexpr int BM = 128;      // weight rows per tile (MMA M)
constexpr int BK = 64;       // K elements per stage (128 bytes of BF16)
constexpr int BN = 128;      // max tokens per tile (MMA N, padded to 16)
constexpr int kThreads = 480;
constexpr int kLoaderThreads = 64;     // warps 1-2: two B rows each
constexpr int kProducerThreads = 256;  // warps 3-10
constexpr int kEpiThreads = 128;       // warps 11-14
constexpr int kProdWarp0 = 3, kEpiWarp0 = 11;
constexpr int kPrefetch = 4;           // k-steps of FP4 codes a producer holds in registers
constexpr int kLoaderDepth = 2;        // cp.async groups a loader keeps in flight
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct GroupedArgs {
  const uint16_t* x;        // [T, H] BF16 (FP16 copy when use_f16: see below)
  const int32_t* pairs;     // [P] pair ids sorted by expert
  const int32_t* offsets;   // [E+1]
  const int32_t* ntile_off; // [E+1] exclusive scan of ceil(count/BN)
  const float* weights;     // [T*k]
  const void* const* ptrs;  // [E] record pointers
  int E, k, H, I;
  uint16_t* hbuf;           // [P, I] BF16, rows in sorted-pair order
  float* y;                 // [T, H] FP32 (zeroed before phase 1)
  int32_t* st;
};

// Phase 0 of NVFP4 runs as an FP16 x FP16 MMA: e2m1 x E4M3 scale is exact in
// FP16 and takes one convert plus one packed multiply per pair; x is
// converted once to FP16 (exact for BF16 values of magnitude in [2^-14,
// 65504]; smaller ones round to FP16 subnormals, at most 2^-25 away).
// MXFP4 scales (2^-127..2^127) do not fit FP16, so MXFP4 stays BF16.
template <int FMT, int PHASE>
struct OperandF16 {
  static constexpr bool value = FMT == MOE_FMT_NVFP4 && PHASE == 0;
};

template <int PHASE>
struct Cfg {
  static constexpr int NA = PHASE == 0 ? 2 : 1;           // A matrices per tile
  static constexpr int STAGES = PHASE == 0 ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2;             // 16 KB
  static constexpr int B_BYTES = BN * BK * 2;             // 16 KB
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = NA * BN;               // 256 or 128
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*bars*/ +
                                 2 * BN * 8 /*per-column token and weight, two tiles*/;
};

struct TileInfo {
  int e, row0, count, mt;  // expert, first sorted-pair row, tokens, weight-row tile
};

// tile id -> (expert, token tile, weight-row tile); experts found by binary
// search over the exclusive scan of their token-tile counts.
__device__ __forceinline__ TileInfo tile_info(const GroupedArgs& a, int tile, int MT) {
  TileInfo ti;
  const int g = tile / MT;
  ti.mt = tile - g * MT;
  int lo = 0, hi = a.E;  // find e with ntile_off[e] <= g < ntile_off[e+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.ntile_off + mid) <= g) lo = mid;
    else hi = mid;
  }
  ti.e = lo;
  const int nt = g - __ldg(a.ntile_off + lo);
  const int beg = __ldg(a.offsets + lo);
  const int cnt = __ldg(a.offsets + lo + 1) - beg;
  ti.row0 = beg + nt * BN;
  ti.count = min(BN, cnt - nt * BN);
  return ti;
}

__device__ __forceinline__ const uint8_t* tile_record(const GroupedArgs& a, int e) {
  const uint8_t* r = reinterpret_cast<const uint8_t*>(a.ptrs[e]);
  if (r == nullptr || (reinterpret_cast<uintptr_t>(r) & 15u) != 0) return nullptr;
  return r;
}

// 32 e2m1 codes (16 bytes) x one or two block scales -> 32 BF16 (exact), as
// four 16-byte chunks.
template <int FMT>
__device__ __forceinline__ void dequant_unit(uint4 q, uint32_t sbits, bool poison, uint4 (&out)[4]) {
  float s0, s1;
  if (FMT == MOE_FMT_NVFP4) {
    const float2 s = moe::e4m3x2_to_f32x2(sbits);
    s0 = s.x;
    s1 = s.y;
  } else {
    s0 = s1 = moe::ue8m0_to_f32(sbits);
  }
  if (poison) s0 = s1 = __uint_as_float(0x7FC00000u);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const float s = wi < 2 ? s0 : s1;
    uint32_t o[4];
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const uint32_t h2 = moe::e2m1x2_to_f16x2((w[wi] >> (8 * bi)) & 0xFFu);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      uint32_t b;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(f.y * s), "f"(f.x * s));
      o[bi] = b;
    }
    out[wi] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Asks the L2 to fetch [src, src + bytes) ahead of use (no data returned).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One tile's weight rows are one contiguous block per matrix (codes and
// scales); prefetch them into L2 so the per-k-step loads hit in L2.
template <int FMT, int PHASE>
__device__ __forceinline__ void prefetch_tile(const GroupedArgs& a, int tile, int MT, int total_tiles) {
  if (tile >= total_tiles) return;
  const TileInfo ti = tile_info(a, tile, MT);
  const uint8_t* rec = tile_record(a, ti.e);
  if (rec == nullptr) return;
  const moe::RecordOffsets ro = moe::record_offsets(a.H, a.I, FMT);
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  const int K = PHASE == 0 ? a.H : a.I;
  const size_t row0 = (size_t)ti.mt * BM;
  const uint32_t cbytes = (uint32_t)(BM * (K / 2)), sbytes = (uint32_t)(BM * (K / G));
  if (PHASE == 0) {
    prefetch_l2(rec + ro.gate + row0 * (K / 2), cbytes);
    prefetch_l2(rec + ro.up + row0 * (K / 2), cbytes);
    prefetch_l2(rec + ro.gate_s + row0 * (K / G), sbytes);
    prefetch_l2(rec + ro.up_s + row0 * (K / G), sbytes);
  } else {
    prefetch_l2(rec + ro.down + row0 * (K / 2), cbytes);
    prefetch_l2(rec + ro.down_s + row0 * (K / G), sbytes);
  }
}

// NVFP4 unit -> 32 FP16 (exact): hardware e2m1x2 -> f16x2, times the block's
// E4M3 scale (as f16x2) in one packed multiply.
__device__ __forceinline__ void dequant_unit_f16(uint4 q, uint32_t sbits, bool poison, uint4 (&out)[4]) {
  uint32_t s2;
  const uint16_t in = (uint16_t)(sbits & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(in));
  uint32_t sc0 = (s2 & 0xFFFFu) * 0x10001u, sc1 = (s2 >> 16) * 0x10001u;  // broadcast halves
  if (poison) sc0 = sc1 = 0x7E007E00u;                                    // f16x2 NaN
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const uint32_t sc = wi < 2 ? sc0 : sc1;
    uint32_t o[4];
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const uint32_t h2 = moe::e2m1x2_to_f16x2((w[wi] >> (8 * bi)) & 0xFFu);
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[bi]) : "r"(h2), "r"(sc));
    }
    out[wi] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int FMT, int PHASE>
__global__ void __launch_bounds__(kThreads, 1) grouped_kernel(GroupedArgs a) {
  constexpr bool kF16 = OperandF16<FMT, PHASE>::value;
  using C = Cfg<PHASE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* tab_ready = drain + 1;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tab_ready + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* col_tok = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE_BYTES + 256);  // [2][BN]
  float* col_w = reinterpret_cast<float*>(col_tok + 2 * BN);                        // [2][BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = PHASE == 0 ? a.H : a.I;  // contraction length
  const int KSTEPS = K / BK;
  const int MT = (PHASE == 0 ? a.I : a.H) / BM;
  const int total_tiles = __ldg(a.ntile_off + a.E) * MT;
  const moe::RecordOffsets ro = moe::record_offsets(a.H, a.I, FMT);
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], kLoaderThreads + kProducerThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiThreads);
    mbar_init(drain, 1);
    mbar_init(&tab_ready[0], kEpiThreads);
    mbar_init(&tab_ready[1], kEpiThreads);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int my_tiles = blockIdx.x < total_tiles ? (total_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int my_steps = my_tiles * KSTEPS;
  auto fail = [&]() {
    moe::status_or(a.st, MOE_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int lt = 0; lt < my_tiles && ok; ++lt) {
        const TileInfo ti = tile_info(a, blockIdx.x + lt * gridDim.x, MT);
        const int n_mma = max(16, (ti.count + 15) & ~15);
        const uint32_t idesc = kF16 ? idesc_f16_f32(BM, n_mma) : idesc_bf16_f32(BM, n_mma);
        if (*abort_flag || !mbar_wait(acc_empty, (lt & 1) ^ 1, globaltimer() + kWaitNs)) {
          fail();
          ok = false;
          break;
        }
        fence_after_sync();
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const int gs = lt * KSTEPS + ks;
          const int stage = gs % C::STAGES;
          if (*abort_flag || !mbar_wait(&full[stage], (gs / C::STAGES) & 1, globaltimer() + kWaitNs)) {
            fail();
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t sbase = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = sbase + C::NA * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bdesc = sw128_kmajor_desc(b_addr + kk * 32);
#pragma unroll
            for (int m = 0; m < C::NA; ++m) {
              const uint64_t adesc = sw128_kmajor_desc(sbase + m * C::A_BYTES + kk * 32);
              mma_bf16(tmem + m * BN, adesc, bdesc, idesc, (ks | kk) != 0);
            }
          }
          mma_commit(&empty[stage]);
        }
        if (ok) mma_commit(acc_full);
      }
      // wait for every MMA issued above before the CTA may release TMEM
      mma_commit(drain);
      mbar_wait(drain, 0, globaltimer() + kWaitNs);
    }
    __syncwarp();
  } else if (warp < kProdWarp0) {
    // ------------------------------------------------------------- B loaders
    const int lid = threadIdx.x - 32;  // 0..63; rows lid and lid + 64
    int pending = 0;                    // steps issued but not yet signalled
    int cur_tile = -1;
    const uint16_t* src_row[2] = {a.x, a.x};
    uint32_t src_bytes[2] = {0, 0};
    for (int gs = 0; gs < my_steps; ++gs) {
      const int lt = gs / KSTEPS, ks = gs - lt * KSTEPS;
      const int stage = gs % C::STAGES;
      if (lt != cur_tile) {
        cur_tile = lt;
        const TileInfo ti = tile_info(a, blockIdx.x + lt * gridDim.x, MT);
        const int n_rows = max(16, (ti.count + 15) & ~15);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = lid + 64 * h;
          src_bytes[h] = n < ti.count ? 16u : 0u;
          src_row[h] = a.x;
          if (n < ti.count) {
            if (PHASE == 0) {
              const int p = __ldg(a.pairs + ti.row0 + n);
              src_row[h] = a.x + (size_t)(p / a.k) * a.H;
            } else {
              src_row[h] = a.hbuf + (size_t)(ti.row0 + n) * a.I;
            }
          }
          if (n >= n_rows) src_bytes[h] = 0xFFFFFFFFu;  // row not part of this tile's MMA
        }
      }
      if (*abort_flag || !mbar_wait(&empty[stage], ((gs / C::STAGES) & 1) ^ 1, globaltimer() + kWaitNs)) {
        fail();
        break;
      }
      const uint32_t b_addr = smem_u32(smem + stage * C::STAGE_BYTES + C::NA * C::A_BYTES);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (src_bytes[h] == 0xFFFFFFFFu) continue;
        const int n = lid + 64 * h;
        const uint16_t* src = src_row[h] + (src_bytes[h] ? ks * BK : 0);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          cp_async16(b_addr + n * 128 + ((ch ^ (n & 7)) << 4), src + (src_bytes[h] ? ch * 8 : 0),
                     src_bytes[h]);
      }
      cp_async_commit();
      ++pending;
      if (pending > kLoaderDepth) {
        cp_async_wait<kLoaderDepth>();
        fence_proxy_async();
        mbar_arrive(&full[(gs - kLoaderDepth) % C::STAGES]);
        --pending;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    if (!*abort_flag) {
      for (int gs = my_steps - pending; gs < my_steps; ++gs) mbar_arrive(&full[gs % C::STAGES]);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------ A dequant producers
    const int pid = threadIdx.x - kProdWarp0 * 32;  // 0..255
    const int r = pid >> 1, half = pid & 1;
    uint4 q[kPrefetch][C::NA];
    uint32_t sb[kPrefetch][C::NA];
    const uint8_t* rec_of[kPrefetch];
    // issue the loads of step gs into slot gs % kPrefetch
    int cached_lt = -1;
    const uint8_t* cached_rec = nullptr;
    size_t cached_row = 0;
    auto issue_slot = [&](int gs, const int slot) {
      const int lt = gs / KSTEPS, ks = gs - lt * KSTEPS;
      if (lt != cached_lt) {
        cached_lt = lt;
        const TileInfo ti = tile_info(a, blockIdx.x + lt * gridDim.x, MT);
        cached_rec = tile_record(a, ti.e);
        cached_row = (size_t)ti.mt * BM + r;
        if (pid == 0) {  // this tile (first time) and the next one into L2
          if (lt == 0) prefetch_tile<FMT, PHASE>(a, blockIdx.x, MT, total_tiles);
          prefetch_tile<FMT, PHASE>(a, blockIdx.x + (lt + 1) * gridDim.x, MT, total_tiles);
        }
      }
      const uint8_t* rec = cached_rec;
      rec_of[slot] = rec;
      if (rec == nullptr) return;
      const size_t row = cached_row;
#pragma unroll
      for (int m = 0; m < C::NA; ++m) {
        size_t coff, soff;
        if (PHASE == 0) {
          coff = m == 0 ? ro.gate : ro.up;
          soff = m == 0 ? ro.gate_s : ro.up_s;
        } else {
          coff = ro.down;
          soff = ro.down_s;
        }
        const uint8_t* cp = rec + coff + row * (K / 2) + ks * (BK / 2) + half * 16;
        const uint8_t* sp = rec + soff + row * (K / G) + (ks * BK + half * 32) / G;
        q[slot][m] = moe::ldg_stream_l2pf(cp);
        sb[slot][m] = FMT == MOE_FMT_NVFP4 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(sp))
                                           : (uint32_t)__ldg(sp);
      }
    };
#pragma unroll
    for (int slot = 0; slot < kPrefetch; ++slot)
      if (slot < my_steps) issue_slot(slot, slot);
    bool alive = true;
    // unrolled by the prefetch depth so every register slot index is static
    for (int gs0 = 0; gs0 < my_steps && alive; gs0 += kPrefetch) {
#pragma unroll
      for (int slot = 0; slot < kPrefetch; ++slot) {
        const int gs = gs0 + slot;
        if (gs >= my_steps || !alive) break;
        const int stage = gs % C::STAGES;
        if ((gs % KSTEPS) == 0 && pid == 0) {
          const TileInfo ti = tile_info(a, blockIdx.x + (gs / KSTEPS) * gridDim.x, MT);
          if (tile_record(a, ti.e) == nullptr)
            moe::status_or(a.st, a.ptrs[ti.e] == nullptr ? MOE_DEV_NULL_EXPERT : MOE_DEV_MISALIGNED);
        }
        if (*abort_flag || !mbar_wait(&empty[stage], ((gs / C::STAGES) & 1) ^ 1, globaltimer() + kWaitNs)) {
          fail();
          alive = false;
          break;
        }
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        const bool poison = rec_of[slot] == nullptr;
#pragma unroll
        for (int m = 0; m < C::NA; ++m) {
          uint4 out[4];
          if constexpr (kF16)
            dequant_unit_f16(poison ? make_uint4(0, 0, 0, 0) : q[slot][m], poison ? 0u : sb[slot][m],
                             poison, out);
          else
            dequant_unit<FMT>(poison ? make_uint4(0, 0, 0, 0) : q[slot][m], poison ? 0u : sb[slot][m],
                              poison, out);
          uint8_t* row_base = sa + m * C::A_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = half * 4 + c;
            *reinterpret_cast<uint4*>(row_base + ((ch ^ (r & 7)) << 4)) = out[c];
          }
        }
        fence_proxy_async();
        mbar_arrive(&full[stage]);
        if (gs + kPrefetch < my_steps) issue_slot(gs + kPrefetch, slot);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    // A warp may only touch TMEM lanes 32*(warp % 4) .. +31.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;           // accumulator row = weight row in tile
    const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    for (int lt = 0; lt < my_tiles; ++lt) {
      const TileInfo ti = tile_info(a, blockIdx.x + lt * gridDim.x, MT);
      // per-column token and router weight, once per tile, double buffered: a
      // thread can be at most one tile ahead of the slowest (acc_empty counts
      // every epilogue thread), so tile lt never overwrites a table in use.
      int* tok = col_tok + (lt & 1) * BN;
      float* wcol = col_w + (lt & 1) * BN;
      if (PHASE == 1) {
        if (et < ti.count) {
          const int p = __ldg(a.pairs + ti.row0 + et);
          tok[et] = p / a.k;
          wcol[et] = __ldg(a.weights + p);
        }
        mbar_arrive(&tab_ready[lt & 1]);
        if (!mbar_wait(&tab_ready[lt & 1], (lt >> 1) & 1, globaltimer() + kWaitNs)) {
          fail();
          break;
        }
      }
      if (*abort_flag || !mbar_wait_backoff(acc_full, lt & 1, globaltimer() + kWaitNs)) {
        fail();
        break;
      }
      fence_after_sync();
      const int col = ti.mt * BM + row;
      for (int c0 = 0; c0 < ti.count; c0 += 16) {
        uint32_t v0[16];
        tmem_ld16(lane_addr + c0, v0);
        if (PHASE == 0) {
          uint32_t v1[16];
          tmem_ld16(lane_addr + BN + c0, v1);
          tmem_ld_wait();
          uint16_t* hrow = a.hbuf + (size_t)(ti.row0 + c0) * a.I + col;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.count) {
              const float g = __uint_as_float(v0[j]);
              const float u = __uint_as_float(v1[j]);
              const float h = g / (1.0f + expf(-g)) * u;
              const __nv_bfloat16 hb = __float2bfloat16_rn(h);
              hrow[(size_t)j * a.I] = *reinterpret_cast<const uint16_t*>(&hb);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.count)
              atomicAdd(a.y + (size_t)tok[c0 + j] * a.H + col, wcol[c0 + j] * __uint_as_float(v0[j]));
          }
        }
      }
      fence_before_sync();
      mbar_arrive(acc_empty);
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// exclusive scan of ceil(count[e] / BN) -> ntile_off[E+1]; one CTA
__global__ void __launch_bounds__(1024) tile_scan_kernel(const int32_t* __restrict__ counts, int E,
                                                         int32_t* __restrict__ ntile_off) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    const int c = e < E ? (counts[e] + BN - 1) / BN : 0;
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
    if (e < E) ntile_off[e] = excl;
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + c;
    __syncthreads();
  }
  if (threadIdx.x == 0) ntile_off[E] = carry;
}

// x (BF16) -> FP16 for the NVFP4 gate/up MMA.  A magnitude at or above 65520
// has no FP16 value: MOE_DEV_FP16_RANGE is set (the product rows become inf).
__global__ void x_to_f16_kernel(const uint16_t* __restrict__ x, long long n, uint16_t* __restrict__ x16,
                                int32_t* __restrict__ st) {
  bool bad = false;
  for (long long i = (blockIdx.x * (long long)blockDim.x + threadIdx.x) * 8; i < n;
       i += (long long)gridDim.x * blockDim.x * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + i));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = moe::bf16_bits_to_f32(wv[j] & 0xFFFFu), hi = moe::bf16_bits_to_f32(wv[j] >> 16);
      bad |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
      const __half2 h = __floats2half2_rn(lo, hi);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(x16 + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) moe::status_or(st, MOE_DEV_FP16_RANGE);
}

// A pair whose expert index is outside [0, E) was dropped by the bucketing;
// its token's output row is set to NaN so the error cannot pass silently.
__global__ void poison_bad_pairs_kernel(const int32_t* __restrict__ idx, int P, int k, int E, int H,
                                        float* __restrict__ y) {
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
    const int e = idx[p];
    if (e < 0 || e >= E) {
      float* row = y + (size_t)(p / k) * H;
      for (int i = 0; i < H; ++i) row[i] = __uint_as_float(0x7FC00000u);
    }
  }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct WsLayout {
  size_t counts, offsets, ntile, pairs, hbuf, x16, bucket, total;
};

WsLayout ws_layout(int T, int k, int E, const moe_expert_shape& s) {
  WsLayout w;
  const size_t P = (size_t)T * k;
  size_t o = 0;
  w.counts = o;  o = align256(o + (size_t)E * 4);
  w.offsets = o; o = align256(o + (size_t)(E + 1) * 4);
  w.ntile = o;   o = align256(o + (size_t)(E + 1) * 4);
  w.pairs = o;   o = align256(o + P * 4);
  w.hbuf = o;    o = align256(o + P * (size_t)s.inter * 2);
  w.x16 = o;     o = align256(o + (s.format == MOE_FMT_NVFP4 ? (size_t)T * s.hidden * 2 : 0));
  w.bucket = o;  o = align256(o + moe_bucket_workspace(T, k, E));
  w.total = o;
  return w;
}

template <int FMT, int PHASE>
int launch_phase(const GroupedArgs& a, cudaStream_t st) {
  using C = Cfg<PHASE>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(grouped_kernel<FMT, PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr = true;
  }
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) return MOE_ERR_CUDA;
  }
  grouped_kernel<FMT, PHASE><<<sms, kThreads, C::SMEM, st>>>(a);
  return moe::launch_status();
}

}  // namespace

extern "C" size_t moe_experts_grouped_workspace(int T, int k, int E, moe_expert_shape s) {
  if (T < 0 || k <= 0 || E <= 0 || !moe::shape_ok(s)) return 0;
  return ws_layout(T, k, E, s).total;
}

extern "C" int moe_experts_grouped(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                                   int T, int k, const void* const* expert_ptrs, int E,
                                   moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                                   int32_t* dev_status, void* stream) {
  if (!x_bf16 || !idx || !weights || !expert_ptrs || !y) return MOE_ERR_INVALID_ARG;
  if (T < 0 || k <= 0 || k > 32 || E <= 0 || E > 65536) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s) || s.hidden % BM != 0 || s.inter % BM != 0) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > (1LL << 28)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, k, E, s);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(x_bf16) || !moe::aligned16(workspace) || !moe::aligned16(y))
    return MOE_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* ntile = reinterpret_cast<int32_t*>(ws + L.ntile);
  int32_t* pairs = reinterpret_cast<int32_t*>(ws + L.pairs);
  int rc = moe_bucket_by_expert(idx, T, k, E, counts, offsets, pairs, ws + L.bucket,
                                L.total - L.bucket, dev_status, stream);
  if (rc != MOE_OK) return rc;
  tile_scan_kernel<<<1, 1024, 0, st>>>(counts, E, ntile);
  if (cudaMemsetAsync(y, 0, (size_t)T * s.hidden * sizeof(float), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  GroupedArgs a;
  a.x = x_bf16;
  a.pairs = pairs;
  a.offsets = offsets;
  a.ntile_off = ntile;
  a.weights = weights;
  a.ptrs = expert_ptrs;
  a.E = E;
  a.k = k;
  a.H = s.hidden;
  a.I = s.inter;
  a.hbuf = reinterpret_cast<uint16_t*>(ws + L.hbuf);
  a.y = y;
  a.st = dev_status;
  if (s.format == MOE_FMT_NVFP4) {
    uint16_t* x16 = reinterpret_cast<uint16_t*>(ws + L.x16);
    const long long n = (long long)T * s.hidden;
    x_to_f16_kernel<<<(unsigned)std::min<long long>((n / 8 + 255) / 256, 1184), 256, 0, st>>>(
        x_bf16, n, x16, dev_status);
    GroupedArgs a0 = a;
    a0.x = x16;
    rc = launch_phase<MOE_FMT_NVFP4, 0>(a0, st);
    if (rc == MOE_OK) rc = launch_phase<MOE_FMT_NVFP4, 1>(a, st);
  } else {
    rc = launch_phase<MOE_FMT_MXFP4, 0>(a, st);
    if (rc == MOE_OK) rc = launch_phase<MOE_FMT_MXFP4, 1>(a, st);
  }
  if (rc != MOE_OK) return rc;
  const int P = T * k;
  poison_bad_pairs_kernel<<<(P + 255) / 256, 256, 0, st>>>(idx, P, k, E, s.hidden, y);
  return moe::launch_status();
}
