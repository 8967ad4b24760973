// Prompt path: the routed-MoE layer for many tokens as a grouped contraction
// on the 5th-generation tensor cores.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "The engine", item 5: the whole prompt runs
// through a layer at once, so each expert's weights are read once per layer
// (not once per prompt chunk).  Here the routed (token, slot) pairs are
// bucketed by expert on the device, and each expert's tokens form the N side
// of an MMA whose M side is 128 weight rows dequantised from the FP4 record on
// the fly:
//
//   phase 0  (gate/up):  Dg = Wg[128 x H] . X^T,  Du = Wu[128 x H] . X^T  (TMEM)
//                        h  = BF16(silu(Dg) * Du)  -> workspace, rows sorted by expert
//   phase 1  (down):     D  = Wd[128 x I] . h^T                            (TMEM)
//                        y[t] += w * D  (FP32 atomic add)
//
// One persistent CTA per SM walks a static list of tiles (token tile of one
// expert, 128-row weight tile).  Per k-step of 64 elements three rings meet:
//   raw ring  (per producer warp, 8-12 steps deep): the FP4 codes and scales
//             of the warp's rows, fetched with cp.async two k-steps at a time
//             and well ahead of use -- the only operand that comes from HBM,
//             so the deep ring is cheap (FP4 is a quarter of the BF16 bytes).
//             Lanes fetch consecutive 16-byte pieces, so one instruction reads
//             8 rows x 64 contiguous bytes: few L1->L2 requests per byte;
//   A ring    (3-4 stages): the dequantised 128 x 64 weight tile(s), FP16 or
//             BF16, 128-byte swizzled, written by the producers;
//   B ring    (4-6 stages): the 64-element slice of up to 128 token rows (x or
//             h), gathered with cp.async from the L2, 8 lanes per 128-byte row
//             slice.
// The accumulators are double-buffered in TMEM, so the epilogue of one tile
// overlaps the mainloop of the next.  Warp roles:
//   warp 0          TMEM allocation; lane 0 issues tcgen05.mma and commits
//   warps 1-2       B gatherers: each thread owns two token rows of the tile
//   warps 3-10      producers: fetch + dequantise A (e2m1 x scale, exact)
//   warps 11-14     epilogue: tcgen05.ld, SwiGLU or the weighted combine
// Every mbarrier wait is bounded by the global timer; a wait that runs out sets
// MOE_DEV_TIMEOUT, the CTA drains its copies and exits.
#include <algorithm>

#include "common.cuh"
#include "decode_math.cuh"
#include "tcgen05.cuh"

namespace {

using namespace moe::tc;

constexpr int BM = 128;      // weight rows per tile (MMA M)
constexpr int BK = 64;       // K elements per step (128 bytes of FP16/BF16)
constexpr int BN = 128;      // max tokens per tile (MMA N, padded to 16)
constexpr int kThreads = 480;
constexpr int kLoaderThreads = 64;     // warps 1-2: two B rows each
constexpr int kProducerThreads = 256;  // warps 3-10
constexpr int kEpiThreads = 128;       // warps 11-14
constexpr int kProdWarp0 = 3, kEpiWarp0 = 11;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct GroupedArgs {
  const uint16_t* x;        // [T, H]: FP16 (x * 2^e_t) for NVFP4 phase 0, else BF16
  const float* xscale;      // [T] 2^-e_t (NVFP4 phase 0), else NULL
  const int32_t* pairs;     // [P] pair ids sorted by expert
  const int4* tiles;        // [G] token tiles: {expert, first sorted row, rows, 0}
  const int32_t* ntiles;    // [1] G
  const float* weights;     // [T*k]
  const void* const* ptrs;  // [E] record pointers
  int E, k, H, I;
  uint16_t* hbuf;           // [P, I] BF16, rows in sorted-pair order
  float* y;                 // [T, H] FP32 (zeroed before phase 1)
  int32_t* st;
};

// Phase 0 of NVFP4 runs as an FP16 x FP16 MMA: e2m1 x E4M3 scale is exact in
// FP16 and takes one convert plus one packed multiply per pair; x is scaled
// per token by a power of two into FP16's range (exact).  MXFP4 scales
// (2^-127..2^127) do not fit FP16, so MXFP4 stays BF16; phase 1 is BF16
// because its B operand, the SwiGLU intermediate, is BF16.
template <int FMT, int PHASE>
struct OperandF16 {
  static constexpr bool value = FMT == MOE_FMT_NVFP4 && PHASE == 0;
};

template <int PHASE>
struct Cfg {
  static constexpr int NA = PHASE == 0 ? 2 : 1;             // A matrices per tile
  static constexpr int UNITS = NA * BM * BK / 32 / kProducerThreads;  // 16-B code units per producer per step
  static constexpr int A_STAGES = PHASE == 0 ? 3 : 4;
  static constexpr int B_STAGES = PHASE == 0 ? 4 : 6;
  static constexpr int RW = PHASE == 0 ? 32 : 16;           // weight rows per producer warp
  static constexpr int RAW_DEPTH = PHASE == 0 ? 3 : 6;      // super-steps (two k-steps) in flight
  static constexpr int A_BYTES = BM * BK * 2;               // 16 KB per matrix
  static constexpr int B_BYTES = BN * BK * 2;               // 16 KB
  static constexpr int RAW_ROW = 64;                        // code bytes of one row per super-step
  static constexpr int RAW_WARP = RW * (RAW_ROW + 8);       // one super-step of one warp: codes, then 8 scale bytes per row
  static constexpr int RAW_STEP = 8 * RAW_WARP;             // one super-step of all producer warps
  static constexpr int ACC_COLS = NA * BN;                  // one accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS;            // double-buffered: 512 or 256
  static constexpr size_t OFF_A = 0;
  static constexpr size_t OFF_B = OFF_A + (size_t)A_STAGES * NA * A_BYTES;
  static constexpr size_t OFF_RAW = OFF_B + (size_t)B_STAGES * B_BYTES;
  static constexpr size_t OFF_BARS = OFF_RAW + (size_t)RAW_DEPTH * RAW_STEP;
  static constexpr size_t BAR_BYTES = 512;
  static constexpr size_t OFF_COLS = OFF_BARS + BAR_BYTES;  // [2][BN] token, weight, x scale
  static constexpr size_t SMEM = 1024 /*align*/ + OFF_COLS + 2 * BN * 12;
};
static_assert(Cfg<0>::UNITS == 2 && Cfg<1>::UNITS == 1, "producer split");
static_assert(Cfg<0>::RW * 8 == 2 * BM && Cfg<1>::RW * 8 == BM, "rows of the producer warps");
static_assert(Cfg<0>::SMEM <= 232448 && Cfg<1>::SMEM <= 232448, "shared memory");

__device__ __forceinline__ int4 tile_of(const GroupedArgs& a, int tile, int MT, int& mt) {
  const int g = tile / MT;
  mt = tile - g * MT;
  return __ldg(a.tiles + g);
}

__device__ __forceinline__ const uint8_t* tile_record(const GroupedArgs& a, int e) {
  const uint8_t* r = reinterpret_cast<const uint8_t*>(a.ptrs[e]);
  if (r == nullptr || (reinterpret_cast<uintptr_t>(r) & 15u) != 0) return nullptr;
  return r;
}

// cp.async of 16 or 4 bytes (L2 only for 16; the L2 fetches the surrounding
// 256 bytes, so the following k-steps of the same row hit in L2).
__device__ __forceinline__ void cp16_l2pf(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// 32 e2m1 codes (16 bytes) x one or two block scales -> 32 BF16 (exact), as
// four 16-byte chunks.  NVFP4: scale bytes s0 (elements 0-15) and s1 (16-31)
// in the low 16 bits of sbits; MXFP4: one UE8M0 byte.
template <int FMT>
__device__ __forceinline__ void dequant_unit_bf16(uint4 q, uint32_t sbits, bool poison, uint4 (&out)[4]) {
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
    uint32_t h[4], o[4];
    moe::dm::cvt_e2m1x8(w[wi], h);
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const float2 f = __half22float2(moe::dm::as_h2(h[bi]));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[bi]) : "f"(f.y * s), "f"(f.x * s));
    }
    out[wi] = make_uint4(o[0], o[1], o[2], o[3]);
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
    uint32_t h[4], o[4];
    moe::dm::cvt_e2m1x8(w[wi], h);
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[bi]) : "r"(h[bi]), "r"(sc));
    out[wi] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int FMT, int PHASE>
__global__ void __launch_bounds__(kThreads, 1) grouped_kernel(GroupedArgs a) {
  constexpr bool kF16 = OperandF16<FMT, PHASE>::value;
  using C = Cfg<PHASE>;
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sRaw = smem + C::OFF_RAW;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);  // [A_STAGES]
  uint64_t* a_empty = a_full + C::A_STAGES;                             // [A_STAGES]
  uint64_t* b_full = a_empty + C::A_STAGES;                             // [B_STAGES]
  uint64_t* b_empty = b_full + C::B_STAGES;                             // [B_STAGES]
  uint64_t* acc_full = b_empty + C::B_STAGES;                           // [2]
  uint64_t* acc_empty = acc_full + 2;                                   // [2]
  uint64_t* tab_ready = acc_empty + 2;                                  // [2]
  uint64_t* drain = tab_ready + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* col_tok = reinterpret_cast<int*>(smem + C::OFF_COLS);  // [2][BN]
  float* col_w = reinterpret_cast<float*>(col_tok + 2 * BN);  // [2][BN]
  float* col_xs = col_w + 2 * BN;                             // [2][BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = PHASE == 0 ? a.H : a.I;  // contraction length
  const int KSTEPS = K / BK;
  const int MT = (PHASE == 0 ? a.I : a.H) / BM;
  const int total_tiles = __ldg(a.ntiles) * MT;
  const moe::RecordOffsets ro = moe::record_offsets(a.H, a.I, FMT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::A_STAGES; ++s) {
      mbar_init(&a_full[s], kProducerThreads);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < C::B_STAGES; ++s) {
      mbar_init(&b_full[s], kLoaderThreads);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
      mbar_init(&tab_ready[b], kEpiThreads);
    }
    mbar_init(drain, 1);
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
        int mt;
        const int4 ti = tile_of(a, blockIdx.x + lt * gridDim.x, MT, mt);
        const int n_mma = max(16, (ti.z + 15) & ~15);
        const uint32_t idesc = kF16 ? idesc_f16_f32(BM, n_mma) : idesc_bf16_f32(BM, n_mma);
        const int buf = lt & 1;
        if (*abort_flag || !mbar_wait(&acc_empty[buf], ((lt >> 1) & 1) ^ 1, globaltimer() + kWaitNs)) {
          fail();
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * C::ACC_COLS);
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const int gs = lt * KSTEPS + ks;
          const int as = gs % C::A_STAGES, bs = gs % C::B_STAGES;
          if (*abort_flag || !mbar_wait(&a_full[as], (gs / C::A_STAGES) & 1, globaltimer() + kWaitNs) ||
              !mbar_wait(&b_full[bs], (gs / C::B_STAGES) & 1, globaltimer() + kWaitNs)) {
            fail();
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t a_addr = smem_u32(sA + (size_t)as * C::NA * C::A_BYTES);
          const uint32_t b_addr = smem_u32(sB + (size_t)bs * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bdesc = sw128_kmajor_desc(b_addr + kk * 32);
#pragma unroll
            for (int m = 0; m < C::NA; ++m) {
              const uint64_t adesc = sw128_kmajor_desc(a_addr + m * C::A_BYTES + kk * 32);
              mma_bf16(d_tmem + m * BN, adesc, bdesc, idesc, (ks | kk) != 0);
            }
          }
          mma_commit(&a_empty[as]);
          mma_commit(&b_empty[bs]);
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      // wait for every MMA issued above before the CTA may release TMEM
      mma_commit(drain);
      mbar_wait(drain, 0, globaltimer() + kWaitNs);
    }
    __syncwarp();
  } else if (warp < kProdWarp0) {
    // ------------------------------------------------------------- B gatherers
    // Thread lid copies 16-byte chunk c = lid % 8 of rows n = lid / 8 + 8 i
    // (i < 16) of every step's B slice, so the 8 lanes of one row read its 128
    // contiguous bytes and one instruction covers 4 rows.  A stage is signalled
    // full once its copies have landed, which the thread checks for its oldest
    // step in flight before it blocks on a free slot (never after), so the MMA
    // is never kept waiting on a later issue.
    constexpr int kDepth = C::B_STAGES - 1;
    constexpr int kRowsPerThread = BN / 8;
    const int lid = threadIdx.x - 32;
    const int c = lid & 7, rb = lid >> 3;
    int pending = 0;
    int cur_tile = -1;
    const uint16_t* src_row[kRowsPerThread];
    uint32_t row_mode = 0;  // bit i: row i is copied (else skipped); bit 16 + i: zero-filled
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) src_row[i] = a.x;
    bool alive = true;
    for (int gs = 0; gs < my_steps; ++gs) {
      const int lt = gs / KSTEPS, ks = gs - lt * KSTEPS;
      const int bs = gs % C::B_STAGES;
      if (lt != cur_tile) {
        cur_tile = lt;
        int mt;
        const int4 ti = tile_of(a, blockIdx.x + lt * gridDim.x, MT, mt);
        const int n_rows = max(16, (ti.z + 15) & ~15);
        row_mode = 0;
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int n = rb + 8 * i;
          src_row[i] = a.x;
          if (n < ti.z) {
            if (PHASE == 0) {
              const int p = __ldg(a.pairs + ti.y + n);
              src_row[i] = a.x + (size_t)(p / a.k) * a.H;
            } else {
              src_row[i] = a.hbuf + (size_t)(ti.y + n) * a.I;
            }
          }
          if (n < n_rows) row_mode |= 1u << i;              // rows past n_rows are not part of the MMA
          if (n >= ti.z && n < n_rows) row_mode |= 1u << (16 + i);  // padding rows of the MMA: zeros
        }
      }
      if (pending == kDepth) {  // signal the oldest step in flight first
        cp_async_wait<kDepth - 1>();
        fence_proxy_async();
        mbar_arrive(&b_full[(gs - kDepth) % C::B_STAGES]);
        --pending;
      }
      if (*abort_flag || !mbar_wait(&b_empty[bs], ((gs / C::B_STAGES) & 1) ^ 1, globaltimer() + kWaitNs)) {
        fail();
        alive = false;
        break;
      }
      const uint32_t b_addr = smem_u32(sB + (size_t)bs * C::B_BYTES);
      const uint32_t sw = (uint32_t)((c ^ rb) << 4);  // the 128-byte swizzle: n & 7 == rb
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        if (!(row_mode & (1u << i))) continue;
        const int n = rb + 8 * i;
        const bool zero = (row_mode >> (16 + i)) & 1u;
        cp_async16(b_addr + n * 128 + sw, src_row[i] + (zero ? 0 : ks * BK + c * 8), zero ? 0u : 16u);
      }
      cp_async_commit();
      ++pending;
    }
    cp_async_wait<0>();
    fence_proxy_async();
    if (alive && !*abort_flag) {
      for (int gs = my_steps - pending; gs < my_steps; ++gs) mbar_arrive(&b_full[gs % C::B_STAGES]);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------ A producers
    // Phase 0: warp pw owns the 32 rows (pw & 3) * 32 .. +31 of matrix pw >> 2
    // (gate, up), lane = row, 64 elements per step (two 16-byte code units and
    // four E4M3 or two UE8M0 scale bytes); phase 1: warp pw owns rows pw * 16
    // .. +15, lane = (row, half), 32 elements per step.  The warp fetches its
    // rows' codes and scales two k-steps (a super-step) at a time into its own
    // slot of the raw ring, RAW_DEPTH super-steps ahead: lanes take
    // consecutive 16-byte pieces of the rows (64 contiguous bytes per row,
    // piece p of row rr stored at position p ^ ((rr >> 1) & 3), so that the
    // lanes' reads and writes spread over the banks), and each row's 8 (or 4)
    // scale bytes with one copy.  Each lane waits for its own
    // copies (cp.async groups), then the warp synchronises so every lane sees
    // the whole slot.
    const int pw = warp - kProdWarp0;  // 0..7
    const int pid = threadIdx.x - kProdWarp0 * 32;
    const int m = PHASE == 0 ? pw >> 2 : 0;
    const int rbase = PHASE == 0 ? (pw & 3) * 32 : pw * 16;  // first row of the warp in the tile
    const int r_local = PHASE == 0 ? lane : lane >> 1;       // this lane's row in the warp
    const int r = rbase + r_local;
    const int half = PHASE == 0 ? 0 : (lane & 1);
    const int c0 = half * 32;  // first element of the lane inside the step
    const size_t coff = PHASE == 0 ? (m == 0 ? ro.gate : ro.up) : ro.down;
    const size_t soff = PHASE == 0 ? (m == 0 ? ro.gate_s : ro.up_s) : ro.down_s;
    const uint32_t raw_w = smem_u32(sRaw) + (uint32_t)(pw * C::RAW_WARP);
    const uint8_t* raw_wp = sRaw + (size_t)pw * C::RAW_WARP;
    constexpr int kSB = 128 / G;  // scale bytes of one row per super-step (8 or 4)
    const int nss = my_steps / 2;  // super-steps (KSTEPS is even: K % 128 == 0)
    int f_tile = -1;
    const uint8_t* f_rec = nullptr;
    size_t f_row0 = 0;
    auto fetch = [&](int ss) {  // super-step ss -> raw slot ss % RAW_DEPTH, then commit
      if (ss < nss) {
        const int lt = (2 * ss) / KSTEPS, ks = 2 * ss - lt * KSTEPS;
        if (lt != f_tile) {
          f_tile = lt;
          int mt;
          const int4 ti = tile_of(a, blockIdx.x + lt * gridDim.x, MT, mt);
          f_rec = tile_record(a, ti.x);
          f_row0 = (size_t)mt * BM + rbase;
        }
        if (f_rec != nullptr) {
          const uint32_t slot = raw_w + (uint32_t)((ss % C::RAW_DEPTH) * C::RAW_STEP);
#pragma unroll
          for (int i = 0; i < C::RW * 4 / 32; ++i) {
            const int ch = i * 32 + lane, rr = ch >> 2, part = ch & 3;
            cp16_l2pf(slot + rr * C::RAW_ROW + ((part ^ ((rr >> 1) & 3)) << 4),
                      f_rec + coff + (f_row0 + rr) * (size_t)(K / 2) + (size_t)ks * (BK / 2) + part * 16);
          }
          if (lane < C::RW) {
            const uint8_t* sp = f_rec + soff + (f_row0 + lane) * (size_t)(K / G) + (size_t)ks * (BK / G);
            if (kSB == 8) cp8(slot + C::RW * C::RAW_ROW + lane * 8, sp);
            else cp4(slot + C::RW * C::RAW_ROW + lane * 8, sp);
          }
        }
      }
      cp_async_commit();  // one group per super-step, empty or not, so the group count stays aligned
    };
    for (int ss = 0; ss < C::RAW_DEPTH; ++ss) fetch(ss);
    int c_tile = -1;
    bool poison = false;
    bool alive = true;
    for (int ss = 0; ss < nss && alive; ++ss) {
      // this super-step's raw bytes: the oldest of the RAW_DEPTH groups in flight
      asm volatile("cp.async.wait_group %0;" ::"n"(C::RAW_DEPTH - 1) : "memory");
      __syncwarp();
      const uint8_t* slot = raw_wp + (size_t)(ss % C::RAW_DEPTH) * C::RAW_STEP;
      const uint2 sw8 = *reinterpret_cast<const uint2*>(slot + C::RW * C::RAW_ROW + r_local * 8);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int gs = 2 * ss + j;
        const int lt = gs / KSTEPS;
        if (lt != c_tile) {
          c_tile = lt;
          int mt;
          const int4 ti = tile_of(a, blockIdx.x + lt * gridDim.x, MT, mt);
          const uint8_t* rec = tile_record(a, ti.x);
          poison = rec == nullptr;
          if (poison && pid == 0)
            moe::status_or(a.st, a.ptrs[ti.x] == nullptr ? MOE_DEV_NULL_EXPERT : MOE_DEV_MISALIGNED);
        }
        uint4 q[C::UNITS];
#pragma unroll
        for (int u = 0; u < C::UNITS; ++u)
          q[u] = *reinterpret_cast<const uint4*>(slot + r_local * C::RAW_ROW +
                                                 (((2 * j + half + u) ^ ((r_local >> 1) & 3)) << 4));
        // scale bytes of the step: NVFP4 4 per step (2 per half), MXFP4 2 per step (1 per half)
        const uint32_t sword = j == 0 ? sw8.x : sw8.y;  // NVFP4: bytes of step j; MXFP4: both steps in sw8.x
        uint32_t sstep;
        if (FMT == MOE_FMT_NVFP4) sstep = sword >> (16 * half);
        else sstep = sw8.x >> (16 * j + 8 * half);
        uint4 out[C::UNITS][4];
#pragma unroll
        for (int u = 0; u < C::UNITS; ++u) {
          const uint4 qq = poison ? make_uint4(0u, 0u, 0u, 0u) : q[u];
          const uint32_t sb =
              poison ? 0u : (FMT == MOE_FMT_NVFP4 ? (sstep >> (16 * u)) & 0xFFFFu : (sstep >> (8 * u)) & 0xFFu);
          if constexpr (kF16) dequant_unit_f16(qq, sb, poison, out[u]);
          else dequant_unit_bf16<FMT>(qq, sb, poison, out[u]);
        }
        const int as = gs % C::A_STAGES;
        // the outcome is made warp-uniform: the warp synchronises again below
        const bool ok = __all_sync(0xffffffffu, !*abort_flag &&
                                   mbar_wait(&a_empty[as], ((gs / C::A_STAGES) & 1) ^ 1, globaltimer() + kWaitNs));
        if (!ok) {
          if (lane == 0) fail();
          alive = false;
          break;
        }
        uint8_t* row_base = sA + (size_t)as * C::NA * C::A_BYTES + (size_t)m * C::A_BYTES + (size_t)r * 128;
#pragma unroll
        for (int u = 0; u < C::UNITS; ++u)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int ch = (c0 / 8) + u * 4 + cc;  // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(row_base + ((ch ^ (r & 7)) << 4)) = out[u][cc];
          }
        fence_proxy_async();
        mbar_arrive(&a_full[as]);
      }
      // every lane has read the slot: refill it with the super-step RAW_DEPTH ahead
      __syncwarp();
      if (alive) fetch(ss + C::RAW_DEPTH);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------------------------------------- epilogue
    // A warp may only touch TMEM lanes 32*(warp % 4) .. +31.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;               // accumulator row = weight row in tile
    const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    for (int lt = 0; lt < my_tiles; ++lt) {
      int mt;
      const int4 ti = tile_of(a, blockIdx.x + lt * gridDim.x, MT, mt);
      const int buf = lt & 1;
      // per-column token, router weight and x scale, once per tile, double
      // buffered: a thread can be at most one tile ahead of the slowest
      // (acc_empty counts every epilogue thread), so tile lt never overwrites
      // a table in use.
      int* tok = col_tok + buf * BN;
      float* wcol = col_w + buf * BN;
      float* xs = col_xs + buf * BN;
      if (et < ti.z) {
        const int p = __ldg(a.pairs + ti.y + et);
        tok[et] = p / a.k;
        wcol[et] = __ldg(a.weights + p);
        xs[et] = a.xscale ? __ldg(a.xscale + p / a.k) : 1.0f;
      }
      mbar_arrive(&tab_ready[buf]);
      if (!mbar_wait(&tab_ready[buf], (lt >> 1) & 1, globaltimer() + kWaitNs)) {
        fail();
        break;
      }
      if (*abort_flag || !mbar_wait_backoff(&acc_full[buf], (lt >> 1) & 1, globaltimer() + kWaitNs)) {
        fail();
        break;
      }
      fence_after_sync();
      const uint32_t acc = lane_addr + (uint32_t)(buf * C::ACC_COLS);
      const int col = mt * BM + row;
      for (int c0 = 0; c0 < ti.z; c0 += 16) {
        uint32_t v0[16];
        tmem_ld16(acc + c0, v0);
        if (PHASE == 0) {
          uint32_t v1[16];
          tmem_ld16(acc + BN + c0, v1);
          tmem_ld_wait();
          uint16_t* hrow = a.hbuf + (size_t)(ti.y + c0) * a.I + col;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.z) {
              const float sc = xs[c0 + j];
              const float g = __uint_as_float(v0[j]) * sc;
              const float u = __uint_as_float(v1[j]) * sc;
              const float h = g / (1.0f + expf(-g)) * u;
              const __nv_bfloat16 hb = __float2bfloat16_rn(h);
              hrow[(size_t)j * a.I] = *reinterpret_cast<const uint16_t*>(&hb);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < ti.z)
              atomicAdd(a.y + (size_t)tok[c0 + j] * a.H + col, wcol[c0 + j] * __uint_as_float(v0[j]));
          }
        }
      }
      fence_before_sync();
      mbar_arrive(&acc_empty[buf]);
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// exclusive scan of ceil(count[e] / BN) -> ntile_off[E+1], then the token-tile
// table: tile ntile_off[e] + n of expert e = {e, offsets[e] + n*BN, rows, 0};
// *ntiles = ntile_off[E].  One CTA.
__global__ void __launch_bounds__(1024) tile_scan_kernel(const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets, int E,
                                                         int32_t* __restrict__ ntile_off, int4* __restrict__ tiles,
                                                         int32_t* __restrict__ ntiles) {
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
    if (e < E) {
      ntile_off[e] = excl;
      const int cnt = counts[e], beg = offsets[e];
      for (int n = 0; n < c; ++n) tiles[excl + n] = make_int4(e, beg + n * BN, min(BN, cnt - n * BN), 0);
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + c;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    ntile_off[E] = carry;
    *ntiles = carry;
  }
}

// x (BF16) -> FP16 x * 2^e_t for the NVFP4 gate/up MMA, one warp per token:
// e_t puts the token's largest magnitude in [2^14, 2^15), so every BF16 value
// down to 2^-24 of that maximum is exact in FP16 (smaller ones are below the
// last bit of any sum they enter); xscale[t] = 2^-e_t undoes it in the
// epilogue (exact).
__global__ void x_to_f16_kernel(const uint16_t* __restrict__ x, int T, int H, uint16_t* __restrict__ x16,
                                float* __restrict__ xscale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= T) return;
  const uint16_t* xr = x + (size_t)warp * H;
  unsigned mx = 0u;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + i));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, max((wv[j] & 0x7FFFu) << 16, ((wv[j] >> 16) & 0x7FFFu) << 16));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  const int e = moe::dm::f16_shift(__uint_as_float(mx));
  const float sc = moe::dm::pow2f(e);
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + i));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = moe::dm::pack_h2(moe::bf16_bits_to_f32(wv[j] & 0xFFFFu) * sc, moe::bf16_bits_to_f32(wv[j] >> 16) * sc);
    *reinterpret_cast<uint4*>(x16 + (size_t)warp * H + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) xscale[warp] = moe::dm::pow2f(-e);
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
  size_t counts, offsets, ntile, tiles, ntiles, pairs, hbuf, x16, xscale, bucket, total;
};

WsLayout ws_layout(int T, int k, int E, const moe_expert_shape& s) {
  WsLayout w;
  const size_t P = (size_t)T * k;
  const size_t max_tiles = (P + BN - 1) / BN + (size_t)E;
  size_t o = 0;
  w.counts = o;  o = align256(o + (size_t)E * 4);
  w.offsets = o; o = align256(o + (size_t)(E + 1) * 4);
  w.ntile = o;   o = align256(o + (size_t)(E + 1) * 4);
  w.tiles = o;   o = align256(o + max_tiles * 16);
  w.ntiles = o;  o = align256(o + 4);
  w.pairs = o;   o = align256(o + P * 4);
  w.hbuf = o;    o = align256(o + P * (size_t)s.inter * 2);
  const bool f16 = s.format == MOE_FMT_NVFP4;
  w.x16 = o;     o = align256(o + (f16 ? (size_t)T * s.hidden * 2 : 0));
  w.xscale = o;  o = align256(o + (f16 ? (size_t)T * 4 : 0));
  w.bucket = o;  o = align256(o + moe_bucket_workspace(T, k, E));
  w.total = o;
  return w;
}

template <int FMT, int PHASE>
int launch_phase(const GroupedArgs& a, cudaStream_t st) {
  using C = Cfg<PHASE>;
  static moe::SmemGrant granted;
  if (!moe::grant_smem(grouped_kernel<FMT, PHASE>, C::SMEM, granted, kThreads)) return MOE_ERR_CUDA;
  const int sms = moe::device_info().sms;
  if (sms <= 0) return MOE_ERR_CUDA;
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
  int4* tiles = reinterpret_cast<int4*>(ws + L.tiles);
  int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
  int32_t* pairs = reinterpret_cast<int32_t*>(ws + L.pairs);
  int rc = moe_bucket_by_expert(idx, T, k, E, counts, offsets, pairs, ws + L.bucket,
                                L.total - L.bucket, dev_status, stream);
  if (rc != MOE_OK) return rc;
  tile_scan_kernel<<<1, 1024, 0, st>>>(counts, offsets, E, ntile, tiles, ntiles);
  if (cudaMemsetAsync(y, 0, (size_t)T * s.hidden * sizeof(float), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  GroupedArgs a;
  a.x = x_bf16;
  a.xscale = nullptr;
  a.pairs = pairs;
  a.tiles = tiles;
  a.ntiles = ntiles;
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
    float* xsc = reinterpret_cast<float*>(ws + L.xscale);
    x_to_f16_kernel<<<(unsigned)((T + 7) / 8), 256, 0, st>>>(x_bf16, T, s.hidden, x16, xsc);
    GroupedArgs a0 = a;
    a0.x = x16;
    a0.xscale = xsc;
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
