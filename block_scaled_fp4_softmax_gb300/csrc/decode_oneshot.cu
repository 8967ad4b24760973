// One-shot decode expert pass (T*k <= 64 pairs whose per-CTA share of the
// selected records fits in shared memory), one launch per MoE layer
// ("Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "The engine", item 4: the single-token NVFP4
// SwiGLU expert kernel; the sum over the k experts weighted by the
// renormalised router probabilities).
//
//  0. Prologue, before the wait for the previous kernel: thread 0 bulk-copies
//     the CTA's router rows and the expert pointer table into shared memory
//     (a launch that runs the whole layer); warp 15, the loader, plans the
//     CTA's share of the selected records and sets up the copy barriers.
//  1. Router (whole-layer launch), warps 0-14: x = RMS chaining of the
//     previous output (or x itself), the logits of the CTA's experts, a grid
//     barrier, then every CTA takes the top-k of all logits itself.
//  2. Copies: the loader's lanes issue every bulk copy of the CTA's share at
//     once (the copy engine of an SM completes only a few copies per
//     microsecond, so the copies are few and large); warps 0-14 stage x as
//     FP16, scaled per token by a power of two (exact).
//  3. gate/up + SwiGLU: each warp takes a contiguous block of the CTA's row
//     pairs, up to three rows at a time, as soon as their piece has landed;
//     h = silu(g) * u goes to global scratch.
//  4. Grid barrier (one release arrival per CTA on a counter that only grows).
//  5. down: the CTA owns whole output rows.  h of its tokens' pairs is staged
//     as FP32; task (row, expert) -> a group of lanes, each lane a few units
//     (16 code bytes = 32 elements) with packed FP32 FMAs, the group reduced
//     by shuffles; each row adds its k weighted expert outputs in expert
//     order and writes y.  Every sum has a fixed order, so y is
//     bit-reproducible.
#include <algorithm>

#include "common.cuh"
#include "decode_math.cuh"
#include "decode_oneshot.h"
#include "router_math.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace os {

// Where a bounded wait gave up: the first one in the launch's workspace
// (byte 192 of the header, a 64-bit word that stays zero while every wait
// succeeds; the ring kernel's barrier words sit at 128) gets
// site << 56 | (layer + 1) << 32 | block.
enum WaitSite : unsigned {
  kSiteRouter = 1, kSiteScales, kSitePiece, kSiteDown, kSiteGrid1, kSiteGrid2, kSiteLayer, kSiteLoader
};
__device__ __forceinline__ void note_timeout(unsigned long long* bar, unsigned site, int layer) {
  unsigned long long* diag = bar + 24;
  atomicCAS(diag, 0ull, (unsigned long long)site << 56 | (unsigned long long)(layer + 1) << 32 | blockIdx.x);
}

// Waits (bounded by wait_ns) for the phase of one barrier with the given
// parity; on timeout flags the launch, records the site and returns false.
__device__ __forceinline__ bool await(uint64_t* bar, uint32_t parity, Tab& tb, const DecodeOneshotArgs& a,
                                      unsigned site, int layer) {
  volatile int* abort_flag = tb.flags;
  if (*abort_flag) return false;
  if (tc::mbar_wait(bar, parity, tc::globaltimer() + a.wait_ns)) return true;
  *abort_flag = 1;
  status_or(a.status, MOE_DEV_TIMEOUT);
  note_timeout(a.bar, site, layer);
  return false;
}

// Exchange words between CTAs: a value's 32 bits and a 32-bit tag in one
// 8-byte word, stored and loaded whole (single-copy atomic), so a reader
// that sees this layer's tag sees the value written with it; the data is its
// own flag and no grid barrier separates writer and reader.  Tags are
// quiet-NaN patterns 0x7FC00001 .. 0x7FFFFFFE, one per layer of the
// workspace's counter (cycling after about 4 million layers); no FP32
// arithmetic of this library yields them (its NaNs are 0x7FFFFFFF and
// 0x7FC00000), so FP32 data that other paths leave in the workspace never
// passes for a tag.
__device__ __forceinline__ uint32_t layer_tag(unsigned long long n) {
  return 0x7FC00000u | (1u + (uint32_t)(n % 0x3FFFFEull));
}
__device__ __forceinline__ void put_tagged(unsigned long long* p, float v, uint32_t tag) {
  const unsigned long long w = (unsigned long long)tag << 32 | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// The value of a word already loaded, or, when it does not carry `tag` yet,
// of the word polled until it does (bounded: on timeout the launch is
// flagged, the site recorded, and NaN returned).
__device__ __forceinline__ float tagged_value(unsigned long long w, const unsigned long long* p, uint32_t tag,
                                              Tab& tb, const DecodeOneshotArgs& a, unsigned site, int layer) {
  if ((uint32_t)(w >> 32) == tag) return __uint_as_float((uint32_t)w);
  volatile int* abort_flag = tb.flags;
  const uint64_t dl = global_ns() + a.wait_ns;
  while (!*abort_flag) {
    w = rt::ld_relaxed_u64(p);
    if ((uint32_t)(w >> 32) == tag) return __uint_as_float((uint32_t)w);
    if (global_ns() > dl) {
      *abort_flag = 1;
      status_or(a.status, MOE_DEV_TIMEOUT);
      note_timeout(a.bar, site, layer);
    }
  }
  return __uint_as_float(0x7FC00000u);
}

// Grid barrier, called by one thread per CTA after a CTA-wide barrier: one
// arrival on a counter that only grows (a release reduction, so the writes
// of every thread of the CTA that precede the CTA-wide barrier are visible
// to the CTAs that pass), then an acquire poll until the counter reaches
// `target` = base + n * grid for the launch's n-th barrier.  base is the
// counter at the start of the launch, rounded down to a multiple of the
// grid: every earlier launch has passed all its barriers by then, and each
// CTA reads the counter before its own first arrival, so fewer than grid
// arrivals of this launch can precede the read.  `between` runs after the
// arrival and before the poll (work that overlaps the wait without holding
// up the release).  False on timeout, which also flags the launch.
template <bool RELEASE = true, class F>
__device__ __forceinline__ bool grid_sync_thread(unsigned long long target, Tab& tb, const DecodeOneshotArgs& a,
                                                 unsigned site, int layer, F&& between) {
  volatile int* abort_flag = tb.flags;
  int good = !*abort_flag;
  if (good) {
    if (RELEASE) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
    else asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
    ++tb.arrived;
    between();
    const uint64_t dl = global_ns() + a.wait_ns;
    while (dm::ld_acquire_u64(a.bar) < target) {
      if (global_ns() > dl) {
        good = 0;
        note_timeout(a.bar, site, layer);
        break;
      }
    }
  }
  if (!good) {
    *abort_flag = 1;
    status_or(a.status, MOE_DEV_TIMEOUT);
  }
  return good;
}
template <bool RELEASE = true>
__device__ __forceinline__ bool grid_sync_thread(unsigned long long target, Tab& tb, const DecodeOneshotArgs& a,
                                                 unsigned site, int layer) {
  return grid_sync_thread<RELEASE>(target, tb, a, site, layer, [] {});
}

// The CTA's share of the router rows of a fused launch: experts
// [re0, re0 + rne) of E, epc per CTA.
struct RouterShare {
  int re0, rne;
  uint32_t wr_bytes;
};
__device__ __forceinline__ RouterShare router_share(const DecodeOneshotArgs& a, bool fused) {
  const int epc = (a.E + (int)gridDim.x - 1) / (int)gridDim.x;
  RouterShare r;
  r.re0 = blockIdx.x * epc;
  r.rne = fused ? max(0, min(epc, a.E - r.re0)) : 0;
  r.wr_bytes = (uint32_t)r.rne * (uint32_t)a.H * 2u;
  return r;
}
// The pointer table goes to shared memory with the router rows when the
// rows are staged and the table's bulk copy is 16-byte aligned.
__device__ __forceinline__ bool ptrs_staged(const DecodeOneshotArgs& a) {
  return a.geo.rstage != 0 && (reinterpret_cast<uintptr_t>(a.ptrs) & 15u) == 0 && (a.E & 1) == 0;
}

// Thread 0: bulk copies of layer l's router rows of this CTA and of the
// pointer table into the x/h region, completing one phase of `bar` (set up
// here for layer 0).
__device__ __forceinline__ void stage_router(const DecodeOneshotArgs& a, uint8_t* smem, uint64_t* bar, int l) {
  const RouterShare r = router_share(a, true);
  if (l == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
  }
  const uint32_t ptr_bytes = ptrs_staged(a) ? (uint32_t)a.E * 8u : 0u;
  tc::mbar_arrive_expect_tx(bar, r.wr_bytes + ptr_bytes);
  if (r.wr_bytes)
    tc::bulk_g2s(tc::smem_u32(smem + a.geo.off_act), a.wr + ((size_t)l * a.E + r.re0) * a.H, r.wr_bytes, bar);
  if (ptr_bytes)
    tc::bulk_g2s(tc::smem_u32(smem + a.geo.off_act + r.wr_bytes), a.ptrs + (size_t)l * a.E, ptr_bytes, bar);
}

// STACK: the launch runs a.layers layers (a whole-stack launch); otherwise
// exactly one, and the layer loop compiles away.
template <int FMT, int UPR, int UPDR, bool STACK>
__global__ void __launch_bounds__(kThreads, 1) oneshot_kernel(DecodeOneshotArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_launch_dependents();
  // A launch runs a.layers >= 1 layers (more than one only for a whole-layer
  // launch, moe_decode_stack): layer 0 from a.x or a.y_prev, every later layer
  // RMS-chained from the previous layer's y.  Each layer has nb grid barriers
  // on the workspace counter: the logits (fused launch), h, and, between the
  // layers of a whole-stack launch, y.  The counter at launch start, over the
  // grid, is the base: layer L's barrier n waits for (base + nb L + n) grid.
  // The logits travel as words tagged with tag(base + nb L + 1) and are
  // checked after their barrier, which therefore needs no release (h and y
  // are FP32, published by release arrivals: tagged h doubles the bytes each
  // CTA reads and measured slower).
  // The mbarriers are set up once; each completes one phase per layer, so
  // layer L waits for the phase of parity L & 1.
  const int nl = STACK ? a.layers : 1;
  for (int L = 0; L < nl; ++L) {
  const uint32_t ph = (uint32_t)L & 1u;
  const uint16_t* L_wr = a.wr ? a.wr + (size_t)L * a.E * a.H : nullptr;
  const void* const* L_ptrs = a.ptrs + (size_t)L * a.E;
  const float* L_bias = a.bias ? a.bias + (size_t)L * a.E : nullptr;
  const uint16_t* L_x = L == 0 ? a.x : nullptr;
  const float* L_yprev = L == 0 ? a.y_prev : a.y;
  int32_t* L_idx_out = a.idx_out ? a.idx_out + (size_t)L * a.T * a.k : nullptr;
  float* L_w_out = a.w_out ? a.w_out + (size_t)L * a.T * a.k : nullptr;
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = FMT == MOE_FMT_NVFP4 ? 2 : 1;
  const bool fused = L_wr != nullptr;
  const unsigned nb = (fused ? 2u : 1u) + (STACK ? 1u : 0u);
  const Geo& g = a.geo;
  const RecordOffsets o = record_offsets(a.H, a.I, FMT);
  const int upr = UPR > 0 ? UPR : a.H >> 5;
  const int updr = UPDR > 0 ? UPDR : a.I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.T * a.k;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  Tab& tb = *reinterpret_cast<Tab*>(smem + g.off_tab);
  const uint8_t* codes1 = smem + g.off_codes1;
  const uint8_t* scales1 = smem + g.off_scales1;
  const uint8_t* codes2 = smem + g.off_codes2;
  const uint8_t* scales2 = smem + g.off_scales2;
  uint4* act = reinterpret_cast<uint4*>(smem + g.off_act);
  volatile int* abort_flag = tb.flags;
  // layer L's barrier n (thread 0, which holds the base)
  auto bar_target = [&](unsigned n) { return (tb.bar_base + nb * L + n) * gridDim.x + a.barrier_extra; };

  // router rows of this CTA's experts (fused launch) and the pointer table:
  // neither depends on the previous kernel, so they are fetched before the
  // wait for it -- into shared memory (the x/h region, which they leave
  // before x arrives there) when the plan has room, else into L2.  Layer
  // L + 1's are fetched during the barrier at the end of layer L.
  const RouterShare rs = router_share(a, fused);
  const int re0 = rs.re0, rne = rs.rne;
  const uint32_t wr_bytes = rs.wr_bytes;
  const bool rstaged = g.rstage != 0;
  const bool pstaged = ptrs_staged(a);
  if (!pstaged)
    for (int i = threadIdx.x; i < (a.E * 8 + 127) / 128; i += kThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(L_ptrs) + (size_t)i * 128));
  if (!rstaged) {
    const char* wb = fused ? reinterpret_cast<const char*>(L_wr + (size_t)re0 * a.H) : nullptr;
    for (size_t off = (size_t)threadIdx.x * 128; off < wr_bytes; off += (size_t)kThreads * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(wb + off));
  }
  if (L == 0) {
    // later layers are reset at the end of the previous one
    if (threadIdx.x == 0) {
      tb.flags[0] = 0;  // a wait that ran out stays flagged for the launch's later layers
      if (rstaged) stage_router(a, smem, &bars[kBarRouter], 0);
    }
    if (threadIdx.x < kMaxPairs) tb.amax[threadIdx.x] = 0u;
    __syncthreads();
  }

  if (warp == kCWarps) {
    // ------------------------------------------------------------ loader
    // The plan of the CTA's copies has no data dependence: lane 0 builds it
    // (and the barriers' arrival counts: one per copy, plus one by lane 0 on
    // every barrier) while, in a fused launch, warps 0-14 run the router.
    // It is the same for every layer.
    if (lane == 0 && L == 0) {
      uint32_t n_scale, n_down;
      build_tables(g, blockIdx.x, o, tb, n_scale, n_down);
      for (int i = 0; i < kMaxPieces; ++i) tc::mbar_init(&bars[i], i < tb.npieces ? 3u : 1u);
      tc::mbar_init(&bars[kBarScales], n_scale + 1);
      tc::mbar_init(&bars[kBarDown], n_down + 1);
      tc::mbar_fence_init();
    }
    __syncwarp();
    if (L == 0) pdl_wait();
    if (!fused) {
      for (int p = lane; p < P; p += 32) {
        tb.recs[p] = dm::checked_record(a.idx[p], a.E, L_ptrs, blockIdx.x == 0 ? a.status : nullptr);
        tb.wts[p] = a.w[p];
      }
      __syncwarp();
    } else {
      asm volatile("bar.sync 3, %0;" ::"n"(kThreads) : "memory");  // the router's records are in place
    }
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");  // barriers set up, records in place
    // One copy per lane; a copy of a missing record still arrives (0 bytes).
    // The gate/up pieces and scales go first.  The down rows are needed only
    // after the second grid barrier, so they are issued once the gate/up bytes
    // have landed: issued together, they would share the HBM stream with the
    // gate/up bytes and delay the gate/up pass by about a third.
    const uint32_t base = tc::smem_u32(smem);
    auto issue_if = [&](auto take) {
      for (int c = lane; c < tb.ncopies; c += 32) {
        if (!take((int)tb.cbar[c])) continue;
        const uint8_t* rec = tb.recs[tb.cpair[c]];
        uint64_t* bar = &bars[tb.cbar[c]];
        tc::mbar_arrive_expect_tx(bar, rec ? tb.cbytes[c] : 0u);
        if (rec) tc::bulk_g2s(base + tb.cdst[c], rec + tb.csrc[c], tb.cbytes[c], bar);
      }
    };
    // Once the launch is flagged (a wait gave up), no more copies are issued:
    // nothing waits for them any more.  Lane 0 decides for the warp.
    const bool live = __shfl_sync(0xffffffffu, (int)(*abort_flag == 0), 0) != 0;
    if (live) issue_if([](int b) { return b != kBarDown; });
    int landed = live;
    if (lane == 0 && live) {
      for (int i = 0; i < kNumBars; ++i)
        if (i != kBarDown) tc::mbar_arrive(&bars[i]);
      const uint64_t dl = tc::globaltimer() + a.wait_ns;
      for (int i = 0; i < kNumBars; ++i)
        if (i != kBarDown && !tc::mbar_wait_backoff(&bars[i], ph, dl)) landed = 0;
      if (!landed) {
        *abort_flag = 1;
        status_or(a.status, MOE_DEV_TIMEOUT);
        note_timeout(a.bar, kSiteLoader, L);
      }
    }
    if (__shfl_sync(0xffffffffu, landed, 0)) {
      issue_if([](int b) { return b == kBarDown; });
      if (lane == 0) {
        tc::mbar_arrive(&bars[kBarDown]);
        // no copy may still be in flight when the layer (or the CTA) ends
        if (!tc::mbar_wait_backoff(&bars[kBarDown], ph, tc::globaltimer() + a.wait_ns)) {
          *abort_flag = 1;
          status_or(a.status, MOE_DEV_TIMEOUT);
          note_timeout(a.bar, kSiteLoader, L);
        }
      }
    }
  } else {

  if (L == 0) {
    pdl_wait();
    // the counter at the start of this launch, over the grid: every earlier
    // launch has added its grid x layers by now, and fewer than a grid of
    // this launch's additions can precede the read (each CTA adds only after
    // its own read), so every CTA gets the same number.  Thread 0 reads it;
    // the router's (or the x staging's) first barrier publishes it.
    if (threadIdx.x == 0) {
      tb.bar_base = rt::ld_relaxed_u64(a.bar) / gridDim.x;
      tb.arrived = 0;
    }
  }

  uint16_t* xb = reinterpret_cast<uint16_t*>(smem + g.off_xb + 1024 + 4096);  // x (BF16), fused launch
  if (fused) {
    // ---------------------------------------------------------- router
    // x = RMS chaining of y_prev (or x itself), the logits of this CTA's
    // experts, a grid barrier, then every CTA takes the top-k of all logits
    // itself; the same fixed orders as the router kernels, so the same bits.
    // Warps 0-14 (named barrier 4); the loader warp plans meanwhile and takes
    // the records through named barrier 3.
    float* rpart = reinterpret_cast<float*>(smem + g.off_xb);
    for (int t = 0; t < a.T; ++t) {
      if (L_yprev) {
        const float* yr = L_yprev + (size_t)t * a.H;
        // a whole-stack launch reads the y it wrote in the previous layer:
        // through L2 only, as L1 is not coherent across SMs
        const float r = rt::rms_inv_fixed_order<4, kCThreads, STACK>(yr, a.H, a.eps, rpart);
        for (int i = threadIdx.x; i < a.H; i += kCThreads) {
          const uint16_t x16 = rt::f32_to_bf16_bits(__fmul_rn(STACK ? __ldcg(yr + i) : yr[i], r));
          xb[(size_t)t * a.H + i] = x16;
          if (blockIdx.x == 0 && a.x_out) a.x_out[(size_t)t * a.H + i] = x16;
        }
      } else {
        for (int i = threadIdx.x * 8; i < a.H; i += kCThreads * 8) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(L_x + (size_t)t * a.H + i));
          *reinterpret_cast<uint4*>(xb + (size_t)t * a.H + i) = v;
          if (blockIdx.x == 0 && a.x_out) *reinterpret_cast<uint4*>(a.x_out + (size_t)t * a.H + i) = v;
        }
      }
    }
    tc::named_sync(4, kCThreads);
    const bool rin = !rstaged || await(&bars[kBarRouter], ph, tb, a, kSiteRouter, L);
    const uint16_t* wsm = reinterpret_cast<const uint16_t*>(smem + g.off_act);
    for (int task = warp; task < a.T * rne; task += kCWarps) {
      const int t = task / rne, q = task - t * rne;
      float v;
      if (rstaged) v = rin ? rt::logit_dot<true>(xb + (size_t)t * a.H, wsm + (size_t)q * a.H, a.H, lane)
                           : __uint_as_float(0x7FC00000u);
      else v = rt::logit_dot(xb + (size_t)t * a.H, L_wr + (size_t)(re0 + q) * a.H, a.H, lane);
      if (lane == 0) {
        const float lv = L_bias ? __fadd_rn(v, L_bias[re0 + q]) : v;
        a.logits[(size_t)t * a.E + re0 + q] = lv;
        put_tagged(a.xlog + (size_t)t * kLogitStride + re0 + q, lv, layer_tag(tb.bar_base + nb * L + 1));
      }
    }
    // the logits' barrier: a relaxed arrival (no wait for the stores above),
    // the words themselves are checked below
    tc::named_sync(4, kCThreads);
    if (threadIdx.x == 0) grid_sync_thread<false>(bar_target(1), tb, a, kSiteGrid1, L);
    tc::named_sync(4, kCThreads);
    unsigned long long* fin = reinterpret_cast<unsigned long long*>(smem + g.off_xb + 1024);
    // every CTA's logits of token t, each word checked for this layer's tag
    // (one still in flight is polled), into the gate/up region, which is free
    // until the copies are issued after the router
    float* lsm = reinterpret_cast<float*>(smem + g.off_codes1);
    const uint32_t want = layer_tag(tb.bar_base + nb * L + 1);
    for (int t = 0; t < a.T; ++t) {
      {
        const unsigned long long* src = a.xlog + (size_t)t * kLogitStride;
        constexpr int kPer = (kLogitStride + kCThreads - 1) / kCThreads;
        unsigned long long wv[kPer];
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int e = threadIdx.x + kCThreads * m;
          wv[m] = e < a.E ? rt::ld_relaxed_u64(src + e) : 0ull;
        }
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int e = threadIdx.x + kCThreads * m;
          if (e < a.E) lsm[e] = tagged_value(wv[m], src + e, want, tb, a, kSiteGrid1, L);
        }
      }
      tc::named_sync(4, kCThreads);
      // set only before the barrier above, so every thread reads the same
      const bool have_logits = *abort_flag == 0;
      int my_e = 0;
      float my_l = 0.0f;
      if (have_logits) rt::topk_block_fast<kCWarps, 4, true>(lsm, a.E, a.k, fin, my_e, my_l);
      if (warp == 0) {
        const float wgt = rt::topk_weight(lane, a.k, my_l);
        if (lane < a.k) {
          const int p = t * a.k + lane;
          const void* const* pt =
              pstaged ? reinterpret_cast<const void* const*>(smem + g.off_act + wr_bytes) : L_ptrs;
          tb.recs[p] = have_logits && rin ? dm::checked_record(my_e, a.E, pt, blockIdx.x == 0 ? a.status : nullptr)
                                          : nullptr;
          tb.wts[p] = wgt;
          if (blockIdx.x == 0) {
            L_idx_out[p] = my_e;
            L_w_out[p] = wgt;
          }
        }
      }
    }
    // the logits' generic stores in the gate/up region come before the
    // loader's bulk copies there
    tc::fence_proxy_async();
    tc::named_sync(4, kCThreads);  // the staged pointers in the x/h region are no longer read
    asm volatile("bar.arrive 3, %0;" ::"n"(kThreads) : "memory");  // records in place for the loader
  }


  // ---------------------------------------------------------------- compute
  // x: per-token max |x| (pass 1), then FP16 quads [t][4][H/32] of x * 2^e
  // (exact: BF16 has 8 significant bits and the scaled values lie in FP16's
  // normal range)
  const int nx8 = a.T * a.H / 8;
  const uint4* xg = reinterpret_cast<const uint4*>(fused ? xb : L_x);
  uint4 xr = make_uint4(0u, 0u, 0u, 0u);
  for (int b = warp * 32; b < nx8; b += kCThreads) {
    const int q = b + lane;
    unsigned m = 0u;
    int key = -1;
    if (q < nx8) {
      const uint4 v = fused ? xg[q] : __ldg(xg + q);
      if (b == warp * 32) xr = v;
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = max(m, max((wv[i] & 0x7FFFu) << 16, ((wv[i] >> 16) & 0x7FFFu) << 16));
      key = q * 8 / a.H;
    }
    if (dm::group_max(key, m)) atomicMax(&tb.amax[key], m);
  }
  tc::named_sync(1, kCThreads);
  if (threadIdx.x < a.T) tb.tsc[threadIdx.x] = dm::pow2f(-dm::f16_shift(__uint_as_float(tb.amax[threadIdx.x])));
  for (int b = warp * 32; b < nx8; b += kCThreads) {
    const int q = b + lane;
    if (q < nx8) {
      const uint4 v = b == warp * 32 ? xr : (fused ? xg[q] : __ldg(xg + q));
      const int t = q * 8 / a.H, hh = q * 8 - t * a.H;
      const float sc = dm::pow2f(dm::f16_shift(__uint_as_float(tb.amax[t])));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t o4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o4[i] = dm::pack_h2(bf16_bits_to_f32(wv[i] & 0xFFFFu) * sc, bf16_bits_to_f32(wv[i] >> 16) * sc);
      act[(size_t)t * 4 * upr + ((hh & 31) >> 3) * upr + (hh >> 5)] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
  asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");  // x staged, records in place

  // gate/up + SwiGLU
  const int n1 = share_lo(blockIdx.x + 1, (int)g.R1, g.grid) - share_lo(blockIdx.x, (int)g.R1, g.grid);
  if constexpr (UPR > 0 && UPR <= 96) {
    // Rows dealt round-robin over the compute warps in the CTA's row order, so
    // that every warp has a row of each piece as the pieces land (the pieces
    // land one after the other, in the order they were issued).  Lane j keeps
    // x of units j, j + 32, j + 64 (of the row's token) in registers and
    // takes those units of the gate and the up row; the lane sums run in unit
    // order and are combined by an xor butterfly, a fixed order per row.
    constexpr int UPL = (UPR + 31) / 32;
    uint4 xr[UPL][4];
    int xt = -1;
    bool scales_in = false;
    for (int q = warp; q < n1; q += kCWarps) {
      int s = 0;
      while (s + 1 < tb.nseg1 && tb.sq0[s + 1] <= q) ++s;
      int pa = 0;
      while (pa + 1 < tb.npieces && tb.pq0[pa + 1] <= q) ++pa;
      const int p = tb.sp[s], t = p / a.k;
      bool ok = tb.recs[p] != nullptr;
      if (ok && !scales_in) ok = scales_in = await(&bars[kBarScales], ph, tb, a, kSiteScales, L);
      if (ok) ok = await(&bars[pa], ph, tb, a, kSitePiece, L);
      if (t != xt) {
        xt = t;
        const uint4* xt4 = act + (size_t)t * 4 * UPR;
#pragma unroll
        for (int i = 0; i < UPL; ++i) {
          const int u = lane + 32 * i;
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) xr[i][wi] = u < UPR ? xt4[wi * UPR + u] : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float gsum = 0.f, usum = 0.f;
      if (ok) {
        const uint8_t* grow = codes1 + tb.poff[pa] + (size_t)(q - tb.pq0[pa]) * (a.H / 2);
        const uint8_t* urow = grow + (size_t)tb.pn[pa] * (a.H / 2);
        const uint8_t* gsr = scales1 + tb.gwo[s] + (size_t)(q - tb.sq0[s]) * (a.H / G);
        const uint8_t* usr = scales1 + tb.uwo[s] + (size_t)(q - tb.sq0[s]) * (a.H / G);
#pragma unroll
        for (int i = 0; i < UPL; ++i) {
          const int u = lane + 32 * i;
          if (u < UPR) {
            gsum += dm::unit_dot_hx<FMT>(*reinterpret_cast<const uint4*>(grow + 16 * u),
                                         dm::scale_bits<FMT>(gsr + sstep * u), xr[i]);
            usum += dm::unit_dot_hx<FMT>(*reinterpret_cast<const uint4*>(urow + 16 * u),
                                         dm::scale_bits<FMT>(usr + sstep * u), xr[i]);
          }
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        gsum += __shfl_xor_sync(0xffffffffu, gsum, d);
        usum += __shfl_xor_sync(0xffffffffu, usum, d);
      }
      if (lane == 0) {
        const float ts = tb.tsc[t];
        const float gv = gsum * ts, uv = usum * ts;
        a.hws[(size_t)p * a.I + tb.si0[s] + (q - tb.sq0[s])] =
            ok ? gv / (1.0f + expf(-gv)) * uv : __uint_as_float(0x7FC00000u);
      }
    }
  } else {
  // Other shapes: warp w takes a contiguous block of the CTA's row pairs and
  // works on up to kRows of them (rows of one pair) at a time, so that each
  // load of x from shared memory serves them all.  Per row, the sums run in
  // the same order as for a single row.
  constexpr int kRows = 3;
  const int per_warp = (n1 + kCWarps - 1) / kCWarps;
  const int q_end = min(n1, (warp + 1) * per_warp);
  bool scales_in = false;
  for (int qb = warp * per_warp; qb < q_end;) {
    int s = 0;
    while (s + 1 < tb.nseg1 && tb.sq0[s + 1] <= qb) ++s;
    int pa = 0;
    while (pa + 1 < tb.npieces && tb.pq0[pa + 1] <= qb) ++pa;
    // rows of one segment, inside piece pa and the next piece
    int room = tb.pq0[pa] + tb.pn[pa] - qb;
    if (pa + 1 < tb.npieces && tb.pseg[pa + 1] == s) room += tb.pn[pa + 1];
    const int nr = min(min(kRows, room), min(q_end, tb.sq0[s] + tb.sn[s]) - qb);
    const int pb = qb + nr - 1 < tb.pq0[pa] + tb.pn[pa] ? pa : pa + 1;
    const int p = tb.sp[s], t = p / a.k;
    bool ok = tb.recs[p] != nullptr;
    if (ok && !scales_in) ok = scales_in = await(&bars[kBarScales], ph, tb, a, kSiteScales, L);
    if (ok) ok = await(&bars[pa], ph, tb, a, kSitePiece, L);
    if (ok && pb != pa) ok = await(&bars[pb], ph, tb, a, kSitePiece, L);
    float gs[kRows], us[kRows];
    uint32_t goff[kRows], uoff[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      gs[r] = 0.f;
      us[r] = 0.f;
      const int q = qb + min(r, nr - 1);
      const int pi = q < tb.pq0[pa] + tb.pn[pa] ? pa : pb;
      goff[r] = tb.poff[pi] + (uint32_t)(q - tb.pq0[pi]) * (uint32_t)(a.H / 2);
      uoff[r] = goff[r] + (uint32_t)tb.pn[pi] * (uint32_t)(a.H / 2);
    }
    if (ok) {
      const uint8_t* gsr = scales1 + tb.gwo[s] + (size_t)(qb - tb.sq0[s]) * (a.H / G);
      const uint8_t* usr = scales1 + tb.uwo[s] + (size_t)(qb - tb.sq0[s]) * (a.H / G);
      const uint4* xt = act + (size_t)t * 4 * upr;
      auto unit = [&](int u) {  // unit u of every row of the batch: gate units, then up units
        const bool is_up = u >= upr;
        const int cix = is_up ? u - upr : u;
        uint4 xv[4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) xv[wi] = xt[wi * upr + cix];
        const uint8_t* sb = (is_up ? usr : gsr) + sstep * cix;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (r < nr) {
            const uint4 qv = *reinterpret_cast<const uint4*>(codes1 + (is_up ? uoff[r] : goff[r]) + 16 * cix);
            const float d = dm::unit_dot_hx<FMT>(qv, dm::scale_bits<FMT>(sb + (size_t)r * (a.H / G)), xv);
            if (is_up) us[r] += d;
            else gs[r] += d;
          }
        }
      };
      if constexpr (UPR > 0) {
#pragma unroll
        for (int m = 0; m < (2 * UPR + 31) / 32; ++m) {
          const int u = lane + 32 * m;
          if (u < 2 * UPR) unit(u);
        }
      } else {
        for (int u = lane; u < 2 * upr; u += 32) unit(u);
      }
    }
    const float ts = tb.tsc[t];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        gs[r] += __shfl_xor_sync(0xffffffffu, gs[r], d);
        us[r] += __shfl_xor_sync(0xffffffffu, us[r], d);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (r < nr) {
          const float gv = gs[r] * ts, uv = us[r] * ts;
          a.hws[(size_t)p * a.I + tb.si0[s] + (qb + r - tb.sq0[s])] =
              ok ? gv / (1.0f + expf(-gv)) * uv : __uint_as_float(0x7FC00000u);
        }
      }
    }
    qb += nr;
  }
  }
  // h's barrier (a release arrival publishes the h rows written above); every
  // warp is also done with x in the x/h region before h is staged there
  tc::named_sync(1, kCThreads);
  if (threadIdx.x == 0) grid_sync_thread(bar_target(fused ? 2u : 1u), tb, a, kSiteGrid2, L);
  tc::named_sync(1, kCThreads);

  // h of the pairs of the CTA's tokens, FP32, staged as 4 quads of 8 floats
  // per 32-element unit: element i of local pair lp at
  // lp * hstride + (((i & 31) >> 3) * I/32 + (i >> 5)) * 8 + (i & 7)
  const int d0 = share_lo(blockIdx.x, (int)g.D, g.grid), d1 = share_lo(blockIdx.x + 1, (int)g.D, g.grid);
  const int nz = d1 - d0;
  const int t_lo = nz > 0 ? tb.dt[0] : 0;
  const int nlp = nz > 0 ? (tb.dt[tb.nseg2 - 1] - t_lo + 1) * a.k : 0;
  float* hs = reinterpret_cast<float*>(act);
  if (*abort_flag == 0) {
    const int n8 = nlp * (a.I / 8);
    const float4* src = reinterpret_cast<const float4*>(a.hws + (size_t)t_lo * a.k * a.I);
    constexpr int kB = 4;
    for (int b0 = threadIdx.x; b0 < n8; b0 += kB * kCThreads) {
      float4 v[kB][2];
#pragma unroll
      for (int m = 0; m < kB; ++m) {
        const int e8 = b0 + m * kCThreads;
        if (e8 < n8) {
          v[m][0] = __ldcg(src + 2 * e8);
          v[m][1] = __ldcg(src + 2 * e8 + 1);
        }
      }
#pragma unroll
      for (int m = 0; m < kB; ++m) {
        const int e8 = b0 + m * kCThreads;
        if (e8 < n8) {
          const int lp = e8 / (a.I / 8), i = (e8 - lp * (a.I / 8)) * 8;
          float* dst = hs + (size_t)lp * g.hstride + (((i & 31) >> 3) * updr + (i >> 5)) * 8;
          *reinterpret_cast<float4*>(dst) = v[m][0];
          *reinterpret_cast<float4*>(dst + 4) = v[m][1];
        }
      }
    }
  }
  tc::named_sync(1, kCThreads);

  // down: task (row z, expert j) -> a group of NG lanes (NG a power of two),
  // lane sub of the group taking units sub, sub + NG, ...; the group's sum is
  // reduced over its lanes in a fixed order and, times the router weight,
  // kept per (row, expert).  32 / NG tasks per warp pass, passes round-robin.
  constexpr int kUnitsPerLane = 5;
  int NG = 1;
  while (NG < 32 && NG * kUnitsPerLane < updr) NG <<= 1;
  const int tasks_per_pass = 32 / NG;
  const int ntask = nz * a.k;
  const int npass = (ntask + tasks_per_pass - 1) / tasks_per_pass;
  // set only before the barrier above, so every thread reads the same
  const bool have_h = *abort_flag == 0;
  const bool down_in = have_h && nz > 0 && await(&bars[kBarDown], ph, tb, a, kSiteDown, L);
  const int sub = lane & (NG - 1);
  float* part = reinterpret_cast<float*>(smem + g.off_part);  // [row][expert]
  for (int ps = warp; ps < npass; ps += kCWarps) {
    const int task = ps * tasks_per_pass + lane / NG;
    float v = 0.f;
    int z = 0, j = 0, s = 0, p = 0;
    if (task < ntask) {
      z = task / a.k;
      j = task - z * a.k;
      while (s + 1 < tb.nseg2 && tb.dz0[s + 1] <= z) ++s;
      p = tb.dt[s] * a.k + j;
      if (!down_in || !tb.recs[p]) {
        v = __uint_as_float(0x7FC00000u);
      } else {
        const int zr = z - tb.dz0[s];
        const uint8_t* crow = codes2 + ((size_t)tb.dz0[s] * a.k + (size_t)j * tb.dn[s] + zr) * (a.I / 2);
        const uint8_t* srow = scales2 + tb.dso[s][j] + (size_t)zr * (a.I / G);
        const float* hq = hs + (size_t)((tb.dt[s] - t_lo) * a.k + j) * g.hstride;
        if constexpr (UPDR > 0) {
          constexpr int kL = [] { int l = 1; while (l < 32 && l * kUnitsPerLane < UPDR) l <<= 1; return l; }();
#pragma unroll
          for (int m = 0; m < (UPDR + kL - 1) / kL; ++m) {
            const int u = sub + kL * m;
            if (u < UPDR)
              v += dm::unit_dot_f32<FMT>(*reinterpret_cast<const uint4*>(crow + 16 * u),
                                         dm::scale_bits<FMT>(srow + sstep * u), hq + 8 * u, 8 * UPDR);
          }
        } else {
          for (int u = sub; u < updr; u += NG)
            v += dm::unit_dot_f32<FMT>(*reinterpret_cast<const uint4*>(crow + 16 * u),
                                       dm::scale_bits<FMT>(srow + sstep * u), hq + 8 * u, 8 * updr);
        }
      }
    }
    for (int d = NG >> 1; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if (task < ntask && sub == 0) part[task] = tb.wts[p] * v;
  }
  tc::named_sync(1, kCThreads);
  // each output row: its k weighted expert outputs in expert order
  const bool failed = *abort_flag != 0;
  for (int z = threadIdx.x; z < nz; z += kCThreads) {
    float v = 0.f;
    for (int jj = 0; jj < a.k; ++jj) v += part[(size_t)z * a.k + jj];
    a.y[d0 + z] = failed ? __uint_as_float(0x7FC00000u) : v;
  }
  }  // compute warps
  if (L + 1 < nl) {
    // The next layer's router rows go into the x/h region, by bulk copies
    // (the async proxy) after this layer's ordinary stores there: every
    // thread orders its own stores before them, then the CTA-wide barrier.
    tc::fence_proxy_async();
    __syncthreads();  // end of layer L: y written, every shared buffer free again
    if (threadIdx.x == 0) {
      // this layer's arrival publishes y; the next layer's router rows are
      // fetched while the barrier completes, once the router barrier's phase
      // of this layer has completed (a flagged launch stages nothing more)
      grid_sync_thread(bar_target(nb), tb, a, kSiteLayer, L, [&] {
        if (!rstaged || *abort_flag) return;
        if (tc::mbar_wait_backoff(&bars[kBarRouter], ph, tc::globaltimer() + a.wait_ns)) {
          stage_router(a, smem, &bars[kBarRouter], L + 1);
        } else {
          *abort_flag = 1;
          status_or(a.status, MOE_DEV_TIMEOUT);
          note_timeout(a.bar, kSiteRouter, L);
        }
      });
    }
    if (threadIdx.x < kMaxPairs) tb.amax[threadIdx.x] = 0u;
    __syncthreads();
  }
  }  // layers
  // every barrier's arrival, also those a flagged launch skipped (and the
  // barrier after the last layer, which a whole-stack launch does not wait
  // for), so that the counter stays a multiple of the grid between launches
  if (threadIdx.x == 0) {
    const Tab& tb = *reinterpret_cast<const Tab*>(smem + a.geo.off_tab);
    const unsigned nb = (a.wr ? 2u : 1u) + (STACK ? 1u : 0u);
    const unsigned long long rest = (unsigned long long)nb * (unsigned long long)nl - (unsigned long long)tb.arrived;
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(a.bar), "l"(rest) : "memory");
  }
}

template <int FMT, int UPR, int UPDR, bool STACK>
int launch_shape(const DecodeOneshotArgs& a, int grid, size_t smem, cudaStream_t stream) {
  static SmemGrant granted;  // per device; also checks that one CTA fits on an SM
  if (!grant_smem(oneshot_kernel<FMT, UPR, UPDR, STACK>, smem, granted, kThreads)) return MOE_ERR_CUDA;
  // Every CTA takes part in the grid barriers, so all must be resident: one
  // CTA per SM, checked by grant_smem above.  A cooperative launch would make
  // the driver guarantee it, but costs about 2.5 us more host time per launch
  // (48 eager launches per decoded token), so the waits are bounded instead.
  return launch_pdl(oneshot_kernel<FMT, UPR, UPDR, STACK>, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int FMT>
int launch_fmt(const DecodeOneshotArgs& a, int grid, cudaStream_t stream) {
  DecodeOneshotArgs b = a;
  b.geo = make_geo(a.T, a.k, a.H, a.I, FMT == MOE_FMT_NVFP4 ? 16 : 32, grid, a.wr != nullptr, a.E);
  // the row strides are compile-time constants for the decode model shape
  const bool stack = a.layers > 1;
  if (a.H == 2560 && a.I == 640)
    return stack ? launch_shape<FMT, 80, 20, true>(b, grid, b.geo.total, stream)
                 : launch_shape<FMT, 80, 20, false>(b, grid, b.geo.total, stream);
  return stack ? launch_shape<FMT, 0, 0, true>(b, grid, b.geo.total, stream)
               : launch_shape<FMT, 0, 0, false>(b, grid, b.geo.total, stream);
}

}  // namespace os
}  // namespace moe

namespace {
// Test hooks of the bounded waits (moe_test_set_wait_limit): 0 = defaults.
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<unsigned> g_barrier_extra{0};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
}  // namespace

int launch_decode_oneshot(const DecodeOneshotArgs& a0, int fmt, int grid, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  DecodeOneshotArgs a = a0;
  const unsigned long long w = g_wait_ns.load(std::memory_order_relaxed);
  a.wait_ns = w ? w : kDefaultWaitNs;
  a.barrier_extra = g_barrier_extra.load(std::memory_order_relaxed);
  return fmt == MOE_FMT_NVFP4 ? moe::os::launch_fmt<MOE_FMT_NVFP4>(a, grid, st)
                              : moe::os::launch_fmt<MOE_FMT_MXFP4>(a, grid, st);
}

extern "C" int moe_test_set_wait_limit(unsigned long long wait_ns, int barrier_extra_arrivals) {
  if (barrier_extra_arrivals < 0 || barrier_extra_arrivals > 1) return MOE_ERR_INVALID_ARG;
  if (wait_ns != 0 && (wait_ns < 1000ull || wait_ns > 10000000000ull)) return MOE_ERR_INVALID_ARG;
  g_wait_ns.store(wait_ns, std::memory_order_relaxed);
  g_barrier_extra.store((unsigned)barrier_extra_arrivals, std::memory_order_relaxed);
  return MOE_OK;
}
