// One-shot decode expert pass (T*k <= 64 pairs whose per-CTA share of the
// selected records fits in shared memory), one launch per MoE layer
// ("Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe", section "The engine", item 4: the single-token NVFP4
// SwiGLU expert kernel; the sum over the k experts weighted by the
// renormalised router probabilities).
//
//  1. Prologue.  Warp 15 reads the routed records and issues every TMA bulk
//     copy of this CTA's share at once; warps 0-14 stage x as FP16 (scaled per
//     token by a power of two, which is exact).
//  2. gate/up + SwiGLU: row pair q of the CTA -> warp q % 15, as soon as its
//     piece has landed; h = silu(g) * u goes to global scratch.
//  3. Grid barrier (one arrival on a counter that only grows).
//  4. down: h of the CTA's down pairs staged as FP16 hi + lo (scaled per pair
//     by a power of two); the units (16 code bytes) of the CTA's down rows
//     are cut into 32-unit slices, slice s -> warp s % 15, one unit per lane,
//     and a segmented scan leaves one partial per (row, slice); each row's
//     partials are added in order and the row's weighted output goes to
//     global scratch.
//  5. Combine: per block of output rows, the CTA whose contribution completes
//     the block (counted with one atomic per block) adds the k weighted
//     expert outputs in expert order and writes y.  Every sum has a fixed
//     order, so y is bit-reproducible.
#include <algorithm>

#include "common.cuh"
#include "decode_math.cuh"
#include "decode_oneshot.h"
#include "tcgen05.cuh"

namespace moe {
namespace os {

constexpr uint64_t kWaitNs = 2000000000ull;

struct Tab {
  const uint8_t* recs[kMaxPairs];
  float wts[kMaxPairs];
  float tsc[kMaxPairs];      // per token: 2^-e of the FP16 scale of x
  unsigned amax[kMaxPairs];  // max |.| as float bits (x per token, then h per segment)
  float pw[kMaxSegs];        // per down segment: router weight * 2^-e of the FP16 scale of h
  int flags[4];              // [0] abort, [1] grid barrier passed
  int npieces, nseg1, nseg2, nlast;
  int pq0[kMaxPieces], pn[kMaxPieces], pseg[kMaxPieces];
  uint32_t poff[kMaxPieces];  // piece: gate rows at codes1 + poff, up rows right after
  int sp[kMaxSegs], si0[kMaxSegs], sq0[kMaxSegs], sn[kMaxSegs];
  uint32_t gwo[kMaxSegs], uwo[kMaxSegs];  // first gate / up scale byte of the segment in scales1
  int dp[kMaxSegs], dn0[kMaxSegs], dz0[kMaxSegs], dn[kMaxSegs];
  uint32_t dso[kMaxSegs];                 // first down scale byte of the segment in scales2
  int last[2 * kMaxSegs * 4];             // (token, block) pairs this CTA combines
};
static_assert(sizeof(Tab) <= 4096, "table region");

struct Win {  // 16-byte aligned window [lo, lo + bytes) around a byte range
  size_t lo;
  uint32_t bytes, delta;
};
__host__ __device__ inline Win window(size_t start, size_t len) {
  Win w;
  w.lo = start & ~(size_t)15;
  const size_t hi = (start + len + 15) & ~(size_t)15;
  w.bytes = (uint32_t)(hi - w.lo);
  w.delta = (uint32_t)(start - w.lo);
  return w;
}

// Fills the piece and segment tables of CTA b (no data dependence: runs
// before the wait for the previous kernel).
__device__ void build_tables(const Geo& g, int b, const RecordOffsets& o, Tab& tb) {
  const long long r0 = (long long)b * g.R1 / g.grid, r1 = (long long)(b + 1) * g.R1 / g.grid;
  int np = 0, ns = 0;
  uint32_t coff = 0, soff = 0;
  for (long long r = r0; r < r1 && ns < kMaxSegs;) {
    const int p = (int)(r / g.I), i0 = (int)(r - (long long)p * g.I);
    const int n = (int)min(r1 - r, (long long)(g.I - i0));
    const int q0 = (int)(r - r0);
    tb.sp[ns] = p;
    tb.si0[ns] = i0;
    tb.sq0[ns] = q0;
    tb.sn[ns] = n;
    const Win gw = window(o.gate_s + (size_t)i0 * (g.H / g.G), (size_t)n * (g.H / g.G));
    tb.gwo[ns] = soff + gw.delta;
    soff += gw.bytes;
    const Win uw = window(o.up_s + (size_t)i0 * (g.H / g.G), (size_t)n * (g.H / g.G));
    tb.uwo[ns] = soff + uw.delta;
    soff += uw.bytes;
    for (int a = 0; a < n && np < kMaxPieces; a += g.np) {
      const int m = min(g.np, n - a);
      tb.pq0[np] = q0 + a;
      tb.pn[np] = m;
      tb.pseg[np] = ns;
      tb.poff[np] = coff;
      coff += (uint32_t)m * g.H;
      ++np;
    }
    ++ns;
    r += n;
  }
  tb.npieces = np;
  tb.nseg1 = ns;
  const long long d0 = (long long)b * g.D / g.grid, d1 = (long long)(b + 1) * g.D / g.grid;
  ns = 0;
  soff = 0;
  for (long long d = d0; d < d1 && ns < kMaxSegs;) {
    const int p = (int)(d / g.H), n0 = (int)(d - (long long)p * g.H);
    const int n = (int)min(d1 - d, (long long)(g.H - n0));
    tb.dp[ns] = p;
    tb.dn0[ns] = n0;
    tb.dz0[ns] = (int)(d - d0);
    tb.dn[ns] = n;
    const Win dw = window(o.down_s + (size_t)n0 * (g.I / g.G), (size_t)n * (g.I / g.G));
    tb.dso[ns] = soff + dw.delta;
    soff += dw.bytes;
    ++ns;
    d += n;
  }
  tb.nseg2 = ns;
  tb.nlast = 0;
  tb.flags[0] = 0;
  tb.flags[1] = 0;
}

// Lane 0 of warp 15: every copy of this CTA's share.  Barriers: [0, npieces)
// one per gate/up piece, kMaxPieces the gate/up scale windows, kMaxPieces + 1
// the down rows and their scale windows.  Each barrier completes once per
// launch (parity 0).
__device__ void issue_copies(const Geo& g, const RecordOffsets& o, const Tab& tb, uint8_t* smem,
                             uint64_t* bars) {
  const uint32_t s1 = tc::smem_u32(smem + g.off_scales1), c1 = tc::smem_u32(smem + g.off_codes1);
  const uint32_t s2 = tc::smem_u32(smem + g.off_scales2), c2 = tc::smem_u32(smem + g.off_codes2);
  const size_t gsb = (size_t)(g.H / g.G), dsb = (size_t)(g.I / g.G);
  // gate/up scale windows first: small, and needed by the first piece
  uint32_t tx = 0;
  for (int s = 0; s < tb.nseg1; ++s)
    if (tb.recs[tb.sp[s]]) {
      tx += window(o.gate_s + (size_t)tb.si0[s] * gsb, (size_t)tb.sn[s] * gsb).bytes;
      tx += window(o.up_s + (size_t)tb.si0[s] * gsb, (size_t)tb.sn[s] * gsb).bytes;
    }
  tc::mbar_arrive_expect_tx(&bars[kMaxPieces], tx);
  for (int s = 0; s < tb.nseg1; ++s) {
    const uint8_t* rec = tb.recs[tb.sp[s]];
    if (!rec) continue;
    const Win gw = window(o.gate_s + (size_t)tb.si0[s] * gsb, (size_t)tb.sn[s] * gsb);
    const Win uw = window(o.up_s + (size_t)tb.si0[s] * gsb, (size_t)tb.sn[s] * gsb);
    tc::bulk_g2s(s1 + tb.gwo[s] - gw.delta, rec + gw.lo, gw.bytes, &bars[kMaxPieces]);
    tc::bulk_g2s(s1 + tb.uwo[s] - uw.delta, rec + uw.lo, uw.bytes, &bars[kMaxPieces]);
  }
  // gate/up code pieces, in row order
  const uint32_t rb = (uint32_t)(g.H / 2);
  for (int pi = 0; pi < tb.npieces; ++pi) {
    const int s = tb.pseg[pi];
    const uint8_t* rec = tb.recs[tb.sp[s]];
    const uint32_t bytes = (uint32_t)tb.pn[pi] * rb;
    tc::mbar_arrive_expect_tx(&bars[pi], rec ? 2 * bytes : 0);
    if (!rec) continue;
    const size_t i = (size_t)tb.si0[s] + (tb.pq0[pi] - tb.sq0[s]);
    tc::bulk_g2s(c1 + tb.poff[pi], rec + o.gate + i * rb, bytes, &bars[pi]);
    tc::bulk_g2s(c1 + tb.poff[pi] + bytes, rec + o.up + i * rb, bytes, &bars[pi]);
  }
  // down rows and scale windows
  const uint32_t drb = (uint32_t)(g.I / 2);
  tx = 0;
  for (int s = 0; s < tb.nseg2; ++s)
    if (tb.recs[tb.dp[s]])
      tx += (uint32_t)tb.dn[s] * drb + window(o.down_s + (size_t)tb.dn0[s] * dsb, (size_t)tb.dn[s] * dsb).bytes;
  tc::mbar_arrive_expect_tx(&bars[kMaxPieces + 1], tx);
  const int rows_per_copy = (int)(kMaxCopy / drb);
  for (int s = 0; s < tb.nseg2; ++s) {
    const uint8_t* rec = tb.recs[tb.dp[s]];
    if (!rec) continue;
    for (int a = 0; a < tb.dn[s]; a += rows_per_copy) {
      const int m = min(rows_per_copy, tb.dn[s] - a);
      tc::bulk_g2s(c2 + (uint32_t)(tb.dz0[s] + a) * drb, rec + o.down + (size_t)(tb.dn0[s] + a) * drb,
                   (uint32_t)m * drb, &bars[kMaxPieces + 1]);
    }
    const Win dw = window(o.down_s + (size_t)tb.dn0[s] * dsb, (size_t)tb.dn[s] * dsb);
    tc::bulk_g2s(s2 + tb.dso[s] - dw.delta, rec + dw.lo, dw.bytes, &bars[kMaxPieces + 1]);
  }
}

// Waits (bounded) for one barrier's parity-0 phase; on timeout flags the
// launch and returns false.
__device__ __forceinline__ bool await(uint64_t* bar, Tab& tb, int32_t* status) {
  volatile int* abort_flag = tb.flags;
  if (*abort_flag) return false;
  if (tc::mbar_wait(bar, 0, tc::globaltimer() + kWaitNs)) return true;
  *abort_flag = 1;
  status_or(status, MOE_DEV_TIMEOUT);
  return false;
}

template <int FMT, int UPR, int UPDR>
__global__ void __launch_bounds__(kThreads, 1) oneshot_kernel(DecodeOneshotArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_launch_dependents();
  constexpr int G = FMT == MOE_FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = FMT == MOE_FMT_NVFP4 ? 2 : 1;
  const Geo g = make_geo(a.T, a.k, a.H, a.I, G, gridDim.x);
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
  float* part = reinterpret_cast<float*>(smem + g.off_part);
  volatile int* abort_flag = tb.flags;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxPieces + 2; ++i) tc::mbar_init(&bars[i], 1);
    tc::mbar_fence_init();
  }
  if (threadIdx.x == 32) build_tables(g, blockIdx.x, o, tb);
  if (threadIdx.x < kMaxPairs) tb.amax[threadIdx.x] = 0u;
  // the pointer table does not depend on the previous kernel: warm L2 with it
  for (int i = threadIdx.x; i < (a.E * 8 + 127) / 128; i += kThreads)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(a.ptrs) + (size_t)i * 128));
  __syncthreads();
  pdl_wait();

  if (warp == kCWarps) {
    // ------------------------------------------------------------ loader
    for (int p = lane; p < P; p += 32) {
      tb.recs[p] = dm::checked_record(a.idx[p], a.E, a.ptrs, blockIdx.x == 0 ? a.status : nullptr);
      tb.wts[p] = a.w[p];
    }
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");  // records are in place
    if (lane == 0) {
      issue_copies(g, o, tb, smem, bars);
      // no copy may still be in flight when the CTA exits
      const uint64_t dl = tc::globaltimer() + kWaitNs;
      for (int i = 0; i < tb.npieces; ++i) tc::mbar_wait_backoff(&bars[i], 0, dl);
      tc::mbar_wait_backoff(&bars[kMaxPieces], 0, dl);
      tc::mbar_wait_backoff(&bars[kMaxPieces + 1], 0, dl);
    }
    __syncthreads();
    return;
  }

  // ---------------------------------------------------------------- compute
  // x: per-token max |x| (pass 1), then FP16 quads [t][4][H/32] of x * 2^e
  // (exact: BF16 has 8 significant bits and the scaled values lie in FP16's
  // normal range)
  const int nx8 = a.T * a.H / 8;
  const uint4* xg = reinterpret_cast<const uint4*>(a.x);
  uint4 xr = make_uint4(0u, 0u, 0u, 0u);
  for (int b = warp * 32; b < nx8; b += kCThreads) {
    const int q = b + lane;
    unsigned m = 0u;
    int key = -1;
    if (q < nx8) {
      const uint4 v = __ldg(xg + q);
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
      const uint4 v = b == warp * 32 ? xr : __ldg(xg + q);
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
  // amax served x; the down phase reuses it for h (ordered by the named
  // barriers below)
  if (threadIdx.x < kMaxPairs) tb.amax[threadIdx.x] = 0u;

  // gate/up + SwiGLU: row pair q of this CTA -> warp q % 15
  const long long r0 = (long long)blockIdx.x * g.R1 / g.grid, r1 = (long long)(blockIdx.x + 1) * g.R1 / g.grid;
  const int n1 = (int)(r1 - r0);
  bool scales_in = false;
  for (int q = warp; q < n1; q += kCWarps) {
    int pi = 0;
    while (pi + 1 < tb.npieces && tb.pq0[pi + 1] <= q) ++pi;
    const int s = tb.pseg[pi];
    const int p = tb.sp[s], t = p / a.k;
    const uint8_t* rec = tb.recs[p];
    bool ok = rec != nullptr;
    if (ok && !scales_in) ok = scales_in = await(&bars[kMaxPieces], tb, a.status);
    if (ok) ok = await(&bars[pi], tb, a.status);
    float gs = 0.f, us = 0.f;
    if (ok) {
      const uint8_t* grow = codes1 + tb.poff[pi] + (size_t)(q - tb.pq0[pi]) * (a.H / 2);
      const uint8_t* urow = grow + (size_t)tb.pn[pi] * (a.H / 2);
      const uint8_t* gsr = scales1 + tb.gwo[s] + (size_t)(q - tb.sq0[s]) * (a.H / G);
      const uint8_t* usr = scales1 + tb.uwo[s] + (size_t)(q - tb.sq0[s]) * (a.H / G);
      const uint4* xt = act + (size_t)t * 4 * upr;
      if constexpr (UPR > 0) {
#pragma unroll
        for (int m = 0; m < (2 * UPR + 31) / 32; ++m) {
          const int u = lane + 32 * m;
          if (u < 2 * UPR) {
            const bool is_up = u >= UPR;
            const int cix = is_up ? u - UPR : u;
            const uint4 qv = *reinterpret_cast<const uint4*>((is_up ? urow : grow) + 16 * cix);
            const float d = dm::unit_dot_h<FMT, UPR>(
                qv, dm::scale_bits<FMT>((is_up ? usr : gsr) + sstep * cix), xt + cix, UPR);
            if (is_up) us += d;
            else gs += d;
          }
        }
      } else {
        for (int u = lane; u < 2 * upr; u += 32) {
          const bool is_up = u >= upr;
          const int cix = is_up ? u - upr : u;
          const uint4 qv = *reinterpret_cast<const uint4*>((is_up ? urow : grow) + 16 * cix);
          const float d = dm::unit_dot_h<FMT, 0>(
              qv, dm::scale_bits<FMT>((is_up ? usr : gsr) + sstep * cix), xt + cix, upr);
          if (is_up) us += d;
          else gs += d;
        }
      }
    }
    const float ts = tb.tsc[t];
    gs = warp_sum(gs) * ts;
    us = warp_sum(us) * ts;
    if (lane == 0)
      a.hws[(size_t)p * a.I + tb.si0[s] + (q - tb.sq0[s])] =
          ok ? gs / (1.0f + expf(-gs)) * us : __uint_as_float(0x7FC00000u);
  }
  __threadfence();

  // grid barrier among the compute threads of every CTA: one arrival on a
  // counter that only grows; this launch's CTAs wait for the next multiple of
  // the grid size
  tc::named_sync(1, kCThreads);
  if (threadIdx.x == 0) {
    int good = !*abort_flag;
    if (good) {
      unsigned long long old;
      asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(a.bar) : "memory");
      const unsigned long long target = (old / gridDim.x + 1) * gridDim.x;
      const uint64_t dl = global_ns() + kWaitNs;
      while (dm::ld_acquire_u64(a.bar) < target) {
        if (global_ns() > dl) {
          good = 0;
          break;
        }
      }
    }
    if (!good) {
      *abort_flag = 1;
      status_or(a.status, MOE_DEV_TIMEOUT);
    }
    tb.flags[1] = good;
  }
  tc::named_sync(1, kCThreads);

  // h of the down segments' pairs: per-pair max |h| (pass 1), then FP16 hi +
  // lo quads [segment][4][I/32] of h * 2^e (pass 2); loads stay in registers
  // between the passes when one batch covers them
  const long long d0 = (long long)blockIdx.x * g.D / g.grid, d1 = (long long)(blockIdx.x + 1) * g.D / g.grid;
  const int nz = (int)(d1 - d0);
  uint4* hhi = act;
  uint4* hlo = act + (size_t)g.segs2 * 4 * updr;
  for (int i = threadIdx.x; i < nz * g.pieces2; i += kCThreads) part[i] = 0.f;
  const bool have_h = tb.flags[1] != 0;
  {
    const int n8 = tb.nseg2 * (a.I / 8);
    constexpr int kB = 4;
    const bool keep = n8 <= kB * kCThreads;
    float4 v[kB][2];
    auto load = [&](int b0) {
#pragma unroll
      for (int m = 0; m < kB; ++m) {
        const int e8 = b0 + m * kCThreads + lane;
        if (e8 < n8) {
          const int s = e8 / (a.I / 8), i = (e8 - s * (a.I / 8)) * 8;
          const float4* src = reinterpret_cast<const float4*>(a.hws + (size_t)tb.dp[s] * a.I + i);
          v[m][0] = __ldcg(src);
          v[m][1] = __ldcg(src + 1);
        }
      }
    };
    if (have_h) {
      for (int b0 = warp * 32; b0 < n8; b0 += kB * kCThreads) {
        load(b0);
#pragma unroll
        for (int m = 0; m < kB; ++m) {
          const int e8 = b0 + m * kCThreads + lane;
          unsigned mx = 0u;
          int key = -1;
          if (e8 < n8) {
            const float f[8] = {v[m][0].x, v[m][0].y, v[m][0].z, v[m][0].w,
                                v[m][1].x, v[m][1].y, v[m][1].z, v[m][1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) mx = max(mx, __float_as_uint(f[i]) & 0x7FFFFFFFu);
            key = e8 / (a.I / 8);
          }
          if (dm::group_max(key, mx)) atomicMax(&tb.amax[key], mx);
        }
      }
    }
    tc::named_sync(1, kCThreads);
    if (threadIdx.x < tb.nseg2)
      tb.pw[threadIdx.x] = tb.wts[tb.dp[threadIdx.x]] *
                           dm::pow2f(-dm::f16_shift(__uint_as_float(tb.amax[threadIdx.x])));
    if (have_h) {
      for (int b0 = warp * 32; b0 < n8; b0 += kB * kCThreads) {
        if (!keep) load(b0);
#pragma unroll
        for (int m = 0; m < kB; ++m) {
          const int e8 = b0 + m * kCThreads + lane;
          if (e8 < n8) {
            const int s = e8 / (a.I / 8), i = (e8 - s * (a.I / 8)) * 8;
            const float sc = dm::pow2f(dm::f16_shift(__uint_as_float(tb.amax[s])));
            const float f[8] = {v[m][0].x * sc, v[m][0].y * sc, v[m][0].z * sc, v[m][0].w * sc,
                                v[m][1].x * sc, v[m][1].y * sc, v[m][1].z * sc, v[m][1].w * sc};
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __half h0 = __float2half_rn(f[2 * e2]), h1 = __float2half_rn(f[2 * e2 + 1]);
              hv[e2] = dm::pack_h2(__half2float(h0), __half2float(h1));
              lv[e2] = dm::pack_h2(f[2 * e2] - __half2float(h0), f[2 * e2 + 1] - __half2float(h1));
            }
            const size_t at = (size_t)s * 4 * updr + ((i & 31) >> 3) * updr + (i >> 5);
            hhi[at] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            hlo[at] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
          }
        }
      }
    }
  }
  tc::named_sync(1, kCThreads);

  // down: 32-unit slices of the (row, unit) space of this CTA's down rows,
  // two slices per warp at a time; a segmented scan over the lanes of one row
  // leaves the row's partial for that slice
  const int NU = nz * updr;
  const int nsl = (NU + 31) / 32;
  const bool down_in = have_h && nsl > 0 && await(&bars[kMaxPieces + 1], tb, a.status);
  auto unit_value = [&](int U, int& z) -> float {
    if (U >= NU) {
      z = -1;
      return 0.f;
    }
    z = U / updr;
    const int u = U - z * updr;
    int s = 0;
    while (s + 1 < tb.nseg2 && tb.dz0[s + 1] <= z) ++s;
    if (!down_in || !tb.recs[tb.dp[s]]) return __uint_as_float(0x7FC00000u);
    const uint4 qv = *reinterpret_cast<const uint4*>(codes2 + (size_t)z * (a.I / 2) + 16 * u);
    const uint8_t* sp = scales2 + tb.dso[s] + (size_t)(z - tb.dz0[s]) * (a.I / G) + sstep * u;
    const size_t col = (size_t)s * 4 * updr + u;
    return dm::unit_dot_h2<FMT, UPDR>(qv, dm::scale_bits<FMT>(sp), hhi + col, hlo + col, updr);
  };
  auto store = [&](int sl, int z, float val) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float tv = __shfl_up_sync(0xffffffffu, val, d);
      const int tz = __shfl_up_sync(0xffffffffu, z, d);
      if (lane >= d && tz == z) val += tv;
    }
    const int zn = __shfl_down_sync(0xffffffffu, z, 1);
    if (z >= 0 && (lane == 31 || zn != z)) part[(size_t)z * g.pieces2 + sl - (z * updr) / 32] = val;
  };
  for (int sl = warp; sl < nsl; sl += 2 * kCWarps) {
    const int sl2 = sl + kCWarps;
    int za, zb;
    const float va = unit_value(sl * 32 + lane, za);
    const float vb = unit_value(sl2 < nsl ? sl2 * 32 + lane : NU, zb);
    store(sl, za, va);
    if (sl2 < nsl) store(sl2, zb, vb);
  }
  tc::named_sync(1, kCThreads);
  // each row: its partials in slice order, times the router weight
  for (int z = threadIdx.x; z < nz; z += kCThreads) {
    int s = 0;
    while (s + 1 < tb.nseg2 && tb.dz0[s + 1] <= z) ++s;
    float v = 0.f;
    for (int i = 0; i < g.pieces2; ++i) v += part[(size_t)z * g.pieces2 + i];
    a.part[(size_t)tb.dp[s] * a.H + tb.dn0[s] + (z - tb.dz0[s])] = *abort_flag ? __uint_as_float(0x7FC00000u)
                                                                                : tb.pw[s] * v;
  }
  __threadfence();
  tc::named_sync(1, kCThreads);
  // combine: count this CTA's rows into each block of output rows it touches;
  // the CTA that completes a block adds the block's k expert outputs
  if (threadIdx.x == 0) {
    int nl = 0;
    for (int s = 0; s < tb.nseg2; ++s) {
      const int t = tb.dp[s] / a.k, n0 = tb.dn0[s], n1 = n0 + tb.dn[s];
      for (int b = n0 / g.blk; b * g.blk < n1; ++b) {
        const int lo = max(n0, b * g.blk), hi = min(n1, (b + 1) * g.blk);
        const unsigned rows = (unsigned)(min(a.H, (b + 1) * g.blk) - b * g.blk);
        const unsigned target = (unsigned)a.k * rows;
        unsigned* c = a.cnt + (size_t)t * kBlkStride + b;
        const unsigned now = atomicAdd(c, (unsigned)(hi - lo)) + (unsigned)(hi - lo);
        if (now == target) {
          atomicExch(c, 0u);
          tb.last[nl++] = t * kBlkStride + b;
        } else if (now > target) {
          status_or(a.status, MOE_DEV_WORKSPACE);
        }
      }
    }
    tb.nlast = nl;
    __threadfence();
  }
  tc::named_sync(1, kCThreads);
  for (int l = 0; l < tb.nlast; ++l) {
    const int t = tb.last[l] / kBlkStride, b = tb.last[l] % kBlkStride;
    const int n_hi = min(a.H, (b + 1) * g.blk);
    for (int n = b * g.blk + threadIdx.x; n < n_hi; n += kCThreads) {
      float v = 0.f;
      for (int j = 0; j < a.k; ++j) v += __ldcg(a.part + (size_t)(t * a.k + j) * a.H + n);
      a.y[(size_t)t * a.H + n] = v;
    }
  }
  __syncthreads();
}

// Raises a kernel's dynamic shared-memory limit once per instantiation (the
// attribute call is not repeated, so later launches can be captured).
template <typename K>
bool grant_smem(K kernel, size_t bytes, size_t* granted) {
  if (bytes <= 48 * 1024 || bytes <= *granted) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return false;
  *granted = bytes;
  return true;
}

template <int FMT, int UPR, int UPDR>
int launch_shape(const DecodeOneshotArgs& a, int grid, size_t smem, cudaStream_t stream) {
  static size_t granted = 0;
  if (!grant_smem(oneshot_kernel<FMT, UPR, UPDR>, smem, &granted)) return MOE_ERR_CUDA;
  return launch_pdl(oneshot_kernel<FMT, UPR, UPDR>, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int FMT>
int launch_fmt(const DecodeOneshotArgs& a, int grid, cudaStream_t stream) {
  const Geo g = make_geo(a.T, a.k, a.H, a.I, FMT == MOE_FMT_NVFP4 ? 16 : 32, grid);
  // the row strides are compile-time constants for the decode model shape
  if (a.H == 2560 && a.I == 640) return launch_shape<FMT, 80, 20>(a, grid, g.total, stream);
  return launch_shape<FMT, 0, 0>(a, grid, g.total, stream);
}

}  // namespace os
}  // namespace moe

bool decode_oneshot_fits(int T, int k, int H, int I, int fmt, int grid, size_t smem_limit) {
  using namespace moe::os;
  if (grid <= 0 || T <= 0 || k <= 0 || (long long)T * k > kMaxPairs) return false;
  const Geo g = make_geo(T, k, H, I, fmt == MOE_FMT_NVFP4 ? 16 : 32, grid);
  if (g.total + 1024 > smem_limit) return false;
  if (g.segs1 > kMaxSegs || g.segs2 > kMaxSegs || max_pieces(g) > kMaxPieces) return false;
  if (g.nblk > kBlkStride) return false;
  // blocks one CTA can complete: those its down rows touch
  if (g.rows2 / g.blk + 2 * g.segs2 > (int)(sizeof(((Tab*)nullptr)->last) / sizeof(int))) return false;
  return true;
}

int launch_decode_oneshot(const DecodeOneshotArgs& a, int fmt, int grid, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  return fmt == MOE_FMT_NVFP4 ? moe::os::launch_fmt<MOE_FMT_NVFP4>(a, grid, st)
                              : moe::os::launch_fmt<MOE_FMT_MXFP4>(a, grid, st);
}
