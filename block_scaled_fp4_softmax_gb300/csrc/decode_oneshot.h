// Plan of the one-shot decode expert pass (T*k <= 64, each CTA's share of the
// selected records fits in shared memory).  Host and device compute it with
// the same code.
//
// Work split over a grid of one CTA per SM:
//  - gate/up: the P*I row pairs (pair p = t*k + j, row i) in order, an equal
//    share per CTA; a share is cut into segments (one pair each) and the
//    segments into pieces of np rows;
//  - down: the T*H output rows (token t, row n) in order, an equal share per
//    CTA, with all k experts of each row, so every output row is finished by
//    one CTA; a share is cut into segments (one token each).
// Every byte of a CTA's share is requested with large TMA bulk copies at
// kernel entry (the copy engine of an SM completes only a few copies per
// microsecond, so few and large is what keeps HBM busy).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace os {

constexpr int kThreads = 512;  // warps 0-14 compute, warp 15 loads
constexpr int kCWarps = 15;
constexpr int kCThreads = kCWarps * 32;
constexpr int kMaxPairs = 64;
constexpr int kMaxPieces = 16;    // gate/up pieces of one CTA
constexpr int kMaxSegs = 4;       // segments of one CTA, per phase
constexpr int kMaxCopies = 96;    // bulk copies of one CTA
constexpr int kMaxK = 32;         // experts per token
constexpr int kPieceBytes = 16384;  // target bytes of one matrix in one piece
constexpr uint32_t kMaxCopy = 32768;
constexpr size_t kBarrierBytes = 256;  // grid-barrier counter
constexpr size_t kCounterBytes = 16384;  // reserved (kept so the workspace layout stays fixed)
constexpr size_t kHeaderBytes = kBarrierBytes + kCounterBytes;
constexpr int kLogitStride = 1024;  // tagged logits per token in the workspace (E <= 1024)

// The one-shot kernel's workspace after the header: tagged logits, then h
// [T*k][I] FP32.  The other decode paths keep their FP32 h right after the
// header.
__host__ __device__ inline size_t oneshot_ws_bytes(int T, int k, int I) {
  return kHeaderBytes + (size_t)T * kLogitStride * 8 + (size_t)T * k * I * 4;
}

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Geo {
  int T, k, H, I, G, grid;
  long long R1, D;    // gate/up row pairs, output rows
  int rows1, rows2;   // most rows of one CTA, per phase
  int segs1, segs2;   // most segments of one CTA, per phase
  int np;             // rows per gate/up piece
  int copies;         // most bulk copies of one CTA
  int hstride;        // floats per pair in the staged h (4 quads x I/32 units x 8, padded)
  int epc;            // router rows per CTA (fused launch)
  int rstage;         // bytes of router operands staged in the x/h region (0: read from global memory)
  // shared-memory regions (bytes from the start of dynamic shared memory)
  size_t off_bar, off_tab, off_codes1, off_scales1, off_codes2, off_scales2, off_act, off_part, off_xb, total;
};

// fused: the launch also runs the router over E experts (256 RMS partial
// sums, 512 top-k finalists and the BF16 x get a region of their own).  The
// CTA's router rows and the expert pointer table are staged in the x/h
// region, which they leave before x arrives there, when they fit in it.
__host__ __device__ inline Geo make_geo(int T, int k, int H, int I, int G, int grid, bool fused = false,
                                        int E = 0) {
  Geo g;
  g.T = T; g.k = k; g.H = H; g.I = I; g.G = G; g.grid = grid;
  g.epc = fused && E > 0 ? (E + grid - 1) / grid : 0;
  const long long P = (long long)T * k;
  g.R1 = P * I;
  g.D = (long long)T * H;
  g.rows1 = (int)((g.R1 + grid - 1) / grid);
  g.rows2 = (int)((g.D + grid - 1) / grid);
  const long long s1 = (g.rows1 - 1) / I + 2, s2 = (g.rows2 - 1) / H + 2;
  g.segs1 = (int)(s1 < P ? s1 : P);
  g.segs2 = (int)(s2 < T ? s2 : T);
  g.np = kPieceBytes / (H / 2);
  if (g.np < 1) g.np = 1;
  const int rows_per_copy = (int)(kMaxCopy / (I / 2));
  g.copies = 2 * ((g.rows1 + g.np - 1) / g.np + g.segs1) + 2 * g.segs1 +
             k * ((g.rows2 + rows_per_copy - 1) / rows_per_copy + 2 * g.segs2);
  g.hstride = 4 * (I / 32) * 8 + 4;
  size_t o = 0;
  g.off_bar = o;                                  // mbarriers: pieces, scales, down, router
  o += (kMaxPieces + 3) * 8;
  g.off_tab = o = round_up(o, 16);                // tables, weights, scales, flags
  o += 8192;
  g.off_codes1 = o = round_up(o, 128);
  // gate + up codes; a fused launch first stages one token's E logits here
  const size_t lg = fused ? (size_t)E * 4 : 0;
  o += (size_t)g.rows1 * H > lg ? (size_t)g.rows1 * H : lg;
  g.off_scales1 = o = round_up(o, 128);
  o += 2 * ((size_t)g.rows1 * (H / G) + 32 * (size_t)g.segs1);
  g.off_codes2 = o = round_up(o, 128);
  o += (size_t)g.rows2 * k * (I / 2);              // down codes, [segment][expert][row]
  g.off_scales2 = o = round_up(o, 128);
  o += (size_t)g.rows2 * k * (I / G) + 32 * (size_t)g.segs2 * k;
  g.off_act = o = round_up(o, 128);
  const size_t a1 = (size_t)T * H * 2, a2 = (size_t)g.segs2 * k * g.hstride * 4;
  const size_t act = a1 > a2 ? a1 : a2;
  const size_t rs = (size_t)g.epc * H * 2 + round_up((size_t)E * 8, 16);
  g.rstage = fused && E > 0 && rs <= act ? (int)rs : 0;
  o += act;                                       // router rows + pointers, then x (FP16), then h (FP32)
  g.off_part = o = round_up(o, 128);
  o += (size_t)g.rows2 * k * 4;                   // weighted expert outputs per row
  g.off_xb = o = round_up(o, 128);
  if (fused) o += 1024 + 4096 + (size_t)T * H * 2;  // RMS partial sums, top-k finalists, x (BF16)
  g.total = round_up(o, 128);
  return g;
}

// First unit of CTA b's equal share of n units over `grid` CTAs (32-bit:
// the plan only admits shapes with n * grid < 2^31).
__host__ __device__ inline int share_lo(int b, int n, int grid) {
  return (int)((unsigned)b * (unsigned)n / (unsigned)grid);
}

// Upper bound of the gate/up pieces of one CTA.
__host__ __device__ inline int max_pieces(const Geo& g) { return (g.rows1 + g.np - 1) / g.np + g.segs1; }

__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }

// Per-CTA tables in shared memory: the routed records and weights, the plan
// of pieces, segments and bulk copies, and a few flags.
struct Tab {
  const uint8_t* recs[kMaxPairs];
  float wts[kMaxPairs];
  float tsc[kMaxPairs];      // per token: 2^-e of the FP16 scale of x
  unsigned amax[kMaxPairs];  // max |x| of each token, as float bits
  int flags[4];              // [0] abort: a wait gave up (the launch writes NaN)
  unsigned long long bar_base;  // layer counter at launch start / grid (thread 0)
  int arrived;                  // layers this CTA has added to the counter (thread 0)
  int npieces, nseg1, nseg2, ncopies;
  int pq0[kMaxPieces], pn[kMaxPieces], pseg[kMaxPieces];
  uint32_t poff[kMaxPieces];  // piece: gate rows at codes1 + poff, up rows right after
  int sp[kMaxSegs], si0[kMaxSegs], sq0[kMaxSegs], sn[kMaxSegs];
  uint32_t gwo[kMaxSegs], uwo[kMaxSegs];  // first gate / up scale byte of the segment in scales1
  int dt[kMaxSegs], dn0[kMaxSegs], dz0[kMaxSegs], dn[kMaxSegs];  // down: token, rows
  uint32_t dso[kMaxSegs][kMaxK];          // first down scale byte of (segment, expert) in scales2
  // bulk copies: shared-memory destination (bytes from the dynamic base),
  // source offset in the record, bytes, barrier, pair
  uint64_t csrc[kMaxCopies];
  uint32_t cdst[kMaxCopies], cbytes[kMaxCopies];
  uint8_t cbar[kMaxCopies], cpair[kMaxCopies];
};
static_assert(sizeof(Tab) <= 8192, "table region");

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

// Barriers: [0, npieces) one per gate/up piece, kBarScales the gate/up scale
// windows, kBarDown the down rows and their scale windows (all completed by
// the loader warp's copies and its lane 0); kBarRouter the router rows and
// the pointer table of a fused launch (thread 0).  Each completes once per
// launch (parity 0).
constexpr int kBarScales = kMaxPieces, kBarDown = kMaxPieces + 1, kNumBars = kMaxPieces + 2;
constexpr int kBarRouter = kNumBars;

// Plans CTA b: pieces, segments and bulk copies.  Every gate/up piece gets
// two copies (gate rows, up rows); n_scale and n_down count the copies of
// the gate/up scale barrier and of the down barrier.  No data dependence:
// runs while the router does.  Writes the plan fields of the table only
// (never the flags, which the router may set meanwhile).
__host__ __device__ inline void build_tables(const Geo& g, int b, const RecordOffsets& o, Tab& tb, uint32_t& n_scale,
                             uint32_t& n_down) {
  int nc = 0;
  auto copy = [&](size_t dst, size_t src, uint32_t bytes, int bar, int pair) {
    tb.cdst[nc] = (uint32_t)dst;
    tb.csrc[nc] = src;
    tb.cbytes[nc] = bytes;
    tb.cbar[nc] = (uint8_t)bar;
    tb.cpair[nc] = (uint8_t)pair;
    ++nc;
  };
  n_scale = 0;
  n_down = 0;
  const size_t gsb = (size_t)(g.H / g.G), dsb = (size_t)(g.I / g.G), rb = (size_t)(g.H / 2), drb = (size_t)(g.I / 2);
  const int r0 = share_lo(b, (int)g.R1, g.grid), r1 = share_lo(b + 1, (int)g.R1, g.grid);
  int np = 0, ns = 0;
  uint32_t coff = 0, soff = 0;
  for (int r = r0; r < r1 && ns < kMaxSegs;) {
    const int p = r / g.I, i0 = r - p * g.I;
    const int n = imin(r1 - r, g.I - i0);
    const int q0 = (int)(r - r0);
    tb.sp[ns] = p;
    tb.si0[ns] = i0;
    tb.sq0[ns] = q0;
    tb.sn[ns] = n;
    const Win gw = window(o.gate_s + (size_t)i0 * gsb, (size_t)n * gsb);
    tb.gwo[ns] = soff + gw.delta;
    copy(g.off_scales1 + soff, gw.lo, gw.bytes, kBarScales, p);
    soff += gw.bytes;
    const Win uw = window(o.up_s + (size_t)i0 * gsb, (size_t)n * gsb);
    tb.uwo[ns] = soff + uw.delta;
    copy(g.off_scales1 + soff, uw.lo, uw.bytes, kBarScales, p);
    soff += uw.bytes;
    n_scale += 2;
    for (int a = 0; a < n && np < kMaxPieces; a += g.np) {
      const int m = imin(g.np, n - a);
      tb.pq0[np] = q0 + a;
      tb.pn[np] = m;
      tb.pseg[np] = ns;
      tb.poff[np] = coff;
      const uint32_t bytes = (uint32_t)(m * rb);
      copy(g.off_codes1 + coff, o.gate + (size_t)(i0 + a) * rb, bytes, np, p);
      copy(g.off_codes1 + coff + bytes, o.up + (size_t)(i0 + a) * rb, bytes, np, p);
      coff += 2 * bytes;
      ++np;
    }
    ++ns;
    r += n;
  }
  tb.npieces = np;
  tb.nseg1 = ns;
  const int d0 = share_lo(b, (int)g.D, g.grid), d1 = share_lo(b + 1, (int)g.D, g.grid);
  const int rows_per_copy = (int)(kMaxCopy / drb);
  ns = 0;
  soff = 0;
  for (int d = d0; d < d1 && ns < kMaxSegs;) {
    const int t = d / g.H, n0 = d - t * g.H;
    const int n = imin(d1 - d, g.H - n0);
    const int z0 = (int)(d - d0);
    tb.dt[ns] = t;
    tb.dn0[ns] = n0;
    tb.dz0[ns] = z0;
    tb.dn[ns] = n;
    // rows [n0, n0 + n) of every expert of token t: codes at
    // codes2 + (z0 * k + j * n) rows, then one scale window per expert
    for (int j = 0; j < g.k; ++j) {
      const int p = t * g.k + j;
      for (int a = 0; a < n; a += rows_per_copy) {
        const int m = imin(rows_per_copy, n - a);
        copy(g.off_codes2 + ((size_t)z0 * g.k + (size_t)j * n + a) * drb, o.down + (size_t)(n0 + a) * drb,
             (uint32_t)(m * drb), kBarDown, p);
        ++n_down;
      }
      const Win dw = window(o.down_s + (size_t)n0 * dsb, (size_t)n * dsb);
      tb.dso[ns][j] = soff + dw.delta;
      copy(g.off_scales2 + soff, dw.lo, dw.bytes, kBarDown, p);
      soff += dw.bytes;
      ++n_down;
    }
    ++ns;
    d += n;
  }
  tb.nseg2 = ns;
  tb.ncopies = nc;
}


}  // namespace os
}  // namespace moe

// One-shot decode expert pass: true when the shape fits (the caller then
// launches it with launch_decode_oneshot).
inline bool decode_oneshot_fits(int T, int k, int H, int I, int fmt, int grid, size_t smem_limit,
                               bool fused = false, int E = 0) {
  using namespace moe::os;
  if (grid <= 0 || T <= 0 || k <= 0 || (long long)T * k > kMaxPairs) return false;
  const Geo g = make_geo(T, k, H, I, fmt == MOE_FMT_NVFP4 ? 16 : 32, grid, fused, E);
  if (g.total + 1024 > smem_limit) return false;
  if (g.segs1 > kMaxSegs || g.segs2 > kMaxSegs || max_pieces(g) > kMaxPieces) return false;
  if (g.copies > kMaxCopies || k > kMaxK) return false;
  if (g.R1 * grid >= (1LL << 31) || g.D * grid >= (1LL << 31)) return false;  // 32-bit shares
  return true;
}

struct DecodeOneshotArgs {
  const uint16_t* x;
  const int32_t* idx;
  const float* w;
  int T, k;
  const void* const* ptrs;
  int E, H, I;
  unsigned long long* bar;  // layer counter (workspace start)
  // the logits exchanged between CTAs, [T][kLogitStride] tagged words (the
  // value's bits in the low 32, the layer's tag in the high 32)
  unsigned long long* xlog;
  float* hws;  // [P][I] SwiGLU intermediate
  float* y;
  int32_t* status;
  // router, when the launch runs the whole layer (wr != NULL): x = RMS
  // chaining of y_prev (or x itself when y_prev is NULL), written to x_out;
  // logits of all E experts; top-k written to idx_out / w_out
  const float* y_prev;
  float eps;
  uint16_t* x_out;
  const uint16_t* wr;
  const float* bias;
  float* logits;
  int32_t* idx_out;
  float* w_out;
  moe::os::Geo geo;  // the plan's geometry, computed by the host for the launch's grid
  // limit of every bounded wait (ns), and arrivals each grid barrier expects
  // beyond the grid (0; a test sets 1 to make the barriers run out)
  unsigned long long wait_ns;
  unsigned barrier_extra;
  // layers of a whole-layer launch (moe_decode_stack: wr, ptrs, bias, idx_out
  // and w_out hold one block per layer; layer 0 from x, the others chained
  // from y); 0 or 1 for one layer
  int layers;
};
// The counter, the tagged logits and h of a launch with T tokens in a
// workspace of at least moe::os::oneshot_ws_bytes(T, k, I) bytes.
inline void oneshot_set_workspace(DecodeOneshotArgs& oa, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  oa.bar = reinterpret_cast<unsigned long long*>(b);
  oa.xlog = reinterpret_cast<unsigned long long*>(b + moe::os::kHeaderBytes);
  oa.hws = reinterpret_cast<float*>(oa.xlog + (size_t)oa.T * moe::os::kLogitStride);
}

int launch_decode_oneshot(const DecodeOneshotArgs& a, int fmt, int grid, void* stream);
