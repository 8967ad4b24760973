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
  o += (size_t)g.rows1 * H;                       // gate + up codes
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

}  // namespace os
}  // namespace moe

// One-shot decode expert pass: true when the shape fits (the caller then
// launches it with launch_decode_oneshot).
bool decode_oneshot_fits(int T, int k, int H, int I, int fmt, int grid, size_t smem_limit,
                         bool fused = false, int E = 0);

struct DecodeOneshotArgs {
  const uint16_t* x;
  const int32_t* idx;
  const float* w;
  int T, k;
  const void* const* ptrs;
  int E, H, I;
  unsigned long long* bar;  // grid-barrier counter (workspace start)
  float* hws;               // [P][I] SwiGLU intermediate
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
};
int launch_decode_oneshot(const DecodeOneshotArgs& a, int fmt, int grid, void* stream);
