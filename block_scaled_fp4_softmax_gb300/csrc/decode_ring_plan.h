// Chunk plan of the ring decode kernel (stream_kernel in decode.cu): which
// rows each chunk of a CTA's share carries.  Host and device code, so the
// plan can be checked on the CPU (tests/ring_plan_check.cu).
#pragma once

#include <cstddef>
#include <cstdint>

namespace moe {
namespace ring {

__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }

// First row of CTA b's share when R rows are split over `grid` CTAs (CTA b
// takes [share_at(b), share_at(b + 1))).
__host__ __device__ inline int share_at(long long b, long long grid, long long R) { return (int)(b * R / grid); }

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

// Host and device agree on the chunk plan.  A gate/up chunk is up to kRG
// consecutive row pairs of one routed pair (gate rows | up rows | gate scale
// window | up scale window); a down chunk is up to kRD consecutive output
// rows of one token for experts [j0, j0 + jn) (per expert: rows of codes |
// scale window).  A bulk copy carries several rows, so each of the few copies
// an SM keeps in flight moves kilobytes rather than one row and a sliver of
// scales.  The slot holds the larger of a gate/up chunk and one expert's down
// part; jn experts' down parts fill it.
constexpr int kRG = 4;  // row pairs per gate/up chunk
constexpr int kRD = 4;  // output rows per down chunk
static_assert(kRG == kRD, "a slot's empty barrier counts one arrival per row of either kind of chunk");
__host__ __device__ inline int gu_scale_room(int H, int G) { return (kRG * (H / G) + 64 + 15) & ~15; }
__host__ __device__ inline int dn_part_bytes(int I, int G) { return kRD * (I / 2) + ((kRD * (I / G) + 32 + 15) & ~15); }
__host__ __device__ inline int plan_slot_bytes(int H, int I, int G) {
  const int p1 = 2 * kRG * (H / 2) + 2 * gu_scale_room(H, G);
  const int p2 = dn_part_bytes(I, G);
  const int s = p1 > p2 ? p1 : p2;
  return (s + 127) & ~127;
}
__host__ __device__ inline int plan_jn(int k, int I, int G, int slot_bytes) {
  const int j = slot_bytes / dn_part_bytes(I, G);
  return j < 1 ? 1 : (j > k ? k : j);
}

// Gate/up chunk c of the CTA's row range [r0, r1) (row r = p * I + i): rows
// [rs, rs + nr), rs = r0 + kRG c.  As kRG <= I it crosses at most one pair
// boundary: piece 0 is rows [i0, i0 + n0) of pair p0, piece 1 (nr - n0 rows,
// possibly none) rows from 0 of pair p0 + 1.  O(1), 32-bit.
struct GuChunk {
  int rs, nr, p0, i0, n0;
};
__host__ __device__ inline GuChunk gu_chunk(int c, int r0, int r1, int I) {
  GuChunk g;
  g.rs = r0 + c * kRG;
  g.nr = imin(kRG, r1 - g.rs);
  g.p0 = g.rs / I;
  g.i0 = g.rs - g.p0 * I;
  g.n0 = imin(g.nr, I - g.i0);
  return g;
}
__host__ __device__ inline int gu_chunks(int r0, int r1) { return (r1 - r0 + kRG - 1) / kRG; }
// Blocks of output rows of [q0, q1) (row q = t * H + n), split at token
// boundaries and into runs of at most kRD rows; a CTA's rows span few tokens.
__host__ __device__ inline bool dn_block(int b, int q0, int q1, int H, int& qs, int& nd) {
  int q = q0;
  while (q < q1) {
    const int seg_end = imin(q1, (q / H + 1) * H);
    const int n = (seg_end - q + kRD - 1) / kRD;
    if (b < n) {
      qs = q + b * kRD;
      nd = imin(kRD, seg_end - qs);
      return true;
    }
    b -= n;
    q = seg_end;
  }
  return false;
}
__host__ __device__ inline int dn_blocks(int q0, int q1, int H) {
  int n = 0;
  for (int q = q0; q < q1;) {
    const int seg_end = imin(q1, (q / H + 1) * H);
    n += (seg_end - q + kRD - 1) / kRD;
    q = seg_end;
  }
  return n;
}

}  // namespace ring
}  // namespace moe
