// Host-side check of the one-shot decode plan (decode_oneshot.h): for many
// shapes and grid sizes, every CTA's plan is built on the CPU and checked
// against the rules the kernel and the copy engine rely on:
//  - every bulk copy starts and ends on 16-byte boundaries, in shared memory
//    and in the record, and stays inside its destination region and its
//    record; no two destinations overlap;
//  - the bytes a barrier expects stay below the mbarrier transaction limit,
//    and each barrier's arrival count matches its copies;
//  - the CTA's gate/up rows and down rows are covered exactly once, and every
//    code and scale byte the compute warps read was copied from the right
//    place of the right pair's record;
//  - the table limits (pieces, segments, copies) hold.
// Exit status 0 when every check passes.
#include <cstdio>
#include <vector>

#include "decode_oneshot.h"

using namespace moe;
using namespace moe::os;

static long long g_fail = 0, g_checks = 0;
#define CHECK(cond, ...)                                                        \
  do {                                                                          \
    ++g_checks;                                                                 \
    if (!(cond)) {                                                              \
      if (g_fail++ < 20) {                                                      \
        std::printf("FAIL line %d: ", __LINE__);                                \
        std::printf(__VA_ARGS__);                                               \
        std::printf("\n");                                                      \
      }                                                                         \
    }                                                                           \
  } while (0)

struct Shape {
  int T, k, H, I, fmt, E;
  bool fused;
};

// The copy that lands [dst, dst + len) in shared memory must come from
// [src, src + len) of pair p's record.
static bool covered(const Tab& tb, size_t dst, size_t len, size_t src, int p) {
  for (int c = 0; c < tb.ncopies; ++c) {
    if (tb.cpair[c] != p) continue;
    const size_t d0 = tb.cdst[c], d1 = d0 + tb.cbytes[c];
    if (dst >= d0 && dst + len <= d1) return tb.csrc[c] + (dst - d0) == src;
  }
  return false;
}

static void check_shape(const Shape& sh, int grid, size_t smem_limit) {
  const int G = sh.fmt == MOE_FMT_NVFP4 ? 16 : 32;
  const Geo g = make_geo(sh.T, sh.k, sh.H, sh.I, G, grid, sh.fused, sh.E);
  const RecordOffsets o = record_offsets(sh.H, sh.I, sh.fmt);
  const size_t regions[] = {g.off_bar, g.off_tab, g.off_codes1, g.off_scales1, g.off_codes2,
                            g.off_scales2, g.off_act, g.off_part, g.off_xb, g.total};
  for (int i = 0; i + 1 < 10; ++i) CHECK(regions[i] <= regions[i + 1], "regions out of order");
  for (int i = 2; i < 10; ++i) CHECK(regions[i] % 128 == 0, "region %d not 128-byte aligned", i);
  CHECK(g.off_codes1 - g.off_tab >= sizeof(Tab), "table region too small");
  CHECK(g.total + 1024 <= smem_limit, "shared memory");
  if (g.rstage) {  // router rows + pointer table staged before x arrives
    CHECK(g.off_act % 16 == 0, "router staging alignment");
    CHECK((size_t)g.epc * sh.H * 2 % 16 == 0, "router rows size");
    CHECK((size_t)g.rstage <= g.off_part - g.off_act, "router staging room");
  }
  const int P = sh.T * sh.k;
  for (int b = 0; b < grid; ++b) {
    Tab tb;
    uint32_t n_scale = 0, n_down = 0;
    build_tables(g, b, o, tb, n_scale, n_down);
    CHECK(tb.ncopies <= kMaxCopies && tb.npieces <= kMaxPieces, "table limits");
    CHECK(tb.nseg1 <= kMaxSegs && tb.nseg2 <= kMaxSegs, "segment limits");
    // copies: alignment, bounds, regions, barriers
    std::vector<unsigned long long> bar_bytes(kNumBars, 0);
    std::vector<int> bar_copies(kNumBars, 0);
    for (int c = 0; c < tb.ncopies; ++c) {
      const size_t d = tb.cdst[c], n = tb.cbytes[c];
      CHECK(n > 0 && n % 16 == 0, "copy %d size %zu", c, n);
      CHECK(d % 16 == 0 && tb.csrc[c] % 16 == 0, "copy %d alignment", c);
      CHECK(tb.csrc[c] + n <= o.total, "copy %d past the record", c);
      CHECK(tb.cpair[c] < P, "copy %d pair", c);
      const int bar = tb.cbar[c];
      CHECK(bar < kNumBars, "copy %d barrier", c);
      if (bar >= kNumBars) continue;
      bar_bytes[bar] += n;
      ++bar_copies[bar];
      if (bar < kMaxPieces) {
        CHECK(bar < tb.npieces, "copy %d barrier of a missing piece", c);
        CHECK(d >= g.off_codes1 && d + n <= g.off_scales1, "copy %d outside the gate/up code region", c);
      } else if (bar == kBarScales) {
        CHECK(d >= g.off_scales1 && d + n <= g.off_codes2, "copy %d outside the gate/up scale region", c);
      } else {
        CHECK(d >= g.off_codes2 && d + n <= g.off_act, "copy %d outside the down region", c);
      }
      for (int c2 = 0; c2 < c; ++c2)
        CHECK(d + n <= tb.cdst[c2] || (size_t)tb.cdst[c2] + tb.cbytes[c2] <= d, "copies %d and %d overlap", c2, c);
    }
    for (int i = 0; i < kNumBars; ++i) CHECK(bar_bytes[i] < (1ull << 20), "barrier %d expects too many bytes", i);
    for (int i = 0; i < tb.npieces; ++i) CHECK(bar_copies[i] == 2, "piece %d has %d copies", i, bar_copies[i]);
    CHECK(bar_copies[kBarScales] == (int)n_scale && bar_copies[kBarDown] == (int)n_down, "barrier counts");
    // gate/up rows: segments and pieces cover [0, n1) in order
    const int r0 = share_lo(b, (int)g.R1, g.grid), n1 = share_lo(b + 1, (int)g.R1, g.grid) - r0;
    int q = 0;
    for (int s = 0; s < tb.nseg1; ++s) {
      CHECK(tb.sq0[s] == q && tb.sn[s] > 0, "segment %d order", s);
      CHECK(r0 + tb.sq0[s] == tb.sp[s] * sh.I + tb.si0[s] && tb.si0[s] + tb.sn[s] <= sh.I, "segment %d rows", s);
      q += tb.sn[s];
    }
    CHECK(q == n1, "segments cover %d of %d rows", q, n1);
    q = 0;
    for (int pi = 0; pi < tb.npieces; ++pi) {
      const int s = tb.pseg[pi];
      CHECK(tb.pq0[pi] == q && tb.pn[pi] > 0 && tb.pn[pi] <= g.np, "piece %d order", pi);
      CHECK(s < tb.nseg1 && tb.pq0[pi] >= tb.sq0[s] && tb.pq0[pi] + tb.pn[pi] <= tb.sq0[s] + tb.sn[s],
            "piece %d outside its segment", pi);
      q += tb.pn[pi];
    }
    CHECK(q == n1, "pieces cover %d of %d rows", q, n1);
    // every byte a gate/up row reads was copied from its pair's record
    const size_t rb = sh.H / 2, sb = sh.H / G;
    for (int pi = 0; pi < tb.npieces; ++pi) {
      const int s = tb.pseg[pi], p = tb.sp[s];
      for (int r = 0; r < tb.pn[pi]; ++r) {
        const int qq = tb.pq0[pi] + r, i = tb.si0[s] + (qq - tb.sq0[s]);
        const size_t gd = g.off_codes1 + tb.poff[pi] + (size_t)r * rb;
        const size_t ud = gd + (size_t)tb.pn[pi] * rb;
        CHECK(covered(tb, gd, rb, o.gate + (size_t)i * rb, p), "gate codes of row %d", qq);
        CHECK(covered(tb, ud, rb, o.up + (size_t)i * rb, p), "up codes of row %d", qq);
        CHECK(covered(tb, g.off_scales1 + tb.gwo[s] + (size_t)(qq - tb.sq0[s]) * sb, sb, o.gate_s + (size_t)i * sb, p),
              "gate scales of row %d", qq);
        CHECK(covered(tb, g.off_scales1 + tb.uwo[s] + (size_t)(qq - tb.sq0[s]) * sb, sb, o.up_s + (size_t)i * sb, p),
              "up scales of row %d", qq);
      }
    }
    // down rows: segments cover [0, nz), every code and scale byte of every
    // (row, expert) was copied from that pair's record
    const int d0 = share_lo(b, (int)g.D, g.grid), nz = share_lo(b + 1, (int)g.D, g.grid) - d0;
    int z = 0;
    const size_t drb = sh.I / 2, dsb = sh.I / G;
    for (int s = 0; s < tb.nseg2; ++s) {
      CHECK(tb.dz0[s] == z && tb.dn[s] > 0, "down segment %d order", s);
      CHECK(d0 + tb.dz0[s] == tb.dt[s] * sh.H + tb.dn0[s] && tb.dn0[s] + tb.dn[s] <= sh.H, "down segment %d rows", s);
      for (int j = 0; j < sh.k; ++j) {
        const int p = tb.dt[s] * sh.k + j;
        for (int zr = 0; zr < tb.dn[s]; ++zr) {
          const size_t cd = g.off_codes2 + ((size_t)tb.dz0[s] * sh.k + (size_t)j * tb.dn[s] + zr) * drb;
          CHECK(covered(tb, cd, drb, o.down + (size_t)(tb.dn0[s] + zr) * drb, p), "down codes %d/%d/%d", s, j, zr);
          CHECK(covered(tb, g.off_scales2 + tb.dso[s][j] + (size_t)zr * dsb, dsb,
                        o.down_s + (size_t)(tb.dn0[s] + zr) * dsb, p),
                "down scales %d/%d/%d", s, j, zr);
        }
      }
      z += tb.dn[s];
    }
    CHECK(z == nz, "down segments cover %d of %d rows", z, nz);
  }
}

int main() {
  const size_t smem_limit = 232448;  // 227 KB per CTA
  std::vector<Shape> shapes;
  for (int T = 1; T <= 6; ++T)
    for (int fused = 0; fused < 2; ++fused) shapes.push_back({T, 10, 2560, 640, MOE_FMT_NVFP4, 512, fused != 0});
  const int Hs[] = {256, 512, 1024, 2048, 4096};
  const int Is[] = {128, 256, 640, 1024, 2880};
  const int ks[] = {1, 3, 6, 8, 10, 24, 32};
  const int Ts[] = {1, 2, 5, 8, 64};
  const int Es[] = {64, 384, 999, 1000};
  for (int fmt = 0; fmt < 2; ++fmt)
    for (int H : Hs)
      for (int I : Is)
        for (int k : ks)
          for (int T : Ts) {
            if (T * k > kMaxPairs) continue;
            const int E = Es[(H + I + k + T) % 4];
            if (k > E) continue;
            shapes.push_back({T, k, H, I, fmt, E, (H + k) % 2 == 0});
          }
  const int grids[] = {152, 148, 132};
  int fitting = 0, total = 0;
  for (const Shape& sh : shapes)
    for (int grid : grids) {
      ++total;
      if (!decode_oneshot_fits(sh.T, sh.k, sh.H, sh.I, sh.fmt, grid, smem_limit, sh.fused, sh.E)) continue;
      ++fitting;
      check_shape(sh, grid, smem_limit);
    }
  std::printf("plan check: %d of %d shape x grid cases fit the one-shot pass; %lld checks, %lld failed\n", fitting,
              total, g_checks, g_fail);
  return (g_fail == 0 && fitting > 0) ? 0 : 1;
}
