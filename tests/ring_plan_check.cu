// Host-side check of the ring decode kernel's chunk plan (decode_ring_plan.h):
// for many shapes and grid sizes, every CTA's chunks are enumerated on the CPU
// with the kernel's own plan functions and checked against what the kernel
// relies on:
//  - the gate/up chunks of all CTAs cover every (pair, row) exactly once; a
//    chunk holds at most kRG rows and crosses at most one pair boundary;
//  - the down blocks of all CTAs cover every (token, output row) exactly once,
//    at most kRD rows of one token each;
//  - a slot holds a gate/up chunk (codes, and both pieces' scale windows
//    within their room) and jn experts' down parts (codes and scale window);
//  - every bulk copy starts on a 16-byte boundary in the record and in the
//    slot and has a size that is a multiple of 16 bytes;
//  - the scale byte a consumer reads for a row and unit, at the offset the
//    kernel computes, is the record's scale byte of that row and unit as
//    copied by the producer's window.
// Exit status 0 when every check passes.
#include <cstdio>
#include <vector>

#include "common.cuh"
#include "decode_ring_plan.h"

using namespace moe;
using namespace moe::ring;

static long long g_fail = 0, g_checks = 0;
#define CHECK(cond, ...)                                   \
  do {                                                     \
    ++g_checks;                                            \
    if (!(cond)) {                                         \
      if (g_fail++ < 20) {                                 \
        std::printf("FAIL line %d: ", __LINE__);           \
        std::printf(__VA_ARGS__);                          \
        std::printf("\n");                                 \
      }                                                    \
    }                                                      \
  } while (0)

// The producer copies a scale window [w.lo, w.lo + w.bytes) of the record to
// slot offset `at`; the consumer reads record byte `want` at slot offset
// `got`.  True when that slot byte holds that record byte.
static bool maps(const Win& w, size_t at, size_t got, size_t want) {
  if (want < w.lo || want >= w.lo + w.bytes) return false;
  return got == at + (want - w.lo);
}

static void check_shape(int H, int I, int fmt, int T, int k, int grid) {
  const int G = fmt == MOE_FMT_NVFP4 ? 16 : 32;
  const int sstep = fmt == MOE_FMT_NVFP4 ? 2 : 1;  // scale bytes per 32-element unit
  const RecordOffsets o = record_offsets(H, I, fmt);
  const int P = T * k;
  const long long R1 = (long long)P * I, R2 = (long long)T * H;
  const int slot_bytes = plan_slot_bytes(H, I, G);
  const int jn = plan_jn(k, I, G, slot_bytes);
  const uint32_t cbg = (uint32_t)(H / 2), cbd = (uint32_t)(I / 2);
  const uint32_t so = 2u * kRG * cbg, room = (uint32_t)gu_scale_room(H, G);
  const uint32_t per = (uint32_t)dn_part_bytes(I, G);
  CHECK(slot_bytes % 128 == 0, "slot bytes %d", slot_bytes);
  CHECK(jn >= 1 && jn <= k && (long long)jn * per <= slot_bytes, "jn %d", jn);
  CHECK(so + 2 * room <= (uint32_t)slot_bytes, "gate/up chunk exceeds the slot");
  CHECK(o.gate % 16 == 0 && o.up % 16 == 0 && o.down % 16 == 0 && cbg % 16 == 0 && cbd % 16 == 0,
        "code parts not 16-byte aligned");
  std::vector<unsigned char> seen1((size_t)R1, 0), seen2((size_t)R2, 0);
  for (int b = 0; b < grid; ++b) {
    const int r0 = share_at(b, grid, R1), r1 = share_at(b + 1, grid, R1);
    const int q0 = share_at(b, grid, R2), q1 = share_at(b + 1, grid, R2);
    const int n1 = gu_chunks(r0, r1);
    for (int c = 0; c < n1; ++c) {
      const GuChunk g = gu_chunk(c, r0, r1, I);
      CHECK(g.nr >= 1 && g.nr <= kRG && g.rs == r0 + c * kRG && g.rs + g.nr <= r1, "chunk rows");
      CHECK(g.n0 >= 1 && g.n0 <= g.nr && g.i0 + g.n0 <= I && (long long)g.p0 * I + g.i0 == g.rs, "piece 0");
      CHECK(g.n0 == g.nr || g.i0 + g.n0 == I, "piece 0 ends before the pair does");
      CHECK(g.n0 == g.nr || g.p0 + 1 < P, "piece 1 past the last pair");
      for (int r = g.rs; r < g.rs + g.nr; ++r) seen1[r]++;
      // the scale windows of the two pieces, as the producer places them
      Win gw[2], uw[2];
      uint32_t gso = 0, uso = 0, goff[2], uoff[2];
      for (int pc = 0; pc < 2; ++pc) {
        const int n = pc == 0 ? g.n0 : g.nr - g.n0, i = pc == 0 ? g.i0 : 0;
        gw[pc] = window(o.gate_s + (size_t)i * (H / G), (size_t)n * (H / G));
        uw[pc] = window(o.up_s + (size_t)i * (H / G), (size_t)n * (H / G));
        CHECK(gw[pc].lo % 16 == 0 && gw[pc].bytes % 16 == 0 && (so + gso) % 16 == 0 && (so + room + uso) % 16 == 0,
              "scale window alignment");
        CHECK(((size_t)i * cbg + o.gate) % 16 == 0, "gate rows alignment");
        goff[pc] = gso;
        uoff[pc] = uso;
        if (n > 0) {
          gso += gw[pc].bytes;
          uso += uw[pc].bytes;
        }
      }
      CHECK(gso <= room && uso <= room, "scale windows %u %u exceed the room %u (H %d)", gso, uso, room, H);
      // every row's scale bytes at the consumer's offsets
      const Win gw0 = window(o.gate_s + (size_t)g.i0 * (H / G), (size_t)g.n0 * (H / G));
      const Win uw0 = window(o.up_s + (size_t)g.i0 * (H / G), (size_t)g.n0 * (H / G));
      for (int ri = 0; ri < g.nr; ++ri) {
        const int pc = ri < g.n0 ? 0 : 1;
        const int i = pc == 0 ? g.i0 + ri : ri - g.n0, rr = pc == 0 ? ri : ri - g.n0;
        uint32_t cg = gw0.delta, cu = uw0.delta;  // the consumer's offsets, as the kernel computes them
        if (pc == 1) {
          cg = gw0.bytes + window(o.gate_s, (size_t)(g.nr - g.n0) * (H / G)).delta;
          cu = uw0.bytes + window(o.up_s, (size_t)(g.nr - g.n0) * (H / G)).delta;
        }
        for (int u = 0; u < H / 32; u += (H / 32 > 8 ? H / 32 / 7 : 1)) {
          const size_t gotg = (size_t)so + cg + (size_t)rr * (H / G) + (size_t)sstep * u;
          const size_t wantg = o.gate_s + (size_t)i * (H / G) + (size_t)sstep * u;
          CHECK(maps(gw[pc], (size_t)so + goff[pc], gotg, wantg), "gate scale row %d unit %d", i, u);
          const size_t gotu = (size_t)so + room + cu + (size_t)rr * (H / G) + (size_t)sstep * u;
          const size_t wantu = o.up_s + (size_t)i * (H / G) + (size_t)sstep * u;
          CHECK(maps(uw[pc], (size_t)so + room + uoff[pc], gotu, wantu), "up scale row %d unit %d", i, u);
        }
      }
    }
    const int nb2 = dn_blocks(q0, q1, H);
    for (int bi = 0; bi < nb2; ++bi) {
      int qs = -1, nd = 0;
      const bool ok = dn_block(bi, q0, q1, H, qs, nd);
      CHECK(ok && nd >= 1 && nd <= kRD && qs >= q0 && qs + nd <= q1, "down block");
      CHECK(qs / H == (qs + nd - 1) / H, "down block spans two tokens");
      if (!ok) continue;
      for (int q = qs; q < qs + nd; ++q) seen2[q]++;
      const int n0 = qs % H;
      const Win dw = window(o.down_s + (size_t)n0 * (I / G), (size_t)nd * (I / G));
      CHECK(kRD * cbd + dw.bytes <= per && dw.lo % 16 == 0 && dw.bytes % 16 == 0, "down window");
      CHECK(((size_t)n0 * cbd + o.down) % 16 == 0 && ((size_t)nd * cbd) % 16 == 0, "down rows alignment");
      for (int jj = 0; jj < jn; ++jj) CHECK(((size_t)jj * per) % 16 == 0 && (jj + 1) * per <= (uint32_t)slot_bytes, "down part");
      for (int rb = 0; rb < nd; ++rb)
        for (int u = 0; u < I / 32; u += (I / 32 > 8 ? I / 32 / 7 : 1)) {
          const size_t got = (size_t)kRD * cbd + dw.delta + (size_t)rb * (I / G) + (size_t)sstep * u;
          const size_t want = o.down_s + (size_t)(n0 + rb) * (I / G) + (size_t)sstep * u;
          CHECK(maps(dw, (size_t)kRD * cbd, got, want), "down scale row %d unit %d", n0 + rb, u);
        }
    }
    int qx = 0, nx = 0;
    CHECK(!dn_block(nb2, q0, q1, H, qx, nx), "a down block past the last");
  }
  for (long long r = 0; r < R1; ++r) CHECK(seen1[r] == 1, "gate/up row %lld covered %d times (H %d I %d T %d k %d grid %d)",
                                          r, seen1[r], H, I, T, k, grid);
  for (long long q = 0; q < R2; ++q) CHECK(seen2[q] == 1, "output row %lld covered %d times", q, seen2[q]);
}

int main() {
  const int shapes[][2] = {{2560, 640}, {4096, 2880}, {1024, 512}, {512, 256}, {256, 128}, {192, 128}, {128, 64}};
  const int tk[][2] = {{1, 10}, {2, 10}, {4, 10}, {32, 10}, {51, 10}, {64, 8}, {1, 6}, {2, 6}, {5, 4}, {3, 1}, {512, 1}};
  const int grids[] = {152, 148, 132, 7};
  int cases = 0;
  for (auto& sh : shapes)
    for (int fmt = 0; fmt < 2; ++fmt) {
      if (sh[0] % 32 || sh[1] % 32) continue;
      for (auto& t : tk)
        for (int grid : grids) {
          if (t[0] * t[1] > 512) continue;
          check_shape(sh[0], sh[1], fmt, t[0], t[1], grid);
          ++cases;
        }
    }
  std::printf("ring plan: %d cases, %lld checks, %lld failed\n", cases, g_checks, g_fail);
  return g_fail == 0 ? 0 : 1;
}
