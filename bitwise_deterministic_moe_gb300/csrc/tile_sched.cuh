// Tile scheduling shared by the persistent grouped-GEMM kernels that keep
// their expert tables in the scheduler warp's registers (the CTA-pair kernel
// and the block-scaled kernel).
//
// Tile order.  A unit is one m-tile (ROWS rows) of one expert; its NT n-tiles
// are consecutive tiles (they share the X rows in L2).  Units of heavy
// experts (at least HMT m-tiles: compute-bound, each weight slice serves
// several m-tiles) and of light experts (bound by streaming their weights
// from HBM) are merged in proportion -- unit position p is heavy iff
// floor((p+1)H/U) > floor(pH/U) -- so both the tensor cores and HBM stay
// busy; within each class units follow expert order, so an expert's weight
// slices are reused while resident.  The order only decides when a tile
// runs, never what it computes.
#pragma once

#include <cstdint>

namespace dmoe {

// A decoded tile as a scheduler queues it: cur = tile index (-1 = no more
// tiles), e = expert, row0 = first row of the tile (it covers row0 ..
// row0 + ROWS - 1), row_end = end of the expert's rows, columns n0 .. n0 + BN - 1.
struct alignas(16) QTile {
  int cur, e, row0, row_end, n0, pad0, pad1, pad2;
};

// The scheduler warp's expert tables, held in registers: lane l holds experts
// e = 32 l + j (j = 0..31; E <= 1024), with off[e .. e + 32] (o), and the
// exclusive prefixes of the m-tiles of heavy (hp) and light (cp) experts
// before e.  All indices are compile-time after unrolling, so the arrays stay
// in registers.
struct ExpertTables {
  int o[33];
  int hp[32];
  int cp[32];
};

// Loads the offsets, validates them (non-decreasing, off[0] = 0, off[E] = R)
// and builds the prefixes for tiles of ROWS rows, experts with >= HMT m-tiles
// being heavy; returns the units of each class through hu / lu and whether
// the offsets are bad (warp-uniform).  Called by all 32 lanes.
template <int ROWS, int HMT>
__device__ __forceinline__ bool build_tables(ExpertTables& t, const int32_t* offsets, int E, int R, int lane,
                                             int& hu, int& lu) {
  bool bad = false;
#pragma unroll
  for (int j = 0; j <= 32; ++j) {
    const int e = 32 * lane + j;
    t.o[j] = e <= E ? offsets[e] : 0;
    if (e == E && t.o[j] != R) bad = true;
  }
  if (lane == 0 && t.o[0] != 0) bad = true;
  int hsum = 0, csum = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int e = 32 * lane + j;
    int mt = 0;
    if (e < E) {
      if (t.o[j + 1] < t.o[j]) bad = true;
      mt = t.o[j + 1] > t.o[j] ? (t.o[j + 1] - t.o[j] + ROWS - 1) / ROWS : 0;
    }
    t.hp[j] = hsum;
    t.cp[j] = csum;
    hsum += mt >= HMT ? mt : 0;
    csum += mt >= HMT ? 0 : mt;
  }
  int hx = hsum, cx = csum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int hv = __shfl_up_sync(0xffffffffu, hx, d);
    const int cv = __shfl_up_sync(0xffffffffu, cx, d);
    if (lane >= d) {
      hx += hv;
      cx += cv;
    }
  }
  hu = __shfl_sync(0xffffffffu, hx, 31);
  lu = __shfl_sync(0xffffffffu, cx, 31);
  hx -= hsum;
  cx -= csum;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    t.hp[j] += hx;
    t.cp[j] += cx;
  }
  return __any_sync(0xffffffffu, bad);
}

// Decodes tile t (all 32 lanes): the expert is the largest e < E whose class
// prefix is <= u; the lanes whose first expert qualifies form a prefix of the
// warp, the last of them holds e, and within it the qualifying experts are a
// prefix of its 32.  The class's prefix is selected with a mask, element by
// element, so the tables are never addressed through a pointer.
template <int ROWS, int BN>
__device__ __forceinline__ QTile decode_tile_warp(int t, const ExpertTables& tb, int E, int NT, int H, int U,
                                                  int lane) {
  const int p = t / NT;
  const int n_tile = t - p * NT;
  const int i = int((long long)p * H / U);
  const bool heavy = (long long)(p + 1) * H / U > i;
  const int u = heavy ? i : p - i;
  const int hm = heavy ? -1 : 0;
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int pv = (tb.hp[j] & hm) | (tb.cp[j] & ~hm);
    cnt += (32 * lane + j < E && pv <= u) ? 1 : 0;
  }
  const int seg = 31 - __clz(__ballot_sync(0xffffffffu, cnt > 0));   // lane 0 always (prefix 0 <= u)
  int pe = 0, oe = 0, oe1 = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int hj = j == cnt - 1 ? -1 : 0;
    pe = (((tb.hp[j] & hm) | (tb.cp[j] & ~hm)) & hj) | (pe & ~hj);
    oe = (tb.o[j] & hj) | (oe & ~hj);
    oe1 = (tb.o[j + 1] & hj) | (oe1 & ~hj);
  }
  const int c = __shfl_sync(0xffffffffu, cnt, seg);
  pe = __shfl_sync(0xffffffffu, pe, seg);
  oe = __shfl_sync(0xffffffffu, oe, seg);
  oe1 = __shfl_sync(0xffffffffu, oe1, seg);
  QTile q;
  q.cur = t;
  q.e = 32 * seg + c - 1;
  q.row0 = oe + (u - pe) * ROWS;
  q.row_end = oe1;
  q.n0 = n_tile * BN;
  q.pad0 = q.pad1 = q.pad2 = 0;
  return q;
}

}  // namespace dmoe
