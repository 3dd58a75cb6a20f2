// ccl_kernels.cuh -- device code of the labelling library (sm_103a).
//
// The four stages of "every-colour" (blogs.fablnx.com) ch. 05 -- Start,
// Connect, Collapse, Number -- as kernels over 256 x TH pixel tiles:
//
//   k_tile_local  Start + Connect + Collapse inside one tile, in shared
//                 memory.  A lane owns 8 consecutive pixels of a row; runs of
//                 equal colour are found from equal-to-left bit masks and one
//                 warp vote for the last run start left of each lane (ch. 08
//                 switch 1, the warp finds the runs), so that a run is one
//                 union-find node.  Joins go to the row above first and
//                 skip what the left neighbour already joins (ch. 08 "First,
//                 the order of the joins" and switch 2, the Wu-Otoo-Suzuki
//                 scan mask); walks halve paths with the same atomic minimum
//                 (switch 3).  Output: a 2-byte leader map (a pixel's run
//                 start; for a run start, its tile-local leader in the
//                 tile's first and last rows, column 0 and the run holding
//                 the last column, elsewhere an ancestor on the way to it),
//                 a leader bitmap, a leader count per 256-pixel chunk of a
//                 row, and a global parent slot (its own raster index) for
//                 every leader whose region touches the tile border.
//   k_seams       Connect across tile seams: the joins of the same rule whose
//                 partner is in another tile, united in the global parent
//                 array with atomicMin and retry (ch. 06 Fig. 10;
//                 bendabir.com, "Unions are parallel").  A leader that is
//                 re-pointed leaves the bitmap and its chunk count.
//   k_scan_*      Number, first part: exclusive prefix sum of chunk counts
//                 (ch. 08 switch 5; ch. 12, a prefix sum inside Number).
//   k_resolve     Collapse + Number for the border leaders re-pointed across
//                 seams (from the tiles' border lists): each walks to its
//                 final leader and stores that leader's label, negated, in
//                 its own slot.
//   k_number      Number, last part: a leader's label is 1 + the number of
//                 leaders before it in raster order; every pixel takes its
//                 tile-local leader's label, finishing the walk in the leader
//                 map (Collapse inside the tile is lazy: see k_tile_local).
//
// After labelling, on request (ccl_region_stats): region statistics --
// area, bounding box, first pixel, coordinate sums -- as a reduction over the
// final labels: k_stats_offsets, k_stats_init, k_region_stats.
//
// In the ignoring modes (binary: value 0; or one named value, "every-colour"
// ch. 08 switch 4 "Ignore the paper") pixels equal to Geom::bgval are
// background: label 0, part of no run's joins.
//
// Leaders are always the smallest raster index of their set (ch. 04: the
// larger leader points at the smaller one), so the labels come out in the
// raster order of each region's first pixel.
#pragma once

#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "ccl.h"

namespace ccl_dev {

constexpr int TW = 256;             // tile width == numbering chunk width
constexpr int LOG_TW = 8;
constexpr int TH = 16;              // tile height
constexpr int TILE = TW * TH;
constexpr int NT = 256;             // threads per block
constexpr int NWARPS = NT / 32;
constexpr int RPW = TH / NWARPS;    // tile rows per warp
constexpr int PX = TW / 32;         // consecutive pixels per lane
constexpr int CHUNK = 256;          // pixels of a row counted together
constexpr int SCAN_ITEMS = 16;
constexpr int SCAN_BLOCK = NT * SCAN_ITEMS;
constexpr uint16_t LBG = 0xFFFF;    // background in the tile-local leader map
constexpr unsigned FULL = 0xffffffffu;
static_assert(PX == 8, "a lane owns 8 pixels");
static_assert(TH % NWARPS == 0, "whole rows per warp");

constexpr int FLAG_WALK_CAP = 1;    // a union-find walk or retry loop hit its cap
constexpr int FLAG_INTERNAL = 2;    // an invariant of the numbering pass failed
constexpr int FLAG_STATS_CAP = 4;   // more regions than the statistics array holds
constexpr int FLAG_BAD_LABEL = 8;   // a label outside 0..n of its image, or a negative count

struct Geom {
  int H, W;
  int tilesX, tilesY;
  int WPR;                      // bitmap words per row = ceil(W / 32)
  int CPR;                      // chunks per row       = ceil(W / 256)
  long long HW;                 // pixels per image
  long long tilesPerImage;
  unsigned long long wmagic;    // exact d / W for 0 <= d < 2^31: (d * wmagic) >> wshift
  int wshift;
  unsigned long long tmagic;    // the same for d / tilesPerImage
  int tshift;
  unsigned long long xmagic;    // the same for d / tilesX
  int xshift;
  int vec_img;                  // image rows allow 8-pixel vector loads
  int vec_out;                  // leader-map and label rows allow vector access
  uint32_t bgval;               // background value when background is ignored
};

// Per-tile border data written by k_tile_local:
//  rec   4*TH words per tile: colours of the left column, leaders of the left
//        column, colours of the right column, leaders of the right column
//        (leaders as image raster indices, -1 for background);
//  list  up to BLCAP tile-local indices per tile: leaders whose region
//        touches the tile border (count in cnt).
constexpr int BLCAP = 2 * TW + 2 * TH;
struct Border {
  uint32_t* rec;
  uint16_t* list;
  uint32_t* cnt;
};

struct TileCoord {
  int b, tx, y0, x0, th, tw;
};

// quotient of 0 <= d < 2^31 by the divisor whose magic pair is (m, sh)
__device__ __forceinline__ int div_magic(int d, unsigned long long m, int sh) {
  return (int)(((unsigned long long)(unsigned)d * m) >> sh);
}

// (tile indices are below 2^31: the host refuses larger grids)
__device__ __forceinline__ TileCoord tile_coord_of(const Geom& g, long long tile) {
  TileCoord t;
  const int ti = (int)tile;
  t.b = div_magic(ti, g.tmagic, g.tshift);
  const int rest = ti - t.b * (int)g.tilesPerImage;
  const int ty = div_magic(rest, g.xmagic, g.xshift);
  t.tx = rest - ty * g.tilesX;
  t.y0 = ty * TH;
  t.x0 = t.tx * TW;
  t.th = min(TH, g.H - t.y0);
  t.tw = min(TW, g.W - t.x0);
  return t;
}

__device__ __forceinline__ TileCoord tile_coord(const Geom& g) { return tile_coord_of(g, blockIdx.x); }

__device__ __forceinline__ int div_w(int d, const Geom& g) { return div_magic(d, g.wmagic, g.wshift); }

__device__ __forceinline__ void raise_flag(int* status, int f) { atomicOr(status, f); }

// Event counters, compiled in only for the counters build (-DCCL_COUNTERS;
// read with ccl_debug_counters): walks and their steps in shared and global
// memory, links, kept seam pairs and resolve steps.  Each event is one global
// atomic, so that build is slow; the product build has none of it.
#ifdef CCL_COUNTERS
__device__ unsigned long long g_counters[CCL_NCOUNTERS];
#define CCL_COUNT(i) atomicAdd(&g_counters[i], 1ull)
#else
#define CCL_COUNT(i) ((void)0)
#endif

// ---------------------------------------------------------------- pixel I/O
// Eight consecutive pixels, widened to 32 bits.

template <typename T>
__device__ __forceinline__ void load8(const T* p, bool vec, int n, uint32_t c[PX]);

template <>
__device__ __forceinline__ void load8<uint8_t>(const uint8_t* p, bool vec, int n, uint32_t c[PX]) {
  if (vec) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[j] = (v.x >> (8 * j)) & 0xFFu;
      c[j + 4] = (v.y >> (8 * j)) & 0xFFu;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) c[j] = j < n ? (uint32_t)__ldg(p + j) : 0u;
  }
}

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, bool vec, int n, uint32_t c[PX]) {
  if (vec) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[2 * j] = w[j] & 0xFFFFu;
      c[2 * j + 1] = w[j] >> 16;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) c[j] = j < n ? (uint32_t)__ldg(p + j) : 0u;
  }
}

// 24-bit RGB, three bytes a pixel with no padding: the form "every-colour"
// reads its drawings in (ch. 08 "Tried and dropped": a packed 32-bit copy of
// the picture was slower and took twice the memory).  A pixel compares as
// its 24-bit value.
struct Rgb24 {
  uint8_t v[3];
  __device__ __forceinline__ operator uint32_t() const {
    return (uint32_t)v[0] | ((uint32_t)v[1] << 8) | ((uint32_t)v[2] << 16);
  }
};
static_assert(sizeof(Rgb24) == 3, "three bytes a pixel");

// Eight RGB pixels are 24 bytes: from an 8-byte boundary, three 8-byte
// loads (a warp reads 768 contiguous bytes) and the bytes regrouped.
template <>
__device__ __forceinline__ void load8<Rgb24>(const Rgb24* p, bool vec, int n, uint32_t c[PX]) {
  if (vec) {
    const uint2* q = reinterpret_cast<const uint2*>(p);
    const uint2 a = __ldg(q), b = __ldg(q + 1), d = __ldg(q + 2);
    c[0] = a.x & 0xFFFFFFu;
    c[1] = __byte_perm(a.x, a.y, 0x0543) & 0xFFFFFFu;
    c[2] = __byte_perm(a.y, b.x, 0x0432) & 0xFFFFFFu;
    c[3] = b.x >> 8;
    c[4] = b.y & 0xFFFFFFu;
    c[5] = __byte_perm(b.y, d.x, 0x0543) & 0xFFFFFFu;
    c[6] = __byte_perm(d.x, d.y, 0x0432) & 0xFFFFFFu;
    c[7] = d.y >> 8;
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) c[j] = j < n ? (uint32_t)p[j] : 0u;
  }
}

template <>
__device__ __forceinline__ void load8<uint32_t>(const uint32_t* p, bool vec, int n, uint32_t c[PX]) {
  if (vec) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) c[j] = j < n ? __ldg(p + j) : 0u;
  }
}

// ------------------------------------------------------------ shared memory
// Union-find over tile-local indices r * TW + x.  Reads go through a
// volatile pointer so every step sees other threads' links.

__device__ __forceinline__ int find_s(volatile int* par, int x, int cap, int* status) {
  CCL_COUNT(CCL_CNT_TILE_WALKS);
  for (int s = 0; s < cap; ++s) {
    CCL_COUNT(CCL_CNT_TILE_STEPS);
    const int p = par[x];
    if (p == x) return x;
    const int gp = par[p];
    if (gp == p) return p;
    atomicMin((int*)&par[x], gp);   // path halving: an arrow only ever moves down
    x = gp;
  }
  raise_flag(status, FLAG_WALK_CAP);
  return x;
}

__device__ __forceinline__ void union_s(volatile int* par, int a, int b, int cap, int* status) {
  for (int s = 0; s < cap; ++s) {
    a = find_s(par, a, cap, status);
    b = find_s(par, b, cap, status);
    if (a == b) return;
    if (a > b) { const int t = a; a = b; b = t; }
    CCL_COUNT(CCL_CNT_TILE_LINKS);
    const int old = atomicMin((int*)&par[b], a);   // larger leader under smaller
    if (old == b) return;
    b = old;                                         // someone got there first
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// ------------------------------------------------------------ global memory
// Union-find over image raster indices.  Only leaders' slots are touched:
// every walk starts at a tile-local leader and every node after that is a
// leader too.

// Every loaded arrow is range-checked before it is followed: if a capped
// walk in an earlier stage left a pixel pointing at a non-leader, whose slot
// was never written, the walk stops with -1 instead of leaving the image.
__device__ __forceinline__ int find_g(int* P, int x, int n, int cap, int* status) {
  CCL_COUNT(CCL_CNT_GLOBAL_WALKS);
  for (int s = 0; s < cap; ++s) {
    CCL_COUNT(CCL_CNT_GLOBAL_STEPS);
    const int p = __ldcg(P + x);
    if (p == x) return x;
    if ((unsigned)p >= (unsigned)n) {
      raise_flag(status, FLAG_INTERNAL);
      return -1;
    }
    const int gp = __ldcg(P + p);
    if (gp == p) return p;
    if ((unsigned)gp >= (unsigned)n) {
      raise_flag(status, FLAG_INTERNAL);
      return -1;
    }
    atomicMin(P + x, gp);
    x = gp;
  }
  raise_flag(status, FLAG_WALK_CAP);
  return -1;
}

__device__ __forceinline__ void drop_leader(int b, uint32_t* bm, uint32_t* cnt, const Geom& g) {
  const int by = div_w(b, g);
  const int bx = b - by * g.W;
  atomicAnd(bm + (size_t)by * g.WPR + (bx >> 5), ~(1u << (bx & 31)));
  atomicSub(cnt + (size_t)by * g.CPR + (bx >> LOG_TW), 1u);
}

__device__ __forceinline__ void union_g(int* P, int a, int b, uint32_t* bm, uint32_t* cnt,
                                        const Geom& g, int cap, int* status) {
  const int n = (int)g.HW;
  for (int s = 0; s < cap; ++s) {
    a = find_g(P, a, n, cap, status);
    b = find_g(P, b, n, cap, status);
    if (a < 0 || b < 0 || a == b) return;
    if (a > b) { const int t = a; a = b; b = t; }
    CCL_COUNT(CCL_CNT_GLOBAL_LINKS);
    const int old = atomicMin(P + b, a);
    if (old == b) {            // b stopped being a leader, exactly once
      drop_leader(b, bm, cnt, g);
      return;
    }
    b = old;
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// image raster index of the tile-local leader of pixel (y, x), -1 for background.
// For a pixel in the first or last row of its tile: the leader map holds its
// run start, and a run start of those rows holds its tile-local leader, so
// two hops give the leader.  (k_seams asks only for such pixels.)
__device__ __forceinline__ int leader_of(const uint16_t* Li, int y, int x, const Geom& g) {
  const int ty0 = y & ~(TH - 1), tx0 = x & ~(TW - 1);
  uint16_t l = Li[(long long)y * g.W + x];
  if (l >= TILE) return -1;   // background (LBG)
  int ly = ty0 + (l >> LOG_TW), lx = tx0 + (l & (TW - 1));
  if (ly >= g.H || lx >= g.W) return -1;   // only a corrupted map can get here
  if (ly != y || lx != x) {
    l = Li[(long long)ly * g.W + lx];
    if (l >= TILE) return -1;
    ly = ty0 + (l >> LOG_TW);
    lx = tx0 + (l & (TW - 1));
    if (ly >= g.H || lx >= g.W) return -1;
  }
  return ly * g.W + lx;
}

// ------------------------------------------------------------------ kernels

// Occupancy matters more than a few spilled registers here: the in-tile
// union-find (short, divergent walks in shared memory) runs best with every
// warp slot of the SM filled, so the kernel is held to 32 registers (8
// blocks of 256 threads per SM) and keeps no copy of the image in shared
// memory: Start compares each row with the row above while both are in
// registers (the row above was just loaded by a sibling warp: an L1 or L2
// hit) and keeps only the join bits for Connect.
template <typename T, int CONN, bool BIN>
__global__ void __launch_bounds__(NT, 8) k_tile_local(const T* __restrict__ img, uint16_t* __restrict__ L16,
                                                   int32_t* __restrict__ P, uint32_t* __restrict__ bm,
                                                   uint32_t* __restrict__ cnt, Border bd, Geom g,
                                                   int cap, int* status, long long tile0) {
  __shared__ int nborder;
  __shared__ __align__(16) int par[TILE];
  __shared__ __align__(16) uint8_t mark[TILE];
  __shared__ __align__(16) uint16_t jlist[NWARPS][TW];   // a row's joins, dealt out to the lanes
  const long long tile = tile0 + blockIdx.x;   // launches may cover a band of tiles
  const TileCoord t = tile_coord_of(g, tile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const long long ioff = (long long)t.b * g.HW;
  const T* im = img + ioff;
  uint16_t* Li = L16 + ioff;
  int32_t* Pi = P + ioff;
  uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  uint32_t* cnti = cnt + (long long)t.b * g.H * g.CPR;
  for (int i = threadIdx.x * 16; i < TILE; i += NT * 16)
    *reinterpret_cast<uint4*>(mark + i) = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) nborder = 0;
  const int nval = max(0, min(PX, t.tw - xl));
  const unsigned vmask = (1u << nval) - 1u;
  const bool vec = g.vec_img && nval == PX;
  // per row of this warp: foreground pixels, pixels equal to their left
  // neighbour (same run), and the row position of the last run start left
  // of this lane
  unsigned fgm[RPW], eqm[RPW], tdm[RPW];
  int befm[RPW];

  // ---- Start: every pixel points at the first pixel of its run
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    fgm[k] = 0;
    eqm[k] = 0;
    tdm[k] = 0;
    befm[k] = -1;
    if (r >= t.th) continue;   // warp-uniform
    uint32_t c[PX];
    load8<T>(im + (long long)(t.y0 + r) * g.W + t.x0 + xl, vec, nval, c);
    unsigned fg = vmask;
    if (BIN) {
#pragma unroll
      for (int j = 0; j < PX; ++j)
        if (c[j] == g.bgval) fg &= ~(1u << j);
    }
    const uint32_t cl = __shfl_up_sync(FULL, c[PX - 1], 1);
    // (all-pixels mode: the lane on the left is whole wherever this lane
    // has a pixel, so its last pixel is foreground)
    const unsigned fgl = BIN ? __shfl_up_sync(FULL, fg, 1) : 0x80u;
    unsigned eq = (lane > 0 && c[0] == cl) ? (fg & (fgl >> (PX - 1)) & 1u) : 0u;
#pragma unroll
    for (int j = 1; j < PX; ++j) eq |= (c[j] == c[j - 1] ? 1u : 0u) << j;
    eq &= fg & (fg << 1 | 1u);
    const unsigned starts = fg & ~eq;
    // the joins with the row above (Connect makes them): this row's pixels
    // against the row above, while they are in registers
    if (r > 0) {   // warp-uniform
      uint32_t u[PX];
      load8<T>(im + (long long)(t.y0 + r - 1) * g.W + t.x0 + xl, vec, nval, u);
      const uint32_t uL = __shfl_up_sync(FULL, u[PX - 1], 1);
      const uint32_t uR = __shfl_down_sync(FULL, u[0], 1);
      unsigned mU = 0, mUL = 0, mUR = 0;
#pragma unroll
      for (int j = 0; j < PX; ++j) {
        const uint32_t cj = c[j];
        mU |= (cj == u[j] ? 1u : 0u) << j;
        mUL |= (j > 0 ? cj == u[j - 1] : (lane > 0 && cj == uL)) ? (1u << j) : 0u;
        if (CONN == 8)
          mUR |= (j < PX - 1 ? cj == u[j + 1] : (lane < 31 && cj == uR)) ? (1u << j) : 0u;
      }
      mU &= fg;
      mUL &= fg;
      mUR &= fg & ((vmask >> 1) | ((lane < 31 && xl + PX < t.tw) ? 0x80u : 0u));
      if (CONN == 8)
        tdm[k] = (mU & ~eq) | ((mUL & ~mU & ~eq) << 8) | ((mUR & ~mU) << 16);
      else
        tdm[k] = mU & ~(eq & mUL);
    }
    // the last run start left of this lane: the last start of the nearest
    // lane on the left that has one
    const unsigned left = __ballot_sync(FULL, starts != 0u) & ((1u << lane) - 1u);
    int cur = __shfl_sync(FULL, xl + 31 - __clz(starts), 31 - __clz(left | 1u));
    if (!left) cur = -1;
    befm[k] = cur;
    // (all-pixels mode: every pixel of the lane is foreground; the entries
    // past the tile's last column are never read)
    int pv[PX];
#pragma unroll
    for (int j = 0; j < PX; ++j) {
      if ((starts >> j) & 1u) cur = xl + j;
      pv[j] = (!BIN || ((fg >> j) & 1u)) ? r * TW + cur : -1;
    }
    int4* pp = reinterpret_cast<int4*>(par + r * TW + xl);
    pp[0] = make_int4(pv[0], pv[1], pv[2], pv[3]);
    pp[1] = make_int4(pv[4], pv[5], pv[6], pv[7]);
    fgm[k] = fg;
    eqm[k] = eq;
  }
  __syncthreads();

  // ---- Connect inside the tile.  Runs are already one node each, so every
  // join goes to the row above; a pixel equal to its left neighbour leaves
  // up-left and up to it (8-connectivity), or up when up-left matches too
  // (4-connectivity).  Neighbours outside the tile count as absent here;
  // k_seams makes those joins.  Start found the joins (tdm: bit j up, j+8
  // up-left, j+16 up-right of the lane's pixel j).
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    if (r >= t.th || r == 0) continue;   // warp-uniform
    unsigned todo = tdm[k];
    const int i0 = r * TW + xl;
    // A lane walks its own joins one after another, so a warp loops as often
    // as its busiest lane.  When some lane has more than one join, the row's
    // joins are first listed in shared memory (tile index | direction << 12)
    // and dealt out to all 32 lanes.
    const int nj = __popc(todo);
    bool own = !__any_sync(FULL, nj > 1);
    int total = 0, pos = 0;
    if (!own) {
      int inc = nj;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += y;
      }
      total = __shfl_sync(FULL, inc, 31);
      pos = inc - nj;
      own = total > TW;   // more than the list holds: keep them in place
    }
    if (own) {
      while (todo) {
        const int bpos = __ffs(todo) - 1;
        todo &= todo - 1;
        const int j = bpos & 7;
        const int d = (bpos >> 3) == 0 ? 0 : ((bpos >> 3) == 1 ? -1 : 1);
        const int a = i0 + j, b = i0 + j - TW + d;
        const int pa = par[a], pb = par[b];   // run starts (a pixel's entry never changes)
        if (pa != pb) union_s(par, pa, pb, cap, status);   // else joined already
      }
    } else {
      while (todo) {
        const int bpos = __ffs(todo) - 1;
        todo &= todo - 1;
        jlist[warp][pos++] = (uint16_t)((i0 + (bpos & 7)) | ((bpos >> 3) << 12));
      }
      __syncwarp();
      for (int q = lane; q < total; q += 32) {
        const int e = jlist[warp][q];
        const int a = e & (TILE - 1), dc = e >> 12;
        const int b = a - TW + (dc == 0 ? 0 : (dc == 1 ? -1 : 1));
        const int pa = par[a], pb = par[b];
        if (pa != pb) union_s(par, pa, pb, cap, status);
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // ---- Collapse inside the tile, where it is read: the run starts of the
  // tile's first and last rows (k_seams reads their leaders through the
  // leader map), of column 0 and of the run holding the last column (border
  // marks and records) walk to their leader and store it.  Every other start
  // keeps the ancestor Connect left it; k_number finishes those walks.  The
  // leader map of a row is then a copy of par: a pixel's run start, a start's
  // leader or ancestor.  Leaders are the starts whose entry is themselves.
  unsigned rootm[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    rootm[k] = 0;
    if (r >= t.th) continue;   // warp-uniform
    const unsigned starts = fgm[k] & ~eqm[k];
    const int i0 = r * TW + xl;
    const bool edgeRow = r == 0 || r == t.th - 1;
    unsigned m = edgeRow ? starts : (starts & (lane == 0 ? 1u : 0u));
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int root = find_s(par, i0 + j, cap, status);
      par[i0 + j] = root;
      mark[root] = 1;
    }
    // the tile's right column: the leader of its run, marked
    const int jr = t.tw - 1 - xl;
    if (jr >= 0 && jr < PX && ((fgm[k] >> jr) & 1u)) {
      const unsigned sm = starts & ((2u << jr) - 1u);
      const int sr = r * TW + (sm ? xl + 31 - __clz(sm) : befm[k]);
      const int root = find_s(par, sr, cap, status);
      par[sr] = root;
      mark[root] = 1;
    }
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    if (r >= t.th) continue;   // warp-uniform
    const int i0 = r * TW + xl;
    const int4 p0 = reinterpret_cast<const int4*>(par + i0)[0];
    const int4 p1 = reinterpret_cast<const int4*>(par + i0)[1];
    const int pj[PX] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const unsigned starts = fgm[k] & ~eqm[k];
    unsigned rm = 0;
    uint32_t lw[PX / 2];
#pragma unroll
    for (int j = 0; j < PX; ++j) {
      rm |= (pj[j] == i0 + j) ? (1u << j) : 0u;
      // a start that is not a leader: its grandparent (halves the walk left
      // to k_number); any other pixel: its run start
      int e = pj[j];
      if (((starts >> j) & 1u) && e != i0 + j) e = par[e];
      const uint32_t v = min((uint32_t)e, (uint32_t)LBG);   // background (-1) -> LBG
      if (j & 1) lw[j >> 1] = __byte_perm(lw[j >> 1], v, 0x5410);
      else lw[j >> 1] = v;
    }
    rm &= vmask;
    rootm[k] = rm;
    uint16_t* lrow = Li + (long long)(t.y0 + r) * g.W + t.x0 + xl;
    if (g.vec_out && nval == PX) {
      *reinterpret_cast<uint4*>(lrow) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j)
        if (j < nval) lrow[j] = (uint16_t)(lw[j >> 1] >> (16 * (j & 1)));
    }
    const unsigned b1 = __shfl_down_sync(FULL, rm, 1);
    const unsigned b2 = __shfl_down_sync(FULL, rm, 2);
    const unsigned b3 = __shfl_down_sync(FULL, rm, 3);
    if ((lane & 3) == 0 && xl < t.tw)
      bmi[(long long)(t.y0 + r) * g.WPR + ((t.x0 + xl) >> 5)] = rm | (b1 << 8) | (b2 << 16) | (b3 << 24);
    const unsigned n = __reduce_add_sync(FULL, (unsigned)__popc(rm));
    if (lane == 0) cnti[(long long)(t.y0 + r) * g.CPR + t.tx] = n;
  }
  __syncthreads();

  // ---- border records: colour and leader of the left and right columns
  uint32_t* rec = bd.rec + tile * 4 * TH;
  if (threadIdx.x < 2 * t.th) {
    const int right = (int)threadIdx.x >= t.th, r = (int)threadIdx.x - right * t.th;
    const int i = r * TW + (right ? t.tw - 1 : 0);
    const int p = par[i];
    const int lead = p < 0 ? -1 : find_s(par, i, cap, status);
    rec[2 * right * TH + r] = (uint32_t)im[(long long)(t.y0 + r) * g.W + t.x0 + (right ? t.tw - 1 : 0)];
    rec[(2 * right + 1) * TH + r] =
        lead < 0 ? 0xFFFFFFFFu : (uint32_t)((t.y0 + (lead >> LOG_TW)) * g.W + t.x0 + (lead & (TW - 1)));
  }

  // ---- leaders whose region touches the border: a global parent slot and
  // an entry in the tile's border list
  uint16_t* blist = bd.list + tile * BLCAP;
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    if (r >= t.th) continue;   // warp-uniform
    // the marks of the lane's 8 pixels (bytes 0 or 1) as 8 bits
    const uint2 mk = *reinterpret_cast<const uint2*>(mark + r * TW + xl);
    unsigned m = rootm[k] & (((mk.x * 0x01020408u) >> 24) | (((mk.y * 0x01020408u) >> 24) << 4));
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int i = r * TW + xl + j;
      const int gi = (t.y0 + r) * g.W + t.x0 + xl + j;
      Pi[gi] = gi;
      const int slot = atomicAdd(&nborder, 1);
      if (slot < BLCAP) blist[slot] = (uint16_t)i;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) bd.cnt[tile] = (uint32_t)min(nborder, BLCAP);
}

// Connect across tile seams: the joins of the same rule as inside a tile,
// evaluated on the true neighbourhood, whose partner lies in another tile.
// A tile handles its top seam (its first row against the row above) and its
// left seam (its left column against the left tile's right column, from the
// border records).
//
// One warp per tile, SEAM_WARPS tiles per block, so that many tiles' global
// walks are in flight on an SM at once (the kernel is bound by the latency
// of those dependent loads, not by its few bytes).  A lane owns 8
// consecutive columns of the seam rows, as in k_tile_local.  The warp first
// keeps every distinct pair of leaders to join once (a small hash set: along
// a seam many joins link the same two regions), then its lanes unite the
// kept pairs side by side.
constexpr int SEAM_WARPS = 2;
constexpr int SEAM_HASH = 128;

template <typename T, int CONN, bool BIN>
__global__ void __launch_bounds__(32 * SEAM_WARPS, 32) k_seams(const T* __restrict__ img,
                                                               const uint16_t* __restrict__ L16, int32_t* P,
                                                               uint32_t* bm, uint32_t* cnt, Border bd, Geom g,
                                                               long long nTiles, int cap, int* status) {
  __shared__ __align__(16) uint16_t lcS[SEAM_WARPS][TW], laS[SEAM_WARPS][TW];   // leader map, rows y0 and y0-1
  __shared__ unsigned long long seenS[SEAM_WARPS][SEAM_HASH];
  constexpr unsigned long long EMPTY = ~0ull;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const long long tile = (long long)blockIdx.x * SEAM_WARPS + w;
  if (tile >= nTiles) return;   // the whole warp; nothing below waits on the block
  uint16_t* lc = lcS[w];
  uint16_t* la = laS[w];
  unsigned long long* seen = seenS[w];
#pragma unroll
  for (int i = lane; i < SEAM_HASH; i += 32) seen[i] = EMPTY;
  const TileCoord t = tile_coord_of(g, tile);
  const long long ioff = (long long)t.b * g.HW;
  const T* im = img + ioff;
  const uint16_t* Li = L16 + ioff;
  int32_t* Pi = P + ioff;
  uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  uint32_t* cnti = cnt + (long long)t.b * g.H * g.CPR;
  const bool top = t.y0 > 0;
  const long long row = (long long)t.y0 * g.W + t.x0;
  const int nval = max(0, min(PX, t.tw - xl));
  const bool vimg = g.vec_img && nval == PX;
  const bool vmap = g.vec_out && nval == PX;

  // ---- the two seam rows: colours in registers, leader-map entries in
  // shared memory (a walk's second hop may land in another lane's columns)
  uint32_t c[PX], u[PX];
  load8<T>(im + row + xl, vimg, nval, c);
  if (vmap) {
    *reinterpret_cast<uint4*>(lc + xl) = __ldg(reinterpret_cast<const uint4*>(Li + row + xl));
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) lc[xl + j] = j < nval ? Li[row + xl + j] : LBG;
  }
  if (top) {
    load8<T>(im + row - g.W + xl, vimg, nval, u);
    if (vmap) {
      *reinterpret_cast<uint4*>(la + xl) = __ldg(reinterpret_cast<const uint4*>(Li + row - g.W + xl));
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j) la[xl + j] = j < nval ? Li[row - g.W + xl + j] : LBG;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PX; ++j) u[j] = 0;
  }
  // neighbours beyond the tile's columns: left of column 0, above-right of
  // the last column
  uint32_t cEdge = 0, uEdge = 0;
  if (lane == 0 && t.x0 > 0) {
    cEdge = im[row - 1];
    if (top) uEdge = im[row - g.W - 1];
  }
  const bool rightTile = t.tw == TW && t.x0 + TW < g.W;
  if (lane == 31 && rightTile && top) uEdge = im[row - g.W + TW];
  // (every lane takes part in each shuffle; the edge lanes then substitute)
  const uint32_t cls = __shfl_up_sync(FULL, c[PX - 1], 1);
  const uint32_t uls = __shfl_up_sync(FULL, u[PX - 1], 1);
  const uint32_t urs = __shfl_down_sync(FULL, u[0], 1);
  const uint32_t cl = lane == 0 ? cEdge : cls;
  const uint32_t ul = lane == 0 ? uEdge : uls;
  const uint32_t ur = lane == 31 ? uEdge : urs;
  const unsigned vmask = (1u << nval) - 1u;
  unsigned fg = vmask;
  if (BIN) {
#pragma unroll
    for (int j = 0; j < PX; ++j)
      if (c[j] == g.bgval) fg &= ~(1u << j);
  }
  const bool hasL0 = lane > 0 || t.x0 > 0;                 // column xl-1 exists
  const bool hasR7 = nval == PX && t.x0 + xl + PX < g.W;   // column xl+8 exists
  unsigned eqL = 0, eqU = 0, eqUL = 0, eqUR = 0;
#pragma unroll
  for (int j = 0; j < PX; ++j) {
    const uint32_t cj = c[j];
    eqL |= (j > 0 ? cj == c[j - 1] : (hasL0 && cj == cl)) ? (1u << j) : 0u;
    eqU |= (cj == u[j]) ? (1u << j) : 0u;
    eqUL |= (j > 0 ? cj == u[j - 1] : (hasL0 && cj == ul)) ? (1u << j) : 0u;
    if (CONN == 8) eqUR |= (j < PX - 1 ? cj == u[j + 1] : (hasR7 && cj == ur)) ? (1u << j) : 0u;
  }
  eqL &= fg;
  const unsigned upm = top ? fg : 0u;
  eqU &= upm;
  eqUL &= upm;
  eqUR &= upm & ((vmask >> 1) | (hasR7 ? 0x80u : 0u));
  unsigned todo;   // bit j: up, j+8: up-left, j+16: up-right
  if (CONN == 8)
    todo = (eqU & ~eqL) | ((eqUL & ~eqU & ~eqL) << 8) | ((eqUR & ~eqU) << 16);
  else
    todo = eqU & ~(eqL & eqUL);
  __syncwarp();

  const int n = (int)g.HW;
  // keep a pair of leaders once; unite at once when the set is crowded
  auto keep = [&](int a, int b) {
    if (a == b || a < 0 || b < 0 || a >= n || b >= n) return;
    const unsigned long long key =
        ((unsigned long long)(unsigned)min(a, b) << 32) | (unsigned)max(a, b);
    unsigned h = (unsigned)((key * 0x9E3779B97F4A7C15ull) >> 40) & (SEAM_HASH - 1);
    for (int probe = 0; probe < 8; ++probe) {
      const unsigned long long prev = atomicCAS(&seen[h], EMPTY, key);
      if (prev == EMPTY) CCL_COUNT(CCL_CNT_SEAM_PAIRS);
      if (prev == EMPTY || prev == key) return;
      h = (h + 1) & (SEAM_HASH - 1);
    }
    union_g(Pi, a, b, bmi, cnti, g, cap, status);
  };
  // leader of (y0, x): the map gives the run start (in this row), whose entry
  // gives the leader; a run start's own entry already is the leader
  auto leader_here = [&](int x) {
    const int l1 = lc[x], l2 = (l1 >> LOG_TW) == 0 ? lc[l1 & (TW - 1)] : l1;
    return (t.y0 + (l2 >> LOG_TW)) * g.W + t.x0 + (l2 & (TW - 1));
  };
  while (todo) {
    const int bpos = __ffs(todo) - 1;
    todo &= todo - 1;
    const int x = xl + (bpos & 7);
    const int xx = x + ((bpos >> 3) == 0 ? 0 : ((bpos >> 3) == 1 ? -1 : 1));
    int b;
    if (xx >= 0 && xx < t.tw) {   // the tile above: its last row is row y0-1
      const int m1 = la[xx], m2 = (m1 >> LOG_TW) == TH - 1 ? la[m1 & (TW - 1)] : m1;
      b = (t.y0 - TH + (m2 >> LOG_TW)) * g.W + t.x0 + (m2 & (TW - 1));
    } else {
      b = leader_of(Li, t.y0 - 1, t.x0 + xx, g);
    }
    keep(leader_here(x), b);
  }
  // the first column's left neighbour lies in the left tile: its border record
  if (lane == 0 && (eqL & 1u)) keep(leader_here(0), (int)bd.rec[(tile - 1) * 4 * TH + 3 * TH]);

  // ---- left column of the tile (rows below the first) against the left
  // tile's right column
  if (t.x0 > 0 && lane >= 1 && lane < t.th) {
    const int r = lane;
    const uint32_t* recT = bd.rec + tile * 4 * TH;
    const uint32_t* recL = recT - 4 * TH;
    const uint32_t cp = recT[r], cU = recT[r - 1];                     // (r, x0), (r-1, x0)
    const uint32_t cq = recL[2 * TH + r], cUL = recL[2 * TH + r - 1];  // (r, x0-1), (r-1, x0-1)
    const int lp = (int)recT[TH + r], lU = (int)recT[TH + r - 1];
    const int lq = (int)recL[3 * TH + r], lUL = (int)recL[3 * TH + r - 1];
    const bool fgp = !BIN || cp != g.bgval, fgq = !BIN || cq != g.bgval;
    const bool eqLc = fgp && cp == cq;
    if (eqLc) keep(lp, lq);
    if (CONN == 8) {
      const bool eqUc = cp == cU, eqULc = fgp && cp == cUL;
      if (eqULc && !eqUc && !eqLc) keep(lp, lUL);
      // (r, x0-1) joins its up-right (r-1, x0) unless its own up matches
      if (fgq && cq == cU && cq != cUL) keep(lq, lU);
    }
  }
  __syncwarp();
  // ---- every kept pair, the warp's lanes side by side: the pairs are first
  // packed to the front of the set (in place: a slot moves only to a lower
  // or its own index, after its chunk has been read)
  int kept = 0;
#pragma unroll
  for (int base = 0; base < SEAM_HASH; base += 32) {
    const unsigned long long key = seen[base + lane];
    const unsigned bal = __ballot_sync(FULL, key != EMPTY);
    if (key != EMPTY) seen[kept + __popc(bal & ((1u << lane) - 1u))] = key;
    kept += __popc(bal);
    __syncwarp();
  }
  for (int i = lane; i < kept; i += 32) {
    const unsigned long long key = seen[i];
    union_g(Pi, (int)(key >> 32), (int)(key & 0xffffffffu), bmi, cnti, g, cap, status);
  }
}

// ---- exclusive prefix sum of the chunk counts (three passes, no waits)

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total) {
  __shared__ uint32_t warp_sums[NWARPS];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_sums[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const uint32_t s = lane < NWARPS ? warp_sums[lane] : 0;
    uint32_t si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, si, o);
      if (lane >= o) si += y;
    }
    if (lane < NWARPS) warp_sums[lane] = si - s;
    if (lane == NWARPS - 1) *total = si;
  }
  __syncthreads();
  const uint32_t res = inc - v + warp_sums[wid];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(NT) k_scan_reduce(const uint32_t* __restrict__ cnt, long long n,
                                                    uint32_t* __restrict__ bsum) {
  __shared__ uint32_t tot;
  const long long base = (long long)blockIdx.x * SCAN_BLOCK + (long long)threadIdx.x * SCAN_ITEMS;
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < SCAN_ITEMS; ++k)
    if (base + k < n) s += cnt[base + k];
  block_exclusive_scan(s, &tot);
  if (threadIdx.x == 0) bsum[blockIdx.x] = tot;
}

// one block: exclusive scan of the block sums, grand total at bsum[nb]
__global__ void __launch_bounds__(NT) k_scan_top(uint32_t* bsum, int nb) {
  __shared__ uint32_t tot;
  uint32_t carry = 0;
  for (int base = 0; base < nb; base += NT) {
    const int i = base + threadIdx.x;
    const uint32_t v = i < nb ? bsum[i] : 0;
    const uint32_t ex = block_exclusive_scan(v, &tot);
    if (i < nb) bsum[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) bsum[nb] = carry;
}

__global__ void __launch_bounds__(NT) k_scan_down(uint32_t* cnt, long long n, const uint32_t* bsum) {
  __shared__ uint32_t tot;
  const long long base = (long long)blockIdx.x * SCAN_BLOCK + (long long)threadIdx.x * SCAN_ITEMS;
  uint32_t v[SCAN_ITEMS];
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < SCAN_ITEMS; ++k) {
    v[k] = base + k < n ? cnt[base + k] : 0;
    s += v[k];
  }
  uint32_t run = block_exclusive_scan(s, &tot) + bsum[blockIdx.x];
#pragma unroll
  for (int k = 0; k < SCAN_ITEMS; ++k) {
    if (base + k < n) cnt[base + k] = run;
    run += v[k];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) cnt[n] = bsum[gridDim.x];
}

__global__ void k_region_counts(const uint32_t* off, long long chunksPerImage, int batch,
                                int32_t* n_out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch)
    n_out[b] = (int32_t)(off[(long long)(b + 1) * chunksPerImage] - off[(long long)b * chunksPerImage]);
}

// label of leader gidx: 1 + leaders before it in raster order within its image
__device__ __forceinline__ int number_of(int gidx, const uint32_t* bmi, const uint32_t* offi,
                                         uint32_t base0, const Geom& g, int* status) {
  if (gidx < 0 || (long long)gidx >= g.HW) {
    raise_flag(status, FLAG_INTERNAL);
    return 0;
  }
  const int gy = div_w(gidx, g), gx = gidx - gy * g.W;
  const long long w0 = (long long)gy * g.WPR + ((gx >> LOG_TW) << 3);
  const int nw = (gx >> 5) & 7;   // whole words of the chunk before the leader's word
  // every load of the chunk's words is issued before any is used
  const uint32_t chunk = offi[(long long)gy * g.CPR + (gx >> LOG_TW)];
  const uint32_t word = bmi[w0 + nw];
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < 7; ++k)
    if (k < nw) s += __popc(bmi[w0 + k]);
  if (!((word >> (gx & 31)) & 1u)) raise_flag(status, FLAG_INTERNAL);
  s += __popc(word & ((1u << (gx & 31)) - 1u));
  return (int)(chunk - base0 + s + 1u);
}

constexpr int RESOLVE_WARPS = 2;   // tiles (a warp each) per block: small blocks free their slot sooner

// Collapse + Number for the leaders re-pointed across seams, taken from the
// tiles' border lists (a warp per tile).  Each walks to its final leader
// (halving on the way), takes that leader's label and stores it negated in
// its own slot.  A walk that meets a slot already holding a negated label
// stops there: every node on a walk belongs to the same region.
__global__ void __launch_bounds__(32 * RESOLVE_WARPS, 32) k_resolve(Border bd, long long nTiles, int32_t* P,
                                                const uint32_t* __restrict__ bm,
                                                const uint32_t* __restrict__ off, Geom g, int cap,
                                                int* status) {
  const long long tile = (long long)blockIdx.x * RESOLVE_WARPS + (threadIdx.x >> 5);
  if (tile >= nTiles) return;
  const int lane = threadIdx.x & 31;
  const TileCoord t = tile_coord_of(g, tile);
  const long long ioff = (long long)t.b * g.HW;
  int32_t* Pi = P + ioff;
  const uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  const uint32_t* offi = off + (long long)t.b * g.H * g.CPR;
  const uint32_t base0 = offi[0];
  const int n = (int)g.HW;
  const int count = min((int)bd.cnt[tile], BLCAP);
  const uint16_t* list = bd.list + tile * BLCAP;
  for (int k = lane; k < count; k += 32) {
    const int l = list[k];
    const int r = (t.y0 + (l >> LOG_TW)) * g.W + t.x0 + (l & (TW - 1));
    const int v = __ldcg(Pi + r);
    if (v == r || v < 0) continue;   // still a leader, or already resolved
    int node = r, lab = 0, s = 0;
    for (; s < cap; ++s) {
      CCL_COUNT(CCL_CNT_RESOLVE_STEPS);
      const int p = __ldcg(Pi + node);
      if (p < 0) { lab = -p; break; }
      if (p == node) { lab = number_of(node, bmi, offi, base0, g, status); break; }
      if (p >= n) { raise_flag(status, FLAG_INTERNAL); break; }
      const int gp = __ldcg(Pi + p);
      if (gp < 0) { lab = -gp; break; }
      if (gp == p) { lab = number_of(p, bmi, offi, base0, g, status); break; }
      if (gp >= n) { raise_flag(status, FLAG_INTERNAL); break; }
      atomicMin(Pi + node, gp);   // a slot holding a negated label keeps it
      node = gp;
    }
    if (s == cap) raise_flag(status, FLAG_WALK_CAP);
    if (lab > 0) atomicMin(Pi + r, -lab);
  }
}

// Number: labels of the tile's leaders -- from the bitmap and the chunk
// offsets, or, for leaders re-pointed across a seam (all of them are in the
// tile's border list), the negated label k_resolve left in their slot --
// then every pixel takes the label of its tile-local leader, reached by a walk
// in the leader map: pixel -> run start -> ancestors -> leader.  The labels buffer holds the slots of border leaders until
// this kernel overwrites it; a tile reads only its own slots, before writing.
// Both lookup tables end in a sentinel entry (index TILE: map -> TILE, label
// 0), which background and any out-of-range entry are clamped to.
__global__ void __launch_bounds__(NT, 8) k_number(const uint16_t* __restrict__ L16, int32_t* labels,
                                               const uint32_t* __restrict__ bm,
                                               const uint32_t* __restrict__ off, Border bd, Geom g,
                                               int* status, long long tile0) {
  __shared__ __align__(16) int lab[TILE + 1];
  __shared__ __align__(16) uint16_t lmap[TILE + 8];   // the tile's leader map
  const long long tile = tile0 + blockIdx.x;   // launches may cover a band of tiles
  const TileCoord t = tile_coord_of(g, tile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const long long ioff = (long long)t.b * g.HW;
  const uint16_t* Li = L16 + ioff;
  int32_t* Pi = labels + ioff;
  const uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  const uint32_t* offi = off + (long long)t.b * g.H * g.CPR;
  const uint32_t base0 = offi[0];
  const int nval = max(0, min(PX, t.tw - xl));
  const bool vec = g.vec_out && nval == PX;
  if (threadIdx.x == 0) {
    lab[TILE] = 0;
    lmap[TILE] = (uint16_t)TILE;
  }
  // leaders re-pointed across a seam (all in the tile's border list) carry the
  // label k_resolve stored, negated, in their slot: the list entry and then the
  // slot are loaded first, so that both loads overlap the rows' work below
  const uint16_t* list = bd.list + tile * BLCAP;
  const int count = min((int)bd.cnt[tile], BLCAP);
  const int l0 = list[threadIdx.x];   // NT < BLCAP: always inside the tile's list
  const int gi0 = (t.y0 + (l0 >> LOG_TW)) * g.W + t.x0 + (l0 & (TW - 1));
  const int v0 = (int)threadIdx.x < count ? Pi[gi0] : 0;
  uint32_t lw[RPW][PX / 2];   // the lane's 8 leader-map entries per row, two per word

#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
#pragma unroll
    for (int q = 0; q < PX / 2; ++q) lw[k][q] = 0xFFFFFFFFu;
    if (r >= t.th) continue;   // warp-uniform
    const uint16_t* lrow = Li + (long long)(t.y0 + r) * g.W + t.x0 + xl;
    if (vec) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(lrow));
      lw[k][0] = v.x; lw[k][1] = v.y; lw[k][2] = v.z; lw[k][3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j) {
        const uint32_t l = j < nval ? (uint32_t)lrow[j] : 0xFFFFu;
        lw[k][j >> 1] = (j & 1) ? ((lw[k][j >> 1] & 0xFFFFu) | (l << 16))
                                : ((lw[k][j >> 1] & 0xFFFF0000u) | l);
      }
    }
    *reinterpret_cast<uint4*>(lmap + r * TW + xl) = make_uint4(lw[k][0], lw[k][1], lw[k][2], lw[k][3]);
    // word w of the row segment belongs to lanes 4w..4w+3, which all hold it:
    // leaders in the words before it, by a scan over the 8 words
    const uint32_t w = xl < t.tw ? bmi[(long long)(t.y0 + r) * g.WPR + ((t.x0 + xl) >> 5)] : 0u;
    const uint32_t cw = __popc(w);
    uint32_t inc = cw;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t pre = inc - cw;
    const uint32_t o = offi[(long long)(t.y0 + r) * g.CPR + t.tx] - base0;
    const int i0 = r * TW + xl;
    // the bitmap's leaders among this lane's pixels: 1 + leaders before them
    unsigned m = (w >> (xl & 31)) & 0xFFu;
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int bit = (xl + j) & 31;
      lab[i0 + j] = (int)(o + pre + __popc(w & ((1u << bit) - 1u)) + 1u);
    }
  }
  if ((int)threadIdx.x < count) {
    if (v0 < 0) lab[l0 & (TILE - 1)] = -v0;
    else if (v0 != gi0) raise_flag(status, FLAG_INTERNAL);   // neither leader nor resolved
  }
  for (int q = threadIdx.x + NT; q < count; q += NT) {   // lists longer than a block
    const int l = list[q];
    const int gi = (t.y0 + (l >> LOG_TW)) * g.W + t.x0 + (l & (TW - 1));
    const int v = Pi[gi];
    if (v < 0) lab[l & (TILE - 1)] = -v;
    else if (v != gi) raise_flag(status, FLAG_INTERNAL);
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp + k * NWARPS;
    if (r >= t.th) continue;
    int out[PX];
    uint32_t prev = 0xFFFFFFFFu;   // the run start of the pixel before
#pragma unroll
    for (int j = 0; j < PX; ++j) {
      // pixel -> run start -> ... -> leader: the map's entries point ever
      // lower until a leader, whose entry is itself (sentinel: TILE).  The
      // pixels of a run share the walk: it is made once per run start.
      const uint32_t l = min((lw[k][j >> 1] >> (16 * (j & 1))) & 0xFFFFu, (uint32_t)TILE);
      // the pixel before is in the same run: it has the same run start, or
      // it is the run start (whose own entry is its leader or an ancestor)
      if (l == prev || (j > 0 && l == (uint32_t)(r * TW + xl + j - 1))) {
        out[j] = out[j > 0 ? j - 1 : 0];
        prev = l;
      } else {
        uint32_t x = l, y = min((uint32_t)lmap[x], (uint32_t)TILE);
        for (int s = 0; s < TILE && y != x; ++s) {
          x = y;
          y = min((uint32_t)lmap[x], (uint32_t)TILE);
        }
        out[j] = lab[x];
        prev = l;
      }
    }
    int32_t* orow = Pi + (long long)(t.y0 + r) * g.W + t.x0 + xl;
    if (vec) {
      reinterpret_cast<int4*>(orow)[0] = make_int4(out[0], out[1], out[2], out[3]);
      reinterpret_cast<int4*>(orow)[1] = make_int4(out[4], out[5], out[6], out[7]);
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j)
        if (j < nval) orow[j] = out[j];
    }
  }
}

// ------------------------------------------------------ region statistics
// The step after labelling on the pages: regions are labelled so that their
// area and position can be measured (CUDA image segmentation, lpnh.cn,
// §1.1), statistics on every labelled region come next ("GPU Connected
// Component Labeling", mcclanahoochie.com, closing section), and each area
// gets its bounding box (bendabir.com, Prologue).  A reduction by label, as
// the lpnh.cn page builds its global reductions (§2.3, §6.1): each block
// first sums into a private table in shared memory, and only the block's
// totals go to global memory with atomics.

// per-image offsets of the statistics entries: off[b] = n[0] + ... + n[b-1],
// off[batch] = the total (one block)
__global__ void __launch_bounds__(NT) k_stats_offsets(const int32_t* __restrict__ n, int batch,
                                                      long long* off, int* status) {
  __shared__ long long wsum[NWARPS];
  __shared__ long long carry;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < batch; base += NT) {
    const int i = base + threadIdx.x;
    long long v = i < batch ? (long long)n[i] : 0;
    if (v < 0) {
      raise_flag(status, FLAG_BAD_LABEL);
      v = 0;
    }
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) wsum[wid] = inc;
    __syncthreads();
    long long before = carry, total = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
      if (w < wid) before += wsum[w];
      total += wsum[w];
    }
    if (i < batch) off[i] = before + inc - v;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) off[batch] = carry;
}

// every entry below min(total, capacity): the empty statistics
__global__ void k_stats_init(ccl_region_stat* stats, long long capacity, const long long* off,
                             int batch, int* status) {
  const long long total = off[batch];
  const long long n = total < capacity ? total : capacity;
  if (blockIdx.x == 0 && threadIdx.x == 0 && total > capacity) raise_flag(status, FLAG_STATS_CAP);
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    ccl_region_stat z;
    z.area = 0;
    z.y_min = INT_MAX;
    z.x_min = INT_MAX;
    z.y_max = -1;
    z.x_max = -1;
    z.first = INT_MAX;
    z.sum_y = 0;
    z.sum_x = 0;
    stats[e] = z;
  }
}

// one segment's contribution to one entry of the global array
__device__ __forceinline__ void stats_add_global(ccl_region_stat* e, int area, int y_min, int x_min,
                                                 int y_max, int x_max, int first,
                                                 unsigned long long sy, unsigned long long sx) {
  atomicAdd(&e->area, area);
  atomicMin(&e->y_min, y_min);
  atomicMin(&e->x_min, x_min);
  atomicMax(&e->y_max, y_max);
  atomicMax(&e->x_max, x_max);
  atomicMin(&e->first, first);
  atomicAdd(reinterpret_cast<unsigned long long*>(&e->sum_y), sy);
  atomicAdd(reinterpret_cast<unsigned long long*>(&e->sum_x), sx);
}

// A block per 256-column x SR-row area; a warp per row at a time, a lane per
// 8 consecutive labels (as in k_tile_local).  Each lane splits its labels
// into runs of equal label; the warp's runs of one label are merged first
// (lanes grouped by label, their lengths, ends and sums reduced across the
// group) so that a label updates the area's table once per row.  The table
// (open addressing on the label) keeps, per label, the area, box, first
// pixel, coordinate sums and whether any of its pixels lies on an inner edge
// of the area (a row or column with neighbours outside it).  A label that
// does not is wholly inside the area -- a region that reaches outside crosses
// that edge -- so its entry is stored outright; the others are added to the
// global entry with atomics.  A run whose label finds no free slot goes
// straight to the global entry.  Every label must be one 4- or 8-connected
// set, as the labels of this library are.
#ifndef CCL_STATS_HASH
#define CCL_STATS_HASH 1024
#define CCL_STATS_ROWS 16
#define CCL_STATS_NT 256
#endif
constexpr int STATS_HASH = CCL_STATS_HASH;
constexpr int SR = CCL_STATS_ROWS;       // rows of a statistics area
constexpr int STATS_NT = CCL_STATS_NT;   // threads of a statistics block
constexpr int STATS_NWARPS = STATS_NT / 32;
constexpr int STATS_HASH_BITS = STATS_HASH == 4096 ? 12 : STATS_HASH == 2048 ? 11 : STATS_HASH == 1024 ? 10 : 9;
static_assert((1 << STATS_HASH_BITS) == STATS_HASH, "a power of two");
constexpr int EDGE_BIT = 1 << 30;   // in a table entry's area word: a pixel on an inner edge

__global__ void __launch_bounds__(STATS_NT) k_region_stats(const int32_t* __restrict__ labels,
                                                     const int32_t* __restrict__ n_regions,
                                                     const long long* __restrict__ off,
                                                     ccl_region_stat* stats, long long capacity,
                                                     Geom g, int* status) {
  // per slot: label, area (+ EDGE_BIT), smallest / largest column, largest
  // row, first raster index, and the row and column sums relative to the
  // area's corner (the smallest row is the first pixel's)
  __shared__ int hkey[STATS_HASH], harea[STATS_HASH], hxmin[STATS_HASH], hxmax[STATS_HASH];
  __shared__ int hymax[STATS_HASH], hfirst[STATS_HASH];
  __shared__ unsigned hsy[STATS_HASH], hsx[STATS_HASH];
  for (int i = threadIdx.x; i < STATS_HASH; i += STATS_NT) {
    hkey[i] = 0;   // labels start at 1
    harea[i] = 0;
    hxmin[i] = INT_MAX;
    hxmax[i] = -1;
    hymax[i] = -1;
    hfirst[i] = INT_MAX;
    hsy[i] = 0;
    hsx[i] = 0;
  }
  __syncthreads();
  // block -> image, area row, area column
  const int areasY = (int)(((long long)g.H + SR - 1) / SR);
  const long long perImage = (long long)areasY * g.tilesX;
  const int b = (int)(blockIdx.x / perImage);
  const int rest = (int)(blockIdx.x - (long long)b * perImage);
  const int ay = div_magic(rest, g.xmagic, g.xshift), ax = rest - ay * g.tilesX;
  const int y0 = ay * SR, y1 = y0 + min(SR, g.H - y0) - 1;   // rows y0..y1
  const int x0 = ax * TW, x1 = x0 + min(TW, g.W - x0) - 1;   // columns x0..x1
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const int nb = n_regions[b];
  const long long base = off[b];
  const int32_t* li = labels + (long long)b * g.HW;
  const int nval = max(0, min(PX, x1 - x0 + 1 - xl));
  const bool vec = g.vec_out && nval == PX;
  const unsigned vmask = (1u << nval) - 1u;
  // inner edges: a pixel there has neighbours outside the area
  const bool edgeL = x0 > 0, edgeR = x1 < g.W - 1;
  for (int y = y0 + warp; y <= y1; y += STATS_NWARPS) {
    const int32_t* row = li + (long long)y * g.W + x0 + xl;
    int v[PX];
    if (vec) {
      const int4 p = __ldg(reinterpret_cast<const int4*>(row));
      const int4 q = __ldg(reinterpret_cast<const int4*>(row) + 1);
      v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
      v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j) v[j] = j < nval ? __ldg(row + j) : 0;
    }
    const bool edgeRow = (y == y0 && y0 > 0) || (y == y1 && y1 < g.H - 1);
    // runs of equal label inside the lane
    unsigned same = 0;   // bit j: v[j] == v[j-1]
#pragma unroll
    for (int j = 1; j < PX; ++j) same |= (v[j] == v[j - 1] ? 1u : 0u) << j;
    const unsigned starts = vmask & ~same;
    // an end: the next label differs, or the pixel is the lane's last valid one
    unsigned ends = vmask & (~(same >> 1) | (vmask ^ (vmask >> 1)));
    // A run that crosses from lane L into lanes L+1.. is counted once, by
    // lane L: a segmented suffix sum over the lanes gathers the pieces of
    // the lanes it continues into (each lane's first run, while the lanes
    // it passes through hold nothing else).
    const int lastv = nval > 0 ? v[nval - 1] : 0;
    const int prevLast = __shfl_up_sync(FULL, lastv, 1);
    const bool contL = lane > 0 && nval > 0 && v[0] == prevLast;   // my first run began to my left
    const bool single = __popc(ends) == 1;
    const int e0 = ends ? __ffs(ends) - 1 : 0;                      // end of my first run
    const bool contNext = __shfl_down_sync(FULL, contL ? 1 : 0, 1) != 0 && lane < 31;
    // the piece I hand to the lane on my left, and whether the chain goes on past me
    unsigned pl = contL ? (unsigned)(e0 + 1) : 0u;                   // length
    unsigned px = contL ? (unsigned)(2 * xl + e0) * (unsigned)(e0 + 1) / 2u : 0u;   // column sum
    unsigned pm = contL ? (unsigned)(xl + e0) : 0u;                  // last column
    unsigned pe = (contL && ((xl + e0 == x1 - x0 && edgeR) || edgeRow)) ? 1u : 0u;
    bool brk = !(single && contNext);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned nl = __shfl_down_sync(FULL, pl, o), nx = __shfl_down_sync(FULL, px, o);
      const unsigned nm = __shfl_down_sync(FULL, pm, o), ne = __shfl_down_sync(FULL, pe, o);
      const bool nb2 = __shfl_down_sync(FULL, brk ? 1 : 0, o) != 0;
      if (!brk && lane + o < 32) {
        pl += nl;
        px += nx;
        pm = max(pm, nm);
        pe |= ne;
        brk = nb2;
      }
    }
    // the chain that continues my last run: the sums from lane + 1
    const unsigned cl = __shfl_down_sync(FULL, pl, 1), cx = __shfl_down_sync(FULL, px, 1);
    const unsigned cm = __shfl_down_sync(FULL, pm, 1), ce = __shfl_down_sync(FULL, pe, 1);
    bool firstRun = true;
    while (ends) {
      const int e = __ffs(ends) - 1;
      ends &= ends - 1;
      const bool isFirst = firstRun;
      firstRun = false;
      if (isFirst && contL) continue;   // counted by the lane where the run began
      const int sj = 31 - __clz(starts & ((2u << e) - 1u));
      int l = 0;
#pragma unroll
      for (int j = 0; j < PX; ++j)
        if (j == e) l = v[j];
      if (l == 0) continue;
      if (l < 0 || l > nb) {
        raise_flag(status, FLAG_BAD_LABEL);
        continue;
      }
      unsigned xs = (unsigned)(xl + sj), xe = (unsigned)(xl + e);   // columns in the area
      unsigned area = xe - xs + 1u;
      unsigned sxs = (xs + xe) * area / 2u;
      unsigned edge = (edgeRow || (xs == 0u && edgeL) || (x0 + (int)xe == x1 && edgeR)) ? 1u : 0u;
      if (ends == 0u && contNext) {   // my last run goes on into the next lanes
        area += cl;
        sxs += cx;
        xe = max(xe, cm);
        edge |= ce;
      }
      const int first = y * g.W + x0 + (int)xs;
      unsigned h = ((unsigned)l * 2654435761u) >> (32 - STATS_HASH_BITS);
      bool kept = false;
      for (int probe = 0; probe < 16 && !kept; ++probe) {
        const int prev = atomicCAS(&hkey[h], 0, l);
        if (prev == 0 || prev == l) {
          atomicAdd(&harea[h], (int)area);
          if (edge) atomicOr(&harea[h], EDGE_BIT);
          atomicMin(&hxmin[h], (int)xs);
          atomicMax(&hxmax[h], (int)xe);
          atomicMax(&hymax[h], y);
          atomicMin(&hfirst[h], first);
          atomicAdd(&hsy[h], (unsigned)(y - y0) * area);
          atomicAdd(&hsx[h], sxs);
          kept = true;
        }
        h = (h + 1) & (STATS_HASH - 1);
      }
      if (!kept) {   // the table is crowded: straight to the global entry
        const long long ge = base + l - 1;
        if (ge < capacity)
          stats_add_global(stats + ge, (int)area, y, x0 + (int)xs, y, x0 + (int)xe, first,
                           (unsigned long long)y * area,
                           (unsigned long long)sxs + (unsigned long long)x0 * area);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < STATS_HASH; i += STATS_NT) {
    const int l = hkey[i];
    if (l == 0) continue;
    const long long ge = base + l - 1;
    if (ge >= capacity) continue;
    const int area = harea[i] & (EDGE_BIT - 1);
    const int first = hfirst[i];
    const int ymin = div_w(first, g);
    const unsigned long long sy = (unsigned long long)hsy[i] + (unsigned long long)y0 * area;
    const unsigned long long sx = (unsigned long long)hsx[i] + (unsigned long long)x0 * area;
    if (harea[i] & EDGE_BIT) {
      stats_add_global(stats + ge, area, ymin, x0 + hxmin[i], hymax[i], x0 + hxmax[i], first, sy, sx);
    } else {   // wholly inside this area: this block is the entry's only writer
      ccl_region_stat r;
      r.area = area;
      r.y_min = ymin;
      r.x_min = x0 + hxmin[i];
      r.y_max = hymax[i];
      r.x_max = x0 + hxmax[i];
      r.first = first;
      r.sum_y = (int64_t)sy;
      r.sum_x = (int64_t)sx;
      stats[ge] = r;
    }
  }
}

}  // namespace ccl_dev
