// ccl.cu -- connected-component labelling by parallel union-find on sm_103a.
//
// The four stages of "every-colour" (blogs.fablnx.com) ch. 05 -- Start,
// Connect, Collapse, Number -- mapped onto five kernels that keep the
// labels buffer as the only per-pixel memory (ch. 09: 4 bytes of label per
// pixel plus a few bytes of counts per 256 pixels):
//
//   k_tile_local   Start + in-tile Connect + in-tile Collapse for one
//                  TH x TW tile in shared memory.  Runs inside a warp are
//                  found with one ballot (ch. 08 switch 1); each pixel joins
//                  the row above first and skips the joins its left
//                  neighbour already makes (ch. 08 "First, the order of the
//                  joins" and switch 2, Wu-Otoo-Suzuki's scan mask); walks
//                  halve paths with the same atomic minimum (switch 3).
//                  Writes, for every pixel, the image raster index of its
//                  tile-local leader, a bitmap of leaders and a leader count
//                  per 256-pixel chunk of a row.
//   k_seams        Connect across tile seams in global memory: the joins
//                  (same rule) whose partner lies in another tile, united by
//                  atomicMin with retry (ch. 06 Fig. 10; bendabir.com,
//                  "Unions are parallel").  A leader that gets re-pointed
//                  leaves the bitmap and its chunk's count.
//   k_compress     Collapse for the leaders that took part in seam joins:
//                  each points straight at its final leader.
//   scan kernels   Number, first half: exclusive prefix sum of the chunk
//                  counts ("every-colour" ch. 08 switch 5, ch. 12: a prefix
//                  sum in the middle of Number).
//   k_number       Number, second half: a leader's label is 1 + the number
//                  of leaders before it in raster order; every pixel takes its
//                  leader's label.  Written in place over the parent array,
//                  tile by tile, from a shared-memory copy of the tile.
//
// Leaders are always the smallest raster index of their set (the larger
// leader is linked under the smaller, ch. 04), so the final numbering is the
// canonical one: regions numbered in the raster order of their first pixel.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "ccl.h"

namespace {

constexpr int TW = 256;            // tile width  == numbering chunk width
constexpr int LOG_TW = 8;
constexpr int TH = 16;             // tile height
constexpr int TILE = TW * TH;
constexpr int NT = 256;            // threads per block
constexpr int PER_THREAD = TILE / NT;
constexpr int CHUNK = 256;         // pixels of a row counted together
constexpr int SCAN_ITEMS = 16;     // chunk counts per thread in the scan
constexpr int SCAN_BLOCK = NT * SCAN_ITEMS;
constexpr int32_t BG = INT32_MIN;  // background marker in the parent array
constexpr unsigned FULL = 0xffffffffu;

// device status bits
constexpr int FLAG_WALK_CAP = 1;   // a union-find walk or retry loop hit its cap
constexpr int FLAG_INTERNAL = 2;   // an invariant of the numbering pass failed

struct Geom {
  int H, W;
  int tilesX, tilesY;
  int WPR;                 // bitmap words per row   = ceil(W / 32)
  int CPR;                 // numbering chunks per row = ceil(W / 256)
  long long HW;            // pixels per image
  long long tilesPerImage;
};

struct TileCoord {
  int b, tx, y0, x0, th, tw;
};

__device__ __forceinline__ TileCoord tile_coord(const Geom& g) {
  TileCoord t;
  const long long tile = blockIdx.x;
  t.b = (int)(tile / g.tilesPerImage);
  const int rest = (int)(tile - (long long)t.b * g.tilesPerImage);
  const int ty = rest / g.tilesX;
  t.tx = rest - ty * g.tilesX;
  t.y0 = ty * TH;
  t.x0 = t.tx * TW;
  t.th = min(TH, g.H - t.y0);
  t.tw = min(TW, g.W - t.x0);
  return t;
}

__device__ __forceinline__ void raise_flag(int* status, int f) { atomicOr(status, f); }

__device__ __forceinline__ int ld_cg(const int* p) { return __ldcg(p); }

// ------------------------------------------------------------ shared memory
// Union-find over tile-local indices (r * TW + x).  Reads go through a
// volatile pointer so every step sees other threads' links.

__device__ __forceinline__ int find_s(volatile int* par, int x, int cap, int* status) {
  for (int s = 0; s < cap; ++s) {
    const int p = par[x];
    if (p == x) return x;
    const int gp = par[p];
    if (gp == p) return p;
    atomicMin((int*)&par[x], gp);   // path halving: only ever lowers an arrow
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
    const int old = atomicMin((int*)&par[b], a);   // larger leader under smaller
    if (old == b) return;
    b = old;                                         // someone got there first
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// ------------------------------------------------------------ global memory
// Union-find over image raster indices.  Only leaders' slots are ever
// written here: every walk starts at a pixel's tile-local leader, and every
// node after that is a leader too.

__device__ __forceinline__ int find_g(int* P, int x, int cap, int* status) {
  for (int s = 0; s < cap; ++s) {
    const int p = ld_cg(P + x);
    if (p == x) return x;
    const int gp = ld_cg(P + p);
    if (gp == p) return p;
    atomicMin(P + x, gp);
    x = gp;
  }
  raise_flag(status, FLAG_WALK_CAP);
  return x;
}

__device__ __forceinline__ void drop_leader(int b, uint32_t* bm, uint32_t* cnt, const Geom& g) {
  const int by = b / g.W;
  const int bx = b - by * g.W;
  atomicAnd(bm + (size_t)by * g.WPR + (bx >> 5), ~(1u << (bx & 31)));
  atomicSub(cnt + (size_t)by * g.CPR + (bx >> LOG_TW), 1u);
}

__device__ __forceinline__ void union_g(int* P, int a, int b, uint32_t* bm, uint32_t* cnt,
                                        const Geom& g, int cap, int* status) {
  for (int s = 0; s < cap; ++s) {
    a = find_g(P, a, cap, status);
    b = find_g(P, b, cap, status);
    if (a == b) return;
    if (a > b) { const int t = a; a = b; b = t; }
    const int old = atomicMin(P + b, a);
    if (old == b) {            // b stopped being a leader, exactly once
      drop_leader(b, bm, cnt, g);
      return;
    }
    b = old;
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// ------------------------------------------------------------------ kernels

template <typename T, int CONN, bool BIN>
__global__ void __launch_bounds__(NT) k_tile_local(const T* __restrict__ img, int32_t* __restrict__ P,
                                                   uint32_t* __restrict__ bm, uint32_t* __restrict__ cnt,
                                                   Geom g, int cap, int* status) {
  __shared__ T col[TILE];
  __shared__ int par[TILE];
  __shared__ int rowcnt[TH];
  const TileCoord t = tile_coord(g);
  const T* im = img + (long long)t.b * g.HW;
  int32_t* Pi = P + (long long)t.b * g.HW;
  uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  uint32_t* cnti = cnt + (long long)t.b * g.H * g.CPR;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < TH) rowcnt[threadIdx.x] = 0;

  // load the tile (a warp reads 32 consecutive pixels of one row)
#pragma unroll 4
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    T v = 0;
    if (r < t.th && x < t.tw) v = im[(long long)(t.y0 + r) * g.W + t.x0 + x];
    col[i] = v;
  }
  __syncthreads();

  // Start: every pixel points at the first pixel of its run inside the warp
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    const bool valid = r < t.th && x < t.tw;
    const T c = col[i];
    const bool fg = valid && (!BIN || c != 0);
    const bool eqL = fg && x > 0 && col[i - 1] == c;
    const unsigned starts = __ballot_sync(FULL, !(eqL && lane > 0));
    const int rs = 31 - __clz(starts & (FULL >> (31 - lane)));
    par[i] = fg ? (i - lane + rs) : -1;
  }
  __syncthreads();

  // Connect inside the tile: row above first, then (lane 0 only) the left
  // neighbour in the previous warp.  Neighbours outside the tile count as
  // absent here; their joins are made by k_seams.
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    if (!(r < t.th && x < t.tw)) continue;
    const T c = col[i];
    if (BIN && c == 0) continue;
    const bool eqL = x > 0 && col[i - 1] == c;
    if (r > 0) {
      const bool eqU = col[i - TW] == c;
      const bool eqUL = x > 0 && col[i - TW - 1] == c;
      if (CONN == 8) {
        const bool eqUR = x + 1 < t.tw && col[i - TW + 1] == c;
        if (eqU && !eqL) union_s(par, i, i - TW, cap, status);
        if (eqUL && !eqU && !eqL) union_s(par, i, i - TW - 1, cap, status);
        if (eqUR && !eqU) union_s(par, i, i - TW + 1, cap, status);
      } else {
        if (eqU && !(eqL && eqUL)) union_s(par, i, i - TW, cap, status);
      }
    }
    if (lane == 0 && eqL) union_s(par, i, i - 1, cap, status);
  }
  __syncthreads();

  // Collapse inside the tile and write out leaders as image raster indices
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    const bool valid = r < t.th && x < t.tw;
    const int p = par[i];
    const bool fg = valid && p >= 0;
    const int root = fg ? find_s(par, i, cap, status) : -1;
    const unsigned m = __ballot_sync(FULL, fg && root == i);
    if (valid) {
      const int out = fg ? (t.y0 + (root >> LOG_TW)) * g.W + t.x0 + (root & (TW - 1)) : BG;
      Pi[(long long)(t.y0 + r) * g.W + t.x0 + x] = out;
    }
    if (lane == 0 && valid) {
      bmi[(long long)(t.y0 + r) * g.WPR + ((t.x0 + x) >> 5)] = m;
      atomicAdd(&rowcnt[r], __popc(m));
    }
  }
  __syncthreads();
  if (threadIdx.x < t.th)
    cnti[(long long)(t.y0 + threadIdx.x) * g.CPR + t.tx] = (uint32_t)rowcnt[threadIdx.x];
}

// The joins of pixel (y, x) -- same rule as inside a tile, evaluated on the
// true neighbourhood -- whose partner lies outside the pixel's tile.
template <typename T, int CONN, bool BIN>
__device__ __forceinline__ void seam_joins(const T* __restrict__ im, int32_t* P, uint32_t* bm,
                                           uint32_t* cnt, const Geom& g, int y, int x, int y0,
                                           int x0, int cap, int* status) {
  const long long row = (long long)y * g.W;
  const T c = im[row + x];
  if (BIN && c == 0) return;
  const bool hasU = y > 0, hasL = x > 0;
  const bool eqL = hasL && im[row + x - 1] == c;
  const bool eqU = hasU && im[row - g.W + x] == c;
  const bool eqUL = hasU && hasL && im[row - g.W + x - 1] == c;
  const bool eqUR = (CONN == 8) && hasU && x + 1 < g.W && im[row - g.W + x + 1] == c;
  int a = -1;
  auto join = [&](int qy, int qx) {
    if (qy >= y0 && qx >= x0 && qx < x0 + TW) return;   // inside the tile
    if (a < 0) a = ld_cg(P + row + x);
    const int bq = ld_cg(P + (long long)qy * g.W + qx);
    union_g(P, a, bq, bm, cnt, g, cap, status);
  };
  if (CONN == 8) {
    if (eqU && !eqL) join(y - 1, x);
    if (eqUL && !eqU && !eqL) join(y - 1, x - 1);
    if (eqUR && !eqU) join(y - 1, x + 1);
  } else {
    if (eqU && !(eqL && eqUL)) join(y - 1, x);
  }
  if (eqL) join(y, x - 1);
}

template <typename T, int CONN, bool BIN>
__global__ void __launch_bounds__(NT) k_seams(const T* __restrict__ img, int32_t* P, uint32_t* bm,
                                              uint32_t* cnt, Geom g, int cap, int* status) {
  const TileCoord t = tile_coord(g);
  const T* im = img + (long long)t.b * g.HW;
  int32_t* Pi = P + (long long)t.b * g.HW;
  uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  uint32_t* cnti = cnt + (long long)t.b * g.H * g.CPR;
  const int nTop = t.tw, nSide = t.th - 1;
  for (int k = threadIdx.x; k < nTop + 2 * nSide; k += NT) {
    int y, x;
    if (k < nTop) { y = t.y0; x = t.x0 + k; }
    else if (k < nTop + nSide) { y = t.y0 + 1 + (k - nTop); x = t.x0; }
    else { y = t.y0 + 1 + (k - nTop - nSide); x = t.x0 + t.tw - 1; }
    seam_joins<T, CONN, BIN>(im, Pi, bmi, cnti, g, y, x, t.y0, t.x0, cap, status);
  }
}

// Collapse for leaders that took part in seam joins: every such leader's
// tile component touches the tile's border, so walking from the border
// pixels reaches all of them.  Afterwards every pixel's parent is either its
// tile-local leader (untouched since k_tile_local) or its final leader.
__global__ void __launch_bounds__(NT) k_compress(int32_t* P, Geom g, int cap, int* status) {
  const TileCoord t = tile_coord(g);
  int32_t* Pi = P + (long long)t.b * g.HW;
  const int n = 2 * t.tw + 2 * t.th;
  for (int k = threadIdx.x; k < n; k += NT) {
    int y, x;
    if (k < t.tw) { y = t.y0; x = t.x0 + k; }
    else if (k < 2 * t.tw) { y = t.y0 + t.th - 1; x = t.x0 + (k - t.tw); }
    else if (k < 2 * t.tw + t.th) { y = t.y0 + (k - 2 * t.tw); x = t.x0; }
    else { y = t.y0 + (k - 2 * t.tw - t.th); x = t.x0 + t.tw - 1; }
    const long long pi = (long long)y * g.W + x;
    const int r = ld_cg(Pi + pi);
    if (r == BG) continue;
    const int root = find_g(Pi, r, cap, status);
    if (root != r) {
      // both the slot the border pixel points at and the border pixel itself
      // (it may be a re-pointed leader) now point straight at the leader
      atomicMin(Pi + r, root);
      atomicMin(Pi + pi, root);
    }
  }
}

// ---- exclusive prefix sum of the chunk counts (three passes, no waits)

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total) {
  __shared__ uint32_t warp_sums[NT / 32];
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
    uint32_t s = lane < NT / 32 ? warp_sums[lane] : 0;
    uint32_t si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, si, o);
      if (lane >= o) si += y;
    }
    if (lane < NT / 32) warp_sums[lane] = si - s;
    if (lane == NT / 32 - 1) warp_sums[NT / 32 - 1] = si - s, *total = si;
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
  if (b < batch) n_out[b] = (int32_t)(off[(long long)(b + 1) * chunksPerImage] -
                                      off[(long long)b * chunksPerImage]);
}

// label of leader g: 1 + leaders before it in raster order within its image
__device__ __forceinline__ int number_of(int gidx, const uint32_t* bmi, const uint32_t* offi,
                                         uint32_t base0, const Geom& g, int* status) {
  if (gidx < 0 || (long long)gidx >= g.HW) {
    raise_flag(status, FLAG_INTERNAL);
    return 0;
  }
  const int gy = gidx / g.W, gx = gidx - gy * g.W;
  const long long w0 = (long long)gy * g.WPR + ((gx >> LOG_TW) << 3);
  const long long wg = (long long)gy * g.WPR + (gx >> 5);
  uint32_t s = 0;
  for (long long w = w0; w < wg; ++w) s += __popc(bmi[w]);
  s += __popc(bmi[wg] & ((1u << (gx & 31)) - 1u));
  const uint32_t before = offi[(long long)gy * g.CPR + (gx >> LOG_TW)] - base0 + s;
  return (int)(before + 1u);
}

__global__ void __launch_bounds__(NT) k_number(int32_t* P, const uint32_t* __restrict__ bm,
                                               const uint32_t* __restrict__ off, Geom g, int* status) {
  __shared__ int ps[TILE];
  const TileCoord t = tile_coord(g);
  int32_t* Pi = P + (long long)t.b * g.HW;
  const uint32_t* bmi = bm + (long long)t.b * g.H * g.WPR;
  const uint32_t* offi = off + (long long)t.b * g.H * g.CPR;
  const uint32_t base0 = offi[0];
#pragma unroll 4
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    ps[i] = (r < t.th && x < t.tw) ? Pi[(long long)(t.y0 + r) * g.W + t.x0 + x] : BG;
  }
  __syncthreads();
  auto in_tile = [&](int v, int& local) {
    const int vy = v / g.W, vx = v - vy * g.W;
    if (vy < t.y0 || vy >= t.y0 + t.th || vx < t.x0 || vx >= t.x0 + t.tw) return false;
    local = ((vy - t.y0) << LOG_TW) + (vx - t.x0);
    return true;
  };
  // leaders (and leaders re-pointed outside the tile) get their number
  int res[PER_THREAD];
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    res[k] = 0;
    const int v = ps[i];
    if (v == BG || v < 0) continue;
    const int gi = (t.y0 + r) * g.W + t.x0 + x;
    int local;
    if (v == gi) res[k] = number_of(gi, bmi, offi, base0, g, status);
    else if (!in_tile(v, local)) res[k] = number_of(v, bmi, offi, base0, g, status);
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < PER_THREAD; ++k)
    if (res[k] > 0) ps[threadIdx.x + k * NT] = -res[k];
  __syncthreads();
  // everyone else follows at most two arrows inside the tile
#pragma unroll 4
  for (int k = 0; k < PER_THREAD; ++k) {
    const int i = threadIdx.x + k * NT;
    const int r = i >> LOG_TW, x = i & (TW - 1);
    if (!(r < t.th && x < t.tw)) continue;
    int v = ps[i];
    int out = 0;
    if (v == BG) out = 0;
    else if (v < 0) out = -v;
    else {
      int local;
      out = 0;
      for (int hop = 0; hop < 2; ++hop) {
        if (!in_tile(v, local)) break;
        v = ps[local];
        if (v < 0 && v != BG) { out = -v; break; }
      }
      if (out == 0) raise_flag(status, FLAG_INTERNAL);
    }
    Pi[(long long)(t.y0 + r) * g.W + t.x0 + x] = out;
  }
}

// ------------------------------------------------------------------ host

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
int* g_status[MAX_DEVICES] = {nullptr};
cudaMemPool_t g_pool[MAX_DEVICES] = {nullptr};
long long g_walk_cap = 0;   // 0: default

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  Geom g;
  long long nTiles;
  long long nChunks;     // batch * H * CPR
  int nScanBlocks;
  size_t offBm, offCnt, offBsum, total;
};

int make_layout(int batch, int H, int W, Layout* L) {
  Geom& g = L->g;
  g.H = H;
  g.W = W;
  g.tilesX = (W + TW - 1) / TW;
  g.tilesY = (H + TH - 1) / TH;
  g.WPR = (W + 31) / 32;
  g.CPR = (W + CHUNK - 1) / CHUNK;
  g.HW = (long long)H * W;
  g.tilesPerImage = (long long)g.tilesX * g.tilesY;
  L->nTiles = g.tilesPerImage * batch;
  L->nChunks = (long long)batch * H * g.CPR;
  const long long nsb = (L->nChunks + SCAN_BLOCK - 1) / SCAN_BLOCK;
  if (nsb > (1ll << 30) || L->nTiles > (1ll << 31) - 1) return CCL_ERR_TOO_LARGE;
  L->nScanBlocks = (int)nsb;
  size_t o = 0;
  L->offBm = o;
  o = align_up(o + (size_t)batch * H * g.WPR * sizeof(uint32_t), 256);
  L->offCnt = o;
  o = align_up(o + (size_t)(L->nChunks + 1) * sizeof(uint32_t), 256);
  L->offBsum = o;
  o = align_up(o + (size_t)(L->nScanBlocks + 1) * sizeof(uint32_t), 256);
  L->total = o;
  return CCL_OK;
}

int validate(const void* img, int batch, int H, int W, int pb, int conn, int mode,
             const int32_t* labels, const int32_t* n_out, bool* empty) {
  *empty = false;
  if (batch < 0 || H < 0 || W < 0) return CCL_ERR_INVALID_ARG;
  if (pb != 1 && pb != 2 && pb != 4) return CCL_ERR_INVALID_ARG;
  if (conn != 4 && conn != 8) return CCL_ERR_INVALID_ARG;
  if (mode != CCL_MODE_ALL && mode != CCL_MODE_BINARY) return CCL_ERR_INVALID_ARG;
  if ((long long)H * W >= (1ll << 31)) return CCL_ERR_TOO_LARGE;
  if (n_out && ((uintptr_t)n_out & 3)) return CCL_ERR_INVALID_ARG;
  if (batch == 0 || H == 0 || W == 0) {
    *empty = true;
    return CCL_OK;
  }
  if (!img || !labels) return CCL_ERR_INVALID_ARG;
  if (((uintptr_t)img % (uintptr_t)pb) || ((uintptr_t)labels & 3)) return CCL_ERR_INVALID_ARG;
  const uintptr_t n = (uintptr_t)batch * (uintptr_t)H * (uintptr_t)W;
  const uintptr_t ia = (uintptr_t)img, ib = ia + n * (uintptr_t)pb;
  const uintptr_t la = (uintptr_t)labels, lb = la + n * 4;
  if (ia < lb && la < ib) return CCL_ERR_INVALID_ARG;   // overlapping buffers
  return CCL_OK;
}

int device_status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return CCL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_status[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return CCL_ERR_NO_MEMORY;
    if (cudaMemset(p, 0, 256) != cudaSuccess) return CCL_ERR_CUDA;
    g_status[dev] = p;
  }
  *out = g_status[dev];
  return CCL_OK;
}

int device_pool(cudaMemPool_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return CCL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_pool[dev]) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return CCL_ERR_CUDA;
    uint64_t keep = UINT64_MAX;   // keep freed blocks for the next call
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return CCL_OK;
}

template <typename T, int CONN, bool BIN>
void launch_connect(const void* img, int32_t* P, uint32_t* bm, uint32_t* cnt, const Layout& L,
                    int capTile, int capImg, int* status, cudaStream_t st) {
  const unsigned grid = (unsigned)L.nTiles;
  k_tile_local<T, CONN, BIN><<<grid, NT, 0, st>>>((const T*)img, P, bm, cnt, L.g, capTile, status);
  k_seams<T, CONN, BIN><<<grid, NT, 0, st>>>((const T*)img, P, bm, cnt, L.g, capImg, status);
}

template <typename T>
void dispatch_connect(int conn, int mode, const void* img, int32_t* P, uint32_t* bm, uint32_t* cnt,
                      const Layout& L, int capTile, int capImg, int* status, cudaStream_t st) {
  if (conn == 8) {
    if (mode == CCL_MODE_BINARY) launch_connect<T, 8, true>(img, P, bm, cnt, L, capTile, capImg, status, st);
    else launch_connect<T, 8, false>(img, P, bm, cnt, L, capTile, capImg, status, st);
  } else {
    if (mode == CCL_MODE_BINARY) launch_connect<T, 4, true>(img, P, bm, cnt, L, capTile, capImg, status, st);
    else launch_connect<T, 4, false>(img, P, bm, cnt, L, capTile, capImg, status, st);
  }
}

int run(const void* img, int batch, int H, int W, int pb, int conn, int mode, int32_t* labels,
        int32_t* n_out, const Layout& L, void* ws, cudaStream_t st) {
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != CCL_OK) return rc;
  char* base = (char*)ws;
  uint32_t* bm = (uint32_t*)(base + L.offBm);
  uint32_t* cnt = (uint32_t*)(base + L.offCnt);
  uint32_t* bsum = (uint32_t*)(base + L.offBsum);
  long long capT = TILE + 1, capI = L.g.HW + 1;
  const long long user = g_walk_cap;
  if (user > 0) {
    capT = capT < user ? capT : user;
    capI = capI < user ? capI : user;
  }
  const int capTile = (int)capT;
  const int capImg = (int)(capI > INT32_MAX ? INT32_MAX : capI);
  switch (pb) {
    case 1: dispatch_connect<uint8_t>(conn, mode, img, labels, bm, cnt, L, capTile, capImg, status, st); break;
    case 2: dispatch_connect<uint16_t>(conn, mode, img, labels, bm, cnt, L, capTile, capImg, status, st); break;
    default: dispatch_connect<uint32_t>(conn, mode, img, labels, bm, cnt, L, capTile, capImg, status, st); break;
  }
  const unsigned grid = (unsigned)L.nTiles;
  k_compress<<<grid, NT, 0, st>>>(labels, L.g, capImg, status);
  k_scan_reduce<<<L.nScanBlocks, NT, 0, st>>>(cnt, L.nChunks, bsum);
  k_scan_top<<<1, NT, 0, st>>>(bsum, L.nScanBlocks);
  k_scan_down<<<L.nScanBlocks, NT, 0, st>>>(cnt, L.nChunks, bsum);
  if (n_out)
    k_region_counts<<<(batch + 255) / 256, 256, 0, st>>>(cnt, (long long)H * L.g.CPR, batch, n_out);
  k_number<<<grid, NT, 0, st>>>(labels, bm, cnt, L.g, status);
  return cudaPeekAtLastError() == cudaSuccess ? CCL_OK : CCL_ERR_CUDA;
}

int empty_call(int batch, int32_t* n_out, cudaStream_t st) {
  if (n_out && batch > 0)
    if (cudaMemsetAsync(n_out, 0, (size_t)batch * sizeof(int32_t), st) != cudaSuccess)
      return CCL_ERR_CUDA;
  return CCL_OK;
}

}  // namespace

extern "C" {

int ccl_version(void) { return 100; }

const char* ccl_status_string(int s) {
  switch (s) {
    case CCL_OK: return "CCL_OK";
    case CCL_ERR_INVALID_ARG: return "CCL_ERR_INVALID_ARG";
    case CCL_ERR_TOO_LARGE: return "CCL_ERR_TOO_LARGE";
    case CCL_ERR_CUDA: return "CCL_ERR_CUDA";
    case CCL_ERR_NO_MEMORY: return "CCL_ERR_NO_MEMORY";
    case CCL_ERR_DEVICE_LIMIT: return "CCL_ERR_DEVICE_LIMIT";
    default: return "CCL_ERR_UNKNOWN";
  }
}

int ccl_set_option(int option, long long value) {
  if (option != CCL_OPT_WALK_CAP) return CCL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  g_walk_cap = value > 0 ? value : 0;
  return CCL_OK;
}

size_t ccl_workspace_bytes(int batch, int H, int W, int pixel_bytes, int connectivity, int mode) {
  if (batch <= 0 || H <= 0 || W <= 0) return 0;
  if (pixel_bytes != 1 && pixel_bytes != 2 && pixel_bytes != 4) return 0;
  if (connectivity != 4 && connectivity != 8) return 0;
  if (mode != CCL_MODE_ALL && mode != CCL_MODE_BINARY) return 0;
  if ((long long)H * W >= (1ll << 31)) return 0;
  Layout L;
  if (make_layout(batch, H, W, &L) != CCL_OK) return 0;
  return L.total;
}

int ccl_label_ws(const void* img, int batch, int H, int W, int pixel_bytes, int connectivity,
                 int mode, int32_t* labels_i32, int32_t* n_regions_out, void* workspace,
                 size_t workspace_bytes, ccl_stream_t stream) {
  bool empty = false;
  int rc = validate(img, batch, H, W, pixel_bytes, connectivity, mode, labels_i32, n_regions_out,
                    &empty);
  if (rc != CCL_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (empty) return empty_call(batch, n_regions_out, st);
  Layout L;
  rc = make_layout(batch, H, W, &L);
  if (rc != CCL_OK) return rc;
  if (!workspace || ((uintptr_t)workspace & 255)) return CCL_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return CCL_ERR_NO_MEMORY;
  return run(img, batch, H, W, pixel_bytes, connectivity, mode, labels_i32, n_regions_out, L,
             workspace, st);
}

int ccl_label(const void* img, int batch, int H, int W, int pixel_bytes, int connectivity,
              int mode, int32_t* labels_i32, int32_t* n_regions_out, ccl_stream_t stream) {
  bool empty = false;
  int rc = validate(img, batch, H, W, pixel_bytes, connectivity, mode, labels_i32, n_regions_out,
                    &empty);
  if (rc != CCL_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (empty) return empty_call(batch, n_regions_out, st);
  Layout L;
  rc = make_layout(batch, H, W, &L);
  if (rc != CCL_OK) return rc;
  cudaMemPool_t pool;
  rc = device_pool(&pool);
  if (rc != CCL_OK) return rc;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, L.total, pool, st) != cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_NO_MEMORY;
  }
  rc = run(img, batch, H, W, pixel_bytes, connectivity, mode, labels_i32, n_regions_out, L, ws, st);
  if (cudaFreeAsync(ws, st) != cudaSuccess && rc == CCL_OK) rc = CCL_ERR_CUDA;
  return rc;
}

int ccl_label_host(const void* img_host, int batch, int H, int W, int pixel_bytes,
                   int connectivity, int mode, int32_t* labels_host, int32_t* n_regions_host,
                   ccl_stream_t stream) {
  bool empty = false;
  int rc = validate(img_host, batch, H, W, pixel_bytes, connectivity, mode, labels_host,
                    n_regions_host, &empty);
  if (rc != CCL_OK) return rc;
  if (empty) {
    for (int b = 0; b < batch && n_regions_host; ++b) n_regions_host[b] = 0;
    return CCL_OK;
  }
  cudaStream_t st = (cudaStream_t)stream;
  Layout L;
  rc = make_layout(batch, H, W, &L);
  if (rc != CCL_OK) return rc;
  cudaMemPool_t pool;
  rc = device_pool(&pool);
  if (rc != CCL_OK) return rc;
  const size_t npx = (size_t)batch * H * W;
  const size_t imgBytes = align_up(npx * pixel_bytes, 256);
  const size_t labBytes = align_up(npx * 4, 256);
  const size_t nBytes = align_up((size_t)batch * 4, 256);
  char* buf = nullptr;
  if (cudaMallocFromPoolAsync((void**)&buf, imgBytes + labBytes + nBytes + L.total, pool, st) !=
      cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_NO_MEMORY;
  }
  void* dImg = buf;
  int32_t* dLab = (int32_t*)(buf + imgBytes);
  int32_t* dN = (int32_t*)(buf + imgBytes + labBytes);
  void* ws = buf + imgBytes + labBytes + nBytes;
  if (cudaMemcpyAsync(dImg, img_host, npx * pixel_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    rc = CCL_ERR_CUDA;
  if (rc == CCL_OK)
    rc = run(dImg, batch, H, W, pixel_bytes, connectivity, mode, dLab, dN, L, ws, st);
  if (rc == CCL_OK &&
      cudaMemcpyAsync(labels_host, dLab, npx * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    rc = CCL_ERR_CUDA;
  if (rc == CCL_OK && n_regions_host &&
      cudaMemcpyAsync(n_regions_host, dN, (size_t)batch * 4, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess)
    rc = CCL_ERR_CUDA;
  cudaFreeAsync(buf, st);
  const int sync = ccl_last_status(stream);
  return rc != CCL_OK ? rc : sync;
}

int ccl_last_status(ccl_stream_t stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_CUDA;
  }
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != CCL_OK) return rc;
  int h = 0;
  if (cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CCL_ERR_CUDA;
  if (h != 0 && cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return CCL_ERR_CUDA;
  return h != 0 ? CCL_ERR_DEVICE_LIMIT : CCL_OK;
}

}  // extern "C"
