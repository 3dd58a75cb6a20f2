// ccl_stats_kernels.cuh -- region statistics after labelling (sm_103a).
#pragma once

#include "ccl_common.cuh"

namespace ccl_dev {

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
