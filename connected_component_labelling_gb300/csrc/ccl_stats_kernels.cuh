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

// A block per strip of SSEG areas of 256 columns x SR rows, taken one area
// after another.  Blocks are small (four warps), strips short and a run's
// label is read back through L1 rather than kept in shared memory, so that
// many strips are in flight on an SM (twelve): the kernel waits on its
// shared-memory chains more than it issues.  A warp takes one row of the area at a time, a lane 8
// consecutive labels (as in k_tile_local).  The row's runs of equal label
// (run starts from equal-to-left masks) are listed in shared memory and dealt
// out to the warp's lanes, a run each, so that busy rows keep every lane
// working.  Each run updates the area's table (open addressing on the
// label): pixel count and row and column sums relative to the strip's corner
// packed in one 64-bit add, smallest and largest column, largest row, first
// pixel (as row << 11 | column inside the strip), whether any pixel lies on
// an inner edge of the area and whether on one of the strip (a row or column
// with neighbours outside it).  A label on no edge of its area is wholly
// inside it -- a region that reaches outside crosses that edge -- so its
// entry is stored outright; the others are merged into the strip's table,
// whose labels on no edge of the strip are stored outright at the end and the
// rest added to the global entry with atomics: a region crossing many areas
// (a drawing's paper) then costs one global update per strip, not per area.
// A run or area entry that finds no free slot goes straight to the global
// entry.  Every label must be one 4- or 8-connected set, as the labels of
// this library are.
#ifndef CCL_STATS_HASH
#define CCL_STATS_HASH 256
#define CCL_STATS_ROWS 16
#define CCL_STATS_SEGS 4
#define CCL_STATS_NT 128
#endif
constexpr int STATS_HASH = CCL_STATS_HASH;
constexpr int SR = CCL_STATS_ROWS;       // rows of a statistics area
constexpr int SSEG = CCL_STATS_SEGS;     // areas of a strip
constexpr int STRIP_W = SSEG * TW;       // columns of a strip
constexpr int STATS_NT = CCL_STATS_NT;   // threads of a statistics block
constexpr int STATS_NWARPS = STATS_NT / 32;
constexpr int STATS_HASH_BITS = STATS_HASH == 1024 ? 10 : STATS_HASH == 512 ? 9 : 8;
static_assert((1 << STATS_HASH_BITS) == STATS_HASH, "a power of two");
static_assert(STRIP_W <= 2048 && SR <= 16, "strip columns fit 11 bits, rows 4, in the packed first pixel");
// the packed sums of a table slot: column sum (bits 0..25), row sum (26..45),
// pixel count (46..63), all relative to the strip's corner.  A strip's pixels
// keep each field below its top: sum of columns <= SR * STRIP_W^2 / 2 < 2^26,
// of rows <= STRIP_W * SR^2 / 2 < 2^20, count <= SR * STRIP_W < 2^18.
constexpr int ACC_Y = 26, ACC_N = 46;
constexpr int FIRST_ROW_SHIFT = 11;
constexpr uint8_t EDGE_AREA = 1, EDGE_STRIP = 2;

struct StatsTable {
  int key[STATS_HASH], xmin[STATS_HASH], xmax[STATS_HASH], ymax[STATS_HASH], first[STATS_HASH];
  unsigned long long acc[STATS_HASH];
  uint8_t edge[STATS_HASH];
};

__device__ __forceinline__ void table_clear(StatsTable& t, int i) {
  t.key[i] = 0;   // labels start at 1
  t.xmin[i] = INT_MAX;
  t.xmax[i] = -1;
  t.ymax[i] = -1;
  t.first[i] = INT_MAX;
  t.acc[i] = 0ull;
  t.edge[i] = 0;
}

// merge one partial into label l's slot; false when the table is crowded
__device__ __forceinline__ bool table_add(StatsTable& t, int l, unsigned long long acc, int xmin, int xmax,
                                          int ymax, int first, uint8_t edge) {
  unsigned h = ((unsigned)l * 2654435761u) >> (32 - STATS_HASH_BITS);
  for (int probe = 0; probe < 16; ++probe) {
    const int prev = atomicCAS(&t.key[h], 0, l);
    if (prev == 0 || prev == l) {
      atomicAdd(&t.acc[h], acc);
      atomicMin(&t.xmin[h], xmin);
      atomicMax(&t.xmax[h], xmax);
      atomicMax(&t.ymax[h], ymax);
      atomicMin(&t.first[h], first);
      if (edge) atomicOr(reinterpret_cast<unsigned*>(&t.edge[h & ~3u]), (unsigned)edge << (8 * (h & 3u)));
      return true;
    }
    h = (h + 1) & (STATS_HASH - 1);
  }
  return false;
}

// a partial of label l (strip-relative, strip corner (y0, x0)) into its global entry
__device__ __forceinline__ void partial_to_global(ccl_region_stat* e, unsigned long long acc, int xmin, int xmax,
                                                  int ymax, int first, int y0, int x0, const Geom& g) {
  const int area = (int)(acc >> ACC_N);
  const unsigned long long sy = ((acc >> ACC_Y) & ((1ull << (ACC_N - ACC_Y)) - 1ull)) +
                                (unsigned long long)y0 * area;
  const unsigned long long sx = (acc & ((1ull << ACC_Y) - 1ull)) + (unsigned long long)x0 * area;
  const int ymin = y0 + (first >> FIRST_ROW_SHIFT);
  stats_add_global(e, area, ymin, x0 + xmin, ymax, x0 + xmax, ymin * g.W + x0 + (first & (STRIP_W - 1)),
                   sy, sx);
}

__device__ __forceinline__ void partial_store(ccl_region_stat* e, unsigned long long acc, int xmin, int xmax,
                                              int ymax, int first, int y0, int x0, const Geom& g) {
  ccl_region_stat r;
  r.area = (int)(acc >> ACC_N);
  r.y_min = y0 + (first >> FIRST_ROW_SHIFT);
  r.x_min = x0 + xmin;
  r.y_max = ymax;
  r.x_max = x0 + xmax;
  r.first = r.y_min * g.W + x0 + (first & (STRIP_W - 1));
  r.sum_y = (int64_t)(((acc >> ACC_Y) & ((1ull << (ACC_N - ACC_Y)) - 1ull)) + (unsigned long long)y0 * r.area);
  r.sum_x = (int64_t)((acc & ((1ull << ACC_Y) - 1ull)) + (unsigned long long)x0 * r.area);
  *e = r;
}

__global__ void __launch_bounds__(STATS_NT, STATS_NT == 256 ? 6 : 12) k_region_stats(const int32_t* __restrict__ labels,
                                                     const int32_t* __restrict__ n_regions,
                                                     const long long* __restrict__ off,
                                                     ccl_region_stat* stats, long long capacity,
                                                     Geom g, int stripsX, int* status) {
  __shared__ StatsTable ta, ts;                               // the area's and the strip's tables
  __shared__ uint16_t runS[STATS_NWARPS][TW + 1];             // its runs' first columns
  // some partial went straight to a global entry (a crowded table): then a
  // label of the strip's table may have global partials too, so none of that
  // table's entries is stored outright
  __shared__ int spilled;
  for (int i = threadIdx.x; i < STATS_HASH; i += STATS_NT) {
    table_clear(ta, i);
    table_clear(ts, i);
  }
  if (threadIdx.x == 0) spilled = 0;
  __syncthreads();
  // block -> image, strip row, strip column
  const int stripsY = (int)(((long long)g.H + SR - 1) / SR);
  const long long perImage = (long long)stripsY * stripsX;
  const int b = (int)(blockIdx.x / perImage);
  const int rest = (int)(blockIdx.x - (long long)b * perImage);
  const int sy = rest / stripsX, sxi = rest - sy * stripsX;
  const int y0 = sy * SR, y1 = y0 + min(SR, g.H - y0) - 1;                          // rows y0..y1
  const int x0 = sxi * STRIP_W, sw = (int)min((long long)STRIP_W, (long long)g.W - x0);   // columns
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const int nb = n_regions[b];
  const long long base = off[b];
  const int32_t* li = labels + (long long)b * g.HW;
  const bool topIn = y0 > 0, botIn = y1 < g.H - 1;   // rows with neighbours outside
  const bool stripL = x0 > 0, stripR = (long long)x0 + sw < g.W;
  uint16_t* L = runS[warp];
  const int nseg = (sw + TW - 1) / TW;
  for (int s = 0; s < nseg; ++s) {
    const int ax0 = s * TW, aw = min(TW, sw - ax0);   // the area: strip columns ax0 ..
    const bool areaL = ax0 > 0 || stripL, areaR = ax0 + aw < sw || stripR;
    const int nval = max(0, min(PX, aw - xl));
    const bool vec = g.vec_out && nval == PX;
    const unsigned vmask = (1u << nval) - 1u;
    for (int y = y0 + warp; y <= y1; y += STATS_NWARPS) {
      const int32_t* row = li + (long long)y * g.W + x0 + ax0 + xl;
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
      const int vl = __shfl_up_sync(FULL, v[PX - 1], 1);
      unsigned same = (lane > 0 && v[0] == vl) ? 1u : 0u;
#pragma unroll
      for (int j = 1; j < PX; ++j) same |= (v[j] == v[j - 1] ? 1u : 0u) << j;
      unsigned starts = vmask & ~same;
      // the row's runs listed in order (a run's label is read back through L1)
      const int ns = __popc(starts);
      int inc = ns;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += t;
      }
      const int nrun = __shfl_sync(FULL, inc, 31);
      int pos = inc - ns;
      while (starts) {
        const int j = __ffs(starts) - 1;
        starts &= starts - 1;
        L[pos++] = (uint16_t)(xl + j);
      }
      if (lane == 0) L[nrun] = (uint16_t)aw;   // the end of the last run
      __syncwarp();
      const bool edgeRow = (y == y0 && topIn) || (y == y1 && botIn);
      for (int k = lane; k < nrun; k += 32) {
        const int l = __ldg(row - xl + L[k]);
        if (l == 0) continue;
        if (l < 0 || l > nb) {
          raise_flag(status, FLAG_BAD_LABEL);
          continue;
        }
        const int xs = ax0 + L[k], xe = ax0 + L[k + 1] - 1;   // columns in the strip
        const unsigned n = (unsigned)(xe - xs + 1);
        const unsigned long long sxs = (unsigned long long)((unsigned)(xs + xe) * n / 2u);
        const unsigned long long add = ((unsigned long long)n << ACC_N) |
                                       ((unsigned long long)((unsigned)(y - y0) * n) << ACC_Y) | sxs;
        const bool eA = edgeRow || (xs == ax0 && areaL) || (xe == ax0 + aw - 1 && areaR);
        const bool eS = edgeRow || (xs == 0 && stripL) || (xe == sw - 1 && stripR);
        const uint8_t edge = (eA ? EDGE_AREA : 0) | (eS ? EDGE_STRIP : 0);
        const int firstRel = ((y - y0) << FIRST_ROW_SHIFT) | xs;
        if (!table_add(ta, l, add, xs, xe, y, firstRel, edge)) {
          spilled = 1;
          const long long ge = base + l - 1;   // the table is crowded: straight to the global entry
          if (ge < capacity) partial_to_global(stats + ge, add, xs, xe, y, firstRel, y0, x0, g);
        }
      }
      __syncwarp();
    }
    __syncthreads();
    // the area's labels: wholly inside it -> stored; else into the strip's table
    for (int i = threadIdx.x; i < STATS_HASH; i += STATS_NT) {
      const int l = ta.key[i];
      if (l != 0) {
        const long long ge = base + l - 1;
        if (ge < capacity) {
          if (!(ta.edge[i] & EDGE_AREA))
            partial_store(stats + ge, ta.acc[i], ta.xmin[i], ta.xmax[i], ta.ymax[i], ta.first[i], y0, x0, g);
          else if (!table_add(ts, l, ta.acc[i], ta.xmin[i], ta.xmax[i], ta.ymax[i], ta.first[i],
                              ta.edge[i] & EDGE_STRIP)) {
            spilled = 1;
            partial_to_global(stats + ge, ta.acc[i], ta.xmin[i], ta.xmax[i], ta.ymax[i], ta.first[i], y0, x0, g);
          }
        }
        table_clear(ta, i);
      }
    }
    __syncthreads();
  }
  // the strip's labels: wholly inside it (and no partial spilled) -> stored;
  // else added to the global entry
  __syncthreads();
  for (int i = threadIdx.x; i < STATS_HASH; i += STATS_NT) {
    const int l = ts.key[i];
    if (l != 0) {
      const long long ge = base + l - 1;
      if (ge < capacity) {
        if ((ts.edge[i] & EDGE_STRIP) || spilled)
          partial_to_global(stats + ge, ts.acc[i], ts.xmin[i], ts.xmax[i], ts.ymax[i], ts.first[i], y0, x0, g);
        else
          partial_store(stats + ge, ts.acc[i], ts.xmin[i], ts.xmax[i], ts.ymax[i], ts.first[i], y0, x0, g);
      }
    }
  }
}

}  // namespace ccl_dev
