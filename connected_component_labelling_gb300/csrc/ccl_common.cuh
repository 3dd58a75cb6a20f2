// ccl_common.cuh -- constants, tile geometry, pixel loads and memory-order
// helpers shared by the device code of the labelling library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "ccl.h"

namespace ccl_dev {

constexpr int TW = 256;             // tile width == numbering chunk width
constexpr int LOG_TW = 8;
constexpr int TH = 16;              // tile height
constexpr int TILE = TW * TH;       // pixels (and at most runs) of a tile
constexpr int NT = 256;             // threads per tile block
constexpr int NWARPS = NT / 32;
constexpr int RPW = TH / NWARPS;    // consecutive tile rows per warp
constexpr int PX = TW / 32;         // consecutive pixels per lane
constexpr int CHUNK = 256;          // pixels of a row counted together
constexpr int WPT = TW / 32;        // bit-mask words per tile row
constexpr int LRW = TILE / 32;      // leader-run words per tile
constexpr int BLCAP = 2 * TW + 2 * TH;   // border slots per tile (>= border pixels)
constexpr int NBSL = 2 * TW + 2 * TH;    // border pixels of a tile record
constexpr int JCAP = 2 * TW;        // joins of one row (at most two per pixel)
constexpr int SCAN_ITEMS = 16;
constexpr int SCAN_BLOCK = NT * SCAN_ITEMS;
constexpr uint16_t NOSLOT = 0xFFFF; // a background pixel in a border record
constexpr unsigned FULL = 0xffffffffu;
static_assert(PX == 8, "a lane owns 8 pixels");
static_assert(RPW == 2, "a warp owns two consecutive tile rows");
static_assert(TILE <= 4096, "run ids and their rows share 16 bits");
static_assert(NT == TW, "a thread per tile column in the border records");

constexpr int FLAG_WALK_CAP = 1;    // a union-find walk or retry loop hit its cap
constexpr int FLAG_INTERNAL = 2;    // an invariant of the pipeline failed
constexpr int FLAG_STATS_CAP = 4;   // more regions than the statistics array holds
constexpr int FLAG_BAD_LABEL = 8;   // a label outside 0..n of its image, or a negative count
constexpr int FLAG_LABEL_RANGE = 16;   // an image has more regions than int32 labels hold

struct Geom {
  int H, W;
  int tilesX, tilesY;
  int WPR;                      // bit-mask words per image row = ceil(W / 32)
  int CPR;                      // chunks per row = ceil(W / 256) = tilesX
  long long HW;                 // pixels per image
  long long tilesPerImage;
  unsigned long long wmagic;    // exact d / W for 0 <= d < 2^31: (d * wmagic) >> wshift
  int wshift;
  unsigned long long tmagic;    // the same for d / tilesPerImage
  int tshift;
  unsigned long long xmagic;    // the same for d / tilesX
  int xshift;
  // per-tile record sizes of this call, from the full tile's shape
  // (twf = min(256, W) columns, thf = min(16, H) rows)
  int ENT;                      // runs a tile can hold: twf * thf
  int LRT;                      // leader-run words per tile: ceil(ENT / 32)
  int SL;                       // slots per tile: border pixels of a full tile
  int BSLW;                     // border-record entries per tile
  int BOFF, LOFF, ROFF;         // last row, first column, last column in a record
  int SJW, SJL;                 // seam-join words per tile; the first column's start at SJL
  unsigned slotsPerImage;       // tilesPerImage * SL (< 2^32)
  int vec_img;                  // image rows allow 8-pixel vector loads
  int vec_out;                  // label rows allow 16-byte vector stores
  uint32_t bgval;               // background value when background is ignored
};

struct TileCoord {
  int b, tx, ty, y0, x0, th, tw;
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
  t.ty = div_magic(rest, g.xmagic, g.xshift);
  t.tx = rest - t.ty * g.tilesX;
  t.y0 = t.ty * TH;
  t.x0 = t.tx * TW;
  t.th = min(TH, g.H - t.y0);
  t.tw = min(TW, g.W - t.x0);
  return t;
}

__device__ __forceinline__ int div_w(int d, const Geom& g) { return div_magic(d, g.wmagic, g.wshift); }

__device__ __forceinline__ void raise_flag(int* status, int f) { atomicOr(status, f); }

// ------------------------------------------------------------ memory order
// Union-find parents are read while other threads link and halve them.  A
// plain load of such a word is a data race under the CUDA memory model
// ("every-colour", ch. 07 "On the GPU": the fix is an atomic load); these
// are relaxed atomic loads at the scope of the threads that write the word:
// the block for the tile's parents in shared memory, the device for the
// border slots' parents in global memory.

__device__ __forceinline__ int ld_relaxed_cta(const int* p) {
  int v;
  asm volatile("ld.relaxed.cta.shared.b32 %0, [%1];"
               : "=r"(v)
               : "r"((unsigned)__cvta_generic_to_shared(p)));
  return v;
}

__device__ __forceinline__ void st_relaxed_cta(int* p, int v) {
  asm volatile("st.relaxed.cta.shared.b32 [%0], %1;"
               :
               : "r"((unsigned)__cvta_generic_to_shared(p)), "r"(v));
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(__cvta_generic_to_global(p)));
  return v;
}

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

// ------------------------------------------------------------- bit helpers


// bits 0..b of a word (b in 0..31)
__device__ __forceinline__ uint32_t upto(int b) { return (2u << b) - 1u; }

// position of the n-th (0-based) set bit of v, n < popc(v): a binary search
// by population counts of halves
__device__ __forceinline__ int select_bit(uint32_t v, int n) {
  int pos = 0;
  int c = __popc(v & 0xFFFFu);
  if (n >= c) { n -= c; pos += 16; v >>= 16; }
  c = __popc(v & 0xFFu);
  if (n >= c) { n -= c; pos += 8; v >>= 8; }
  c = __popc(v & 0xFu);
  if (n >= c) { n -= c; pos += 4; v >>= 4; }
  c = __popc(v & 0x3u);
  if (n >= c) { n -= c; pos += 2; v >>= 2; }
  if (n >= (int)(v & 1u)) pos += 1;
  return pos;
}

// set bits of the words w[] in the bit range [lo, hi)
__device__ __forceinline__ int range_popc(const uint32_t* w, int lo, int hi) {
  if (hi <= lo) return 0;
  const int a = lo >> 5, z = (hi - 1) >> 5;
  const uint32_t mlo = ~0u << (lo & 31);
  const uint32_t mhi = upto((hi - 1) & 31);
  if (a == z) return __popc(w[a] & mlo & mhi);
  int s = __popc(w[a] & mlo) + __popc(w[z] & mhi);
  for (int i = a + 1; i < z; ++i) s += __popc(w[i]);
  return s;
}

// row of run q: the largest r with rb[r] <= q (rb[0] = 0 <= q < rb[TH])
__device__ __forceinline__ int row_of_run(const int* rb, int q) {
  int r = 0;
#pragma unroll
  for (int s = TH / 2; s > 0; s >>= 1)
    if (rb[r + s] <= q) r += s;
  return r;
}

}  // namespace ccl_dev
