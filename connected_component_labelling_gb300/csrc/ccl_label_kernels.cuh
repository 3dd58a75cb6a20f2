// ccl_label_kernels.cuh -- the labelling kernels (sm_103a).
//
// The four stages of "every-colour" (blogs.fablnx.com) ch. 05 -- Start,
// Connect, Collapse, Number -- over tiles of 256 columns x 16 rows:
//
//   k_tile_local  Start + Connect + Collapse inside one tile.  A lane owns 8
//                 consecutive pixels of a row, a warp two consecutive rows.
//                 Runs of equal colour (cut at the tile's columns) are found
//                 from equal-to-left bit masks (ch. 08 switch 1, the warp
//                 finds the runs); a run is one union-find node, named by its
//                 rank in the tile (row by row, left to right), so that the
//                 node of a pixel is a population count over the row's run
//                 start bits.  Joins go to the row above and skip what the
//                 left neighbour already joins (ch. 08 "First, the order of
//                 the joins" and switch 2); unions link the larger root under
//                 the smaller with an atomic minimum and halve paths (switch
//                 3).  Collapse points every run at its tile-local leader.
//                 Output, compact: a start bit per pixel, the leader of every
//                 run, the tile's leaders as bits in run order, a leader count
//                 per 256-pixel chunk of a row, and for the regions that touch
//                 the tile border a global slot each (its parent entry and the
//                 slot of every border pixel).
//   k_seams       Connect across tile seams: the joins of the same rule whose
//                 partner is in another tile, united over the border slots
//                 with an atomic minimum on (first pixel, slot) pairs, so that
//                 every root is its region's first pixel in raster order
//                 (ch. 06 Fig. 10; bendabir.com, "Unions are parallel").  A
//                 leader that is linked under another leaves the leader bits
//                 and its chunk count.
//   k_scan_*      Number, first part: exclusive prefix sum of the chunk counts
//                 (ch. 08 switch 5; ch. 12, a prefix sum inside Number).
//   k_resolve     Collapse + Number for the border leaders linked across
//                 seams: each walks to its region's root and stores the root's
//                 label for its slot.
//   k_number      Number, last part: a leader's label is 1 + the number of
//                 leaders before it in raster order; every run takes its
//                 leader's label and every pixel its run's.
//
// In the ignoring modes (binary: value 0; or one named value, "every-colour"
// ch. 08 switch 4 "Ignore the paper") pixels equal to Geom::bgval are
// background: label 0, in no run, part of no join.
#pragma once

#include "ccl_common.cuh"

namespace ccl_dev {

// The workspace of one call (device pointers; sizes per image row or tile).
struct Work {
  uint32_t* sm;             // [batch*H][WPR] run start bits (bit x of a row's words)
  uint32_t* fm;             // [batch*H][WPR] foreground bits (ignoring modes only)
  uint32_t* cnt;            // [batch*H*CPR + 1] leaders per chunk, then their offsets
  uint16_t* hdr;            // [nTiles][TH] runs before rows 1..TH (the last: the tile's runs)
  uint16_t* ent;            // [nTiles][ENT] tile-local leader (a run) of every run
  uint32_t* lr;             // [nTiles][LRT] leader bits in run order
  uint16_t* bsl;            // [nTiles][BSLW] slot (in the tile) of every border pixel's leader:
                            //   first row, last row (at BOFF), first column (LOFF), last column (ROFF)
  uint16_t* bls;            // [nTiles][SL] leader run of every slot | its row << 12
  uint32_t* bcnt;           // [nTiles] slots used
  uint32_t* sj;             // [nTiles][SJW] seam joins: first row (a word per lane), first column (at SJL)
  unsigned long long* P;    // [nTiles][SL] parent entry of every slot: key << 32 | parent slot
};
// Slots are numbered inside their image (tile of the image * SL + place in
// the tile): the entries of image b start at index b * slotsPerImage.

// ------------------------------------------------------------ shared memory
// Union-find over the runs of one tile (run ids 0..runs-1).

__device__ __forceinline__ int find_s(int* par, int x, int cap, int* status) {
  CCL_COUNT(CCL_CNT_TILE_WALKS);
  for (int s = 0; s < cap; ++s) {
    CCL_COUNT(CCL_CNT_TILE_STEPS);
    const int p = ld_relaxed_cta(par + x);
    if (p == x) return x;
    const int gp = ld_relaxed_cta(par + p);
    if (gp == p) return p;
    atomicMin(par + x, gp);   // path halving: an arrow only ever moves down
    x = gp;
  }
  raise_flag(status, FLAG_WALK_CAP);
  return x;
}

__device__ __forceinline__ void union_s(int* par, int a, int b, int cap, int* status) {
  for (int s = 0; s < cap; ++s) {
    a = find_s(par, a, cap, status);
    b = find_s(par, b, cap, status);
    if (a == b) return;
    if (a > b) { const int t = a; a = b; b = t; }
    CCL_COUNT(CCL_CNT_TILE_LINKS);
    const int old = atomicMin(par + b, a);   // larger leader under smaller
    if (old == b) return;
    b = old;                                  // someone got there first
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// ------------------------------------------------------------ global memory
// Union-find over the border slots of all tiles.  An entry is the parent's
// key (the image raster index of its leader's first pixel) above the
// parent's slot, so the atomic minimum on an entry links to the parent whose
// region starts first: roots stay their region's first pixel.  A root's
// entry names itself.  Every loaded slot is range-checked before it is
// followed.

constexpr unsigned long long NOENTRY = ~0ull;

// the root's entry (its key << 32 | its slot), or NOENTRY after a fault
__device__ __forceinline__ unsigned long long find_g(unsigned long long* P, uint32_t x, uint32_t n,
                                                     int cap, int* status) {
  CCL_COUNT(CCL_CNT_GLOBAL_WALKS);
  for (int s = 0; s < cap; ++s) {
    CCL_COUNT(CCL_CNT_GLOBAL_STEPS);
    const unsigned long long v = ld_relaxed_gpu(P + x);
    const uint32_t p = (uint32_t)v;
    if (p == x) return v;
    if (p >= n) {
      raise_flag(status, FLAG_INTERNAL);
      return NOENTRY;
    }
    const unsigned long long v2 = ld_relaxed_gpu(P + p);
    const uint32_t gp = (uint32_t)v2;
    if (gp == p) return v2;
    if (gp >= n) {
      raise_flag(status, FLAG_INTERNAL);
      return NOENTRY;
    }
    atomicMin(P + x, v2);   // path halving
    x = gp;
  }
  raise_flag(status, FLAG_WALK_CAP);
  return NOENTRY;
}

// slot s of image b stopped being a leader: its run leaves the leader bits,
// its chunk one count
__device__ __forceinline__ void drop_leader(const Work& wk, uint32_t s, int b, const Geom& g) {
  const long long tile = (long long)b * g.tilesPerImage + s / (uint32_t)g.SL;
  const uint32_t e = wk.bls[(long long)b * g.slotsPerImage + s];
  const int q = e & 0xFFF, r = (int)(e >> 12);
  atomicAnd(wk.lr + tile * g.LRT + (q >> 5), ~(1u << (q & 31)));
  const TileCoord t = tile_coord_of(g, tile);
  atomicSub(wk.cnt + ((long long)b * g.H + t.y0 + r) * g.CPR + t.tx, 1u);
}

// union of slots a and b of image b (entries Pi = P + b * slotsPerImage)
__device__ __forceinline__ void union_g(const Work& wk, unsigned long long* Pi, int img, uint32_t a, uint32_t b,
                                        const Geom& g, int cap, int* status) {
  const uint32_t n = g.slotsPerImage;
  for (int s = 0; s < cap; ++s) {
    const unsigned long long ra = find_g(Pi, a, n, cap, status);
    const unsigned long long rb = find_g(Pi, b, n, cap, status);
    if (ra == NOENTRY || rb == NOENTRY || ra == rb) return;
    const unsigned long long lo = ra < rb ? ra : rb, hi = ra < rb ? rb : ra;
    const uint32_t hs = (uint32_t)hi;
    CCL_COUNT(CCL_CNT_GLOBAL_LINKS);
    const unsigned long long old = atomicMin(Pi + hs, lo);
    if (old == hi) {   // hs stopped being a root, exactly once
      drop_leader(wk, hs, img, g);
      return;
    }
    // hs was linked to `old` meanwhile (and may now point at lo instead):
    // join lo's set with old's
    a = (uint32_t)lo;
    b = (uint32_t)old;
  }
  raise_flag(status, FLAG_WALK_CAP);
}

// ------------------------------------------------------------------ kernels

// Start + Connect + Collapse of one tile; see the file comment.  Held to 32
// registers a thread so that 8 blocks of 256 threads fill an SM.
template <typename T, int CONN, bool BIN>
__global__ void __launch_bounds__(NT, 8) k_tile_local(const T* __restrict__ img, Work wk, Geom g, int cap,
                                                   int* status, long long tile0) {
  __shared__ __align__(16) int par[TILE];                // parent of every run
  __shared__ __align__(16) uint16_t jl[NWARPS][JCAP];    // a row's joins; later the slot of each border leader
  __shared__ uint32_t sw[TH][WPT];                       // run start bits of the rows
  __shared__ uint32_t fw[BIN ? TH : 1][WPT];             // foreground bits (ignoring modes)
  __shared__ int spre[TH][WPT];                          // starts before word m of row r
  __shared__ int rcnt[TH];
  __shared__ int rbS[TH + 1];                            // runs before row r
  __shared__ uint32_t lrs[LRW], bmark[LRW], bcol[LRW];   // leaders; leaders of border regions;
                                                         // runs on the first or last column
  __shared__ int nb;

  const long long tile = tile0 + blockIdx.x;   // launches may cover a band of tiles
  const TileCoord t = tile_coord_of(g, tile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const T* im = img + (long long)t.b * g.HW;
  const long long rowoff0 = (long long)t.b * g.H;

  // every run is its own set; nothing marked yet; rows below the tile empty
  for (int i = threadIdx.x; i < TILE / 4; i += NT)
    reinterpret_cast<int4*>(par)[i] = make_int4(4 * i, 4 * i + 1, 4 * i + 2, 4 * i + 3);
  if (threadIdx.x < LRW) {
    bmark[threadIdx.x] = 0u;
    bcol[threadIdx.x] = 0u;
  }
  if (threadIdx.x == 0) nb = 0;
  if (threadIdx.x < TH * WPT) {
    const int r = threadIdx.x / WPT, m = threadIdx.x % WPT;
    if (r >= t.th) {
      sw[r][m] = 0u;
      spre[r][m] = 0;
      if (BIN) fw[r][m] = 0u;
      if (m == 0) rcnt[r] = 0;
    }
  }
  const int nval = max(0, min(PX, t.tw - xl));
  const unsigned vmask = (1u << nval) - 1u;
  const bool vec = g.vec_img && nval == PX;
  unsigned stm[RPW], fgm[RPW], tdm[RPW];   // per row: starts, foreground, joins
  uint32_t cp[PX];                         // the first row: the second row's row above

  // ---- Start: the runs of the warp's rows and their joins with the row above
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp * RPW + k;
    stm[k] = fgm[k] = tdm[k] = 0u;
    if (r >= t.th) continue;   // warp-uniform
    const int y = t.y0 + r;
    const T* row = im + (long long)y * g.W + t.x0;
    uint32_t c[PX], u[PX];
    load8<T>(row + xl, vec, nval, c);
    const bool up = y > 0;   // a row above exists in the image
    if (k == 0) {
      if (up) {
        load8<T>(row - g.W + xl, vec, nval, u);
      } else {
#pragma unroll
        for (int j = 0; j < PX; ++j) u[j] = 0u;
      }
    } else {
#pragma unroll
      for (int j = 0; j < PX; ++j) u[j] = cp[j];
    }
    // The tile's first row meets the tiles on its left, above-left and
    // above-right in the top seam's joins: the colours of those neighbours.
    uint32_t cE = 0u, ulE = 0u, urE = 0u;
    bool hL = false, hUL = false, hUR = false;
    if (r == 0) {
      if (lane == 0 && t.x0 > 0) {
        hL = true;
        cE = (uint32_t)row[-1];
        if (up) {
          hUL = true;
          ulE = (uint32_t)row[-1 - g.W];
        }
      }
      if (lane == 31 && up && t.tw == TW && t.x0 + TW < g.W) {
        hUR = true;
        urE = (uint32_t)row[TW - g.W];
      }
    }
    unsigned fg = vmask;
    if (BIN) {
#pragma unroll
      for (int j = 0; j < PX; ++j)
        if (c[j] == g.bgval) fg &= ~(1u << j);
    }
    const uint32_t cls = __shfl_up_sync(FULL, c[PX - 1], 1);
    unsigned eq = (lane > 0 ? c[0] == cls : (hL && c[0] == cE)) ? 1u : 0u;
#pragma unroll
    for (int j = 1; j < PX; ++j) eq |= (c[j] == c[j - 1] ? 1u : 0u) << j;
    eq &= fg;
    // the tile's runs begin at its first column whatever lies left of it
    const unsigned starts = fg & ~(lane == 0 ? (eq & ~1u) : eq);
    unsigned todo = 0u;
    if (up) {   // warp-uniform
      const uint32_t uls = __shfl_up_sync(FULL, u[PX - 1], 1);
      const uint32_t urs = __shfl_down_sync(FULL, u[0], 1);
      unsigned mU = 0u, mUL, mUR = 0u;
#pragma unroll
      for (int j = 0; j < PX; ++j) mU |= (c[j] == u[j] ? 1u : 0u) << j;
      mUL = (lane > 0 ? c[0] == uls : (hUL && c[0] == ulE)) ? 1u : 0u;
#pragma unroll
      for (int j = 1; j < PX; ++j) mUL |= (c[j] == u[j - 1] ? 1u : 0u) << j;
      mU &= fg;
      mUL &= fg;
      // starts on the true neighbourhood (the first row sees across the edge)
      const unsigned s2 = fg & ~eq;
      if (CONN == 8) {
#pragma unroll
        for (int j = 0; j < PX - 1; ++j) mUR |= (c[j] == u[j + 1] ? 1u : 0u) << j;
        const bool inR = lane < 31 && xl + PX < t.tw;
        if (inR ? c[PX - 1] == urs : (hUR && c[PX - 1] == urE)) mUR |= 0x80u;
        mUR &= fg & ((vmask >> 1) | 0x80u);
        // bit j: up, j+8: up-left, j+16: up-right of pixel j
        todo = (mU & s2) | ((mUL & ~mU & s2) << 8) | ((mUR & ~mU) << 16);
      } else {
        todo = mU & ~(eq & mUL);
      }
    }
    if (r == 0) {   // the first row's joins are the top seam's: k_seams makes them
      if (up && lane < g.SJL) wk.sj[tile * g.SJW + lane] = todo;
      todo = 0u;
    }
    stm[k] = starts;
    fgm[k] = fg;
    tdm[k] = todo;
    // the row's start bits as words (lane 4m holds word m) and the starts
    // before each word
    const unsigned w = starts | (__shfl_down_sync(FULL, starts, 1) << 8) |
                       (__shfl_down_sync(FULL, starts, 2) << 16) | (__shfl_down_sync(FULL, starts, 3) << 24);
    unsigned fwd = 0u;
    if (BIN)
      fwd = fg | (__shfl_down_sync(FULL, fg, 1) << 8) | (__shfl_down_sync(FULL, fg, 2) << 16) |
            (__shfl_down_sync(FULL, fg, 3) << 24);
    const int pc = __popc(w);
    int inc = pc;
#pragma unroll
    for (int d = 4; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(FULL, inc, d);
      if (lane >= d) inc += v;
    }
    if ((lane & 3) == 0) {
      const int m = lane >> 2;
      sw[r][m] = w;
      spre[r][m] = inc - pc;
      if (BIN) fw[r][m] = fwd;
      if (xl < t.tw) {
        const long long wi = (rowoff0 + y) * g.WPR + t.tx * WPT + m;
        wk.sm[wi] = w;
        if (BIN) wk.fm[wi] = fwd;
      }
    }
    if (lane == 28) rcnt[r] = inc;
    if (k == 0) {
#pragma unroll
      for (int j = 0; j < PX; ++j) cp[j] = c[j];
    }
  }

  // ---- the left seam's joins (first column against the left tile's last):
  // bit r of word 32 left, 33 up-left, 34 the left pixel's up-right
  if (warp == NWARPS - 1 && t.x0 > 0) {
    const int r = lane;
    const bool v = r < t.th;
    const T* prow = im + (long long)(t.y0 + r) * g.W + t.x0;
    const uint32_t p = v ? (uint32_t)prow[0] : 0u, q = v ? (uint32_t)prow[-1] : 0u;
    const uint32_t pu = __shfl_up_sync(FULL, p, 1), qu = __shfl_up_sync(FULL, q, 1);
    const bool fp = !BIN || p != g.bgval, fq = !BIN || q != g.bgval;
    const bool lb = v && fp && p == q;
    const bool ulb = CONN == 8 && v && r >= 1 && fp && p == qu && p != pu && p != q;
    const bool urb = CONN == 8 && v && r >= 1 && fq && q == pu && q != qu;
    const unsigned bl = __ballot_sync(FULL, lb), bul = __ballot_sync(FULL, ulb), bur = __ballot_sync(FULL, urb);
    if (lane == 0) {
      uint32_t* sj = wk.sj + tile * g.SJW + g.SJL;
      sj[0] = bl;
      sj[1] = bul;
      sj[2] = bur;
    }
  }
  __syncthreads();

  // ---- Connect inside the tile.  The node of pixel x of row r is
  // rb[r] + (starts of row r up to x) - 1.
  const int rc = lane < TH ? rcnt[lane] : 0;
  int rinc = rc;
#pragma unroll
  for (int d = 1; d < TH; d <<= 1) {
    const int v = __shfl_up_sync(FULL, rinc, d);
    if (lane >= d) rinc += v;
  }
  const int rbx = rinc - rc;   // rb[lane] for lane < TH
  const int total = __shfl_sync(FULL, rinc, TH - 1);
  if (warp == 0 && lane <= TH) rbS[lane] = lane < TH ? rbx : total;
  // the runs of the inner rows that touch the first or the last column (all
  // runs of the first and the last row touch the border)
  if (warp == NWARPS - 1) {
    const int r = lane & (TH - 1);
    const int rb0 = __shfl_sync(FULL, rbx, r);
    const int rbs = __shfl_sync(FULL, rbx, (r + 1) & (TH - 1));   // every lane takes part
    const int rbn = r + 1 < TH ? rbs : total;
    if (r > 0 && r < t.th - 1) {
      if (lane < TH) {
        if (sw[r][0] & 1u) atomicOr(&bcol[rb0 >> 5], 1u << (rb0 & 31));
      } else {
        const bool f = !BIN || ((fw[BIN ? r : 0][(t.tw - 1) >> 5] >> ((t.tw - 1) & 31)) & 1u);
        if (f) atomicOr(&bcol[(rbn - 1) >> 5], 1u << ((rbn - 1) & 31));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = warp * RPW + k;
    if (r >= t.th || r == 0) continue;   // warp-uniform
    const int rbr = __shfl_sync(FULL, rbx, r), rbu = __shfl_sync(FULL, rbx, r - 1);
    // A lane would walk its own joins one after another, as often as the
    // busiest lane; instead the row's joins are listed (column | direction
    // << 8) and dealt out to all 32 lanes.
    unsigned todo = tdm[k];
    const int nj = __popc(todo);
    int inc = nj;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(FULL, inc, d);
      if (lane >= d) inc += v;
    }
    const int ntot = __shfl_sync(FULL, inc, 31);
    int pos = inc - nj;
    uint16_t* L = jl[warp];
    while (todo) {
      const int bpos = __ffs(todo) - 1;
      todo &= todo - 1;
      L[pos++] = (uint16_t)((xl + (bpos & 7)) | ((bpos >> 3) << 8));
    }
    __syncwarp();
    for (int q = lane; q < ntot; q += 32) {
      const int e = L[q];
      const int x = e & 0xFF, d = e >> 8;
      const int xb = x + (d == 0 ? 0 : (d == 1 ? -1 : 1));
      const int a = rbr + spre[r][x >> 5] + __popc(sw[r][x >> 5] & upto(x & 31)) - 1;
      const int b = rbu + spre[r - 1][xb >> 5] + __popc(sw[r - 1][xb >> 5] & upto(xb & 31)) - 1;
      union_s(par, a, b, cap, status);
    }
    __syncwarp();
  }
  __syncthreads();

  // ---- Collapse: every run points straight at its tile-local leader; the
  // leaders are the runs that are their own leader.  The first run on the
  // tile border to reach a leader marks it and gives it a slot: a parent
  // entry that names itself, with its key, the raster position of its first
  // pixel (its run's rank in the row stands for the column: ranks keep the
  // order, and x0 + rank < x0 + width, the next tile's first column), and
  // its run and row.
  uint16_t* slotOf = &jl[0][0];   // TILE entries
  const int rbFirst = rbS[1], rbLast = rbS[t.th - 1];   // runs of the first row: [0, rbFirst)
  for (int base = warp * 32; base < total; base += NT) {   // warp-uniform bounds
    const int q = base + lane;
    const bool v = q < total;
    int root = -1;
    bool fresh = false;   // the first border run of its leader
    if (v) {
      root = find_s(par, q, cap, status);
      st_relaxed_cta(par + q, root);
      wk.ent[tile * g.ENT + q] = (uint16_t)root;
      if (q < rbFirst || q >= rbLast || ((bcol[q >> 5] >> (q & 31)) & 1u)) {
        const unsigned bit = 1u << (root & 31);
        fresh = !(atomicOr(&bmark[root >> 5], bit) & bit);
      }
    }
    const unsigned bal = __ballot_sync(FULL, v && root == q);
    if (lane == 0) {
      lrs[base >> 5] = bal;
      wk.lr[tile * g.LRT + (base >> 5)] = bal;
    }
    const unsigned fb = __ballot_sync(FULL, fresh);
    if (fb) {   // warp-uniform
      int k0 = 0;
      if (lane == 0) k0 = atomicAdd(&nb, __popc(fb));
      k0 = __shfl_sync(FULL, k0, 0);
      if (fresh) {
        const int k = k0 + __popc(fb & ((1u << lane) - 1u));
        const int r = row_of_run(rbS, root);
        const long long gi = tile * g.SL + k;   // entry index; the slot's id in its image:
        const uint32_t sid = (uint32_t)(gi - (long long)t.b * g.slotsPerImage);
        const uint32_t key = (uint32_t)((long long)(t.y0 + r) * g.W + t.x0 + (root - rbS[r]));
        wk.P[gi] = ((unsigned long long)key << 32) | sid;
        wk.bls[gi] = (uint16_t)(root | (r << 12));
        slotOf[root] = (uint16_t)k;
      }
    }
  }
  __syncthreads();

  // ---- the tile's records: border pixels' slots (a thread per column for
  // the first and last rows), run bases, slot count, leaders per chunk
  uint16_t* bs = wk.bsl + tile * g.BSLW;
  {
    const int x = threadIdx.x;   // NT == TW
    if (x < t.tw) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = e == 0 ? 0 : t.th - 1;
        const bool f = !BIN || ((fw[BIN ? r : 0][x >> 5] >> (x & 31)) & 1u);
        const int id = rbS[r] + spre[r][x >> 5] + __popc(sw[r][x >> 5] & upto(x & 31)) - 1;
        bs[(e == 0 ? 0 : g.BOFF) + x] = f ? slotOf[par[id]] : NOSLOT;
      }
    }
  }
  if (warp == NWARPS - 1) {
    const int r = lane & (TH - 1);
    if (r < t.th) {
      if (lane < TH) {
        bs[g.LOFF + r] = (sw[r][0] & 1u) ? slotOf[par[rbS[r]]] : NOSLOT;
      } else {
        const bool f = !BIN || ((fw[BIN ? r : 0][(t.tw - 1) >> 5] >> ((t.tw - 1) & 31)) & 1u);
        bs[g.ROFF + r] = f ? slotOf[par[rbS[r + 1] - 1]] : NOSLOT;
      }
    }
  }
  if (threadIdx.x < TH) wk.hdr[tile * TH + threadIdx.x] = (uint16_t)rbS[threadIdx.x + 1];
  if (threadIdx.x == 32) wk.bcnt[tile] = (uint32_t)nb;
  if (threadIdx.x >= 64 && threadIdx.x < 64 + t.th) {
    const int r = threadIdx.x - 64;
    wk.cnt[(rowoff0 + t.y0 + r) * g.CPR + t.tx] = (uint32_t)range_popc(lrs, rbS[r], rbS[r + 1]);
  }
}

// Connect across tile seams: the joins of the same rule as inside a tile,
// taken on the true neighbourhood, whose partner lies in another tile.  A
// tile handles its top seam (its first row against the row above, the join
// bits k_tile_local found) and its left seam (its first column against the
// left tile's last).  One warp per tile, SEAM_WARPS tiles per block, so that
// many tiles' global walks are in flight on an SM at once (the kernel is
// bound by the latency of those dependent loads, not by its few bytes).  The
// warp first keeps every distinct pair of slots to join once (a small hash
// set: along a seam many joins link the same two regions), then its lanes
// unite the kept pairs side by side.
constexpr int SEAM_WARPS = 2;
constexpr int SEAM_HASH = 128;

template <int CONN>
__global__ void __launch_bounds__(32 * SEAM_WARPS) k_seams(Work wk, Geom g, long long nTiles, int cap,
                                                           int* status) {
  __shared__ __align__(16) uint16_t ownS[SEAM_WARPS][TW];        // slots of the first row
  __shared__ __align__(16) uint16_t abS[SEAM_WARPS][TW + 16];    // [8 + x]: slots of the row above
  __shared__ unsigned long long seenS[SEAM_WARPS][SEAM_HASH];
  __shared__ uint16_t jlS[SEAM_WARPS][JCAP];                      // the top seam's joins
  constexpr unsigned long long EMPTY = ~0ull;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, xl = lane * PX;
  const long long tile = (long long)blockIdx.x * SEAM_WARPS + w;
  if (tile >= nTiles) return;   // the whole warp; nothing below waits on the block
  unsigned long long* seen = seenS[w];
#pragma unroll
  for (int i = lane; i < SEAM_HASH; i += 32) seen[i] = EMPTY;
  const TileCoord t = tile_coord_of(g, tile);
  // slots of this image: the tile's first, and the entries' base
  const long long tI = tile - (long long)t.b * g.tilesPerImage;   // tile in its image
  const unsigned long long S = (unsigned long long)tI * g.SL;
  unsigned long long* Pi = wk.P + (long long)t.b * g.slotsPerImage;
  __syncwarp();

  // keep a pair of slots once; unite at once when the set is crowded
  auto keep = [&](unsigned long long a, unsigned long long b, bool ok) {
    if (!ok) {   // a join between pixels whose leaders have no slot
      raise_flag(status, FLAG_INTERNAL);
      return;
    }
    if (a == b) return;
    const unsigned long long key = a < b ? (a << 32) | b : (b << 32) | a;
    unsigned h = (unsigned)((key * 0x9E3779B97F4A7C15ull) >> 40) & (SEAM_HASH - 1);
    for (int probe = 0; probe < 8; ++probe) {
      const unsigned long long prev = atomicCAS(&seen[h], EMPTY, key);
      if (prev == EMPTY) CCL_COUNT(CCL_CNT_SEAM_PAIRS);
      if (prev == EMPTY || prev == key) return;
      h = (h + 1) & (SEAM_HASH - 1);
    }
    union_g(wk, Pi, t.b, (uint32_t)a, (uint32_t)b, g, cap, status);
  };

  // ---- top seam
  if (t.y0 > 0) {
    const unsigned todo0 = lane < g.SJL ? wk.sj[tile * g.SJW + lane] : 0u;
    if (__any_sync(FULL, todo0 != 0u)) {
      const long long ta = tile - g.tilesX;   // the tile above (always full height)
      if (xl < t.tw) {
        *reinterpret_cast<uint4*>(&ownS[w][xl]) = *reinterpret_cast<const uint4*>(wk.bsl + tile * g.BSLW + xl);
        *reinterpret_cast<uint4*>(&abS[w][8 + xl]) =
            *reinterpret_cast<const uint4*>(wk.bsl + ta * g.BSLW + g.BOFF + xl);
      }
      if (lane == 0) abS[w][7] = t.tx > 0 ? wk.bsl[(ta - 1) * g.BSLW + g.BOFF + TW - 1] : NOSLOT;
      if (lane == 31) abS[w][8 + TW] = t.tx + 1 < g.tilesX ? wk.bsl[(ta + 1) * g.BSLW + g.BOFF] : NOSLOT;
      // the joins listed (column | direction << 8) and dealt out to all
      // lanes, as inside a tile: a lane's own joins would take as long as
      // the busiest lane's
      const int nj = __popc(todo0);
      int inc = nj;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += v;
      }
      const int ntot = __shfl_sync(FULL, inc, 31);
      int pos = inc - nj;
      uint16_t* Lj = jlS[w];
      unsigned todo = todo0;
      while (todo) {
        const int bpos = __ffs(todo) - 1;
        todo &= todo - 1;
        Lj[pos++] = (uint16_t)((xl + (bpos & 7)) | ((bpos >> 3) << 8));
      }
      __syncwarp();
      for (int q = lane; q < ntot; q += 32) {
        const int e = Lj[q];
        const int x = e & 0xFF, d = e >> 8;
        const int xb = x + (d == 0 ? 0 : (d == 1 ? -1 : 1));
        const unsigned sa = ownS[w][x], sb = abS[w][8 + xb];
        const long long tb = xb < 0 ? ta - 1 : (xb >= TW ? ta + 1 : ta);
        keep(S + sa, (unsigned long long)(tb - (long long)t.b * g.tilesPerImage) * g.SL + sb,
             sa != NOSLOT && sb != NOSLOT);
      }
    }
  }
  // ---- left seam
  if (t.x0 > 0) {
    const uint32_t* sj = wk.sj + tile * g.SJW + g.SJL;
    const uint32_t bl = sj[0], bul = sj[1], bur = sj[2];
    const int r = lane;
    const bool v = r < t.th;
    const unsigned so = v ? wk.bsl[tile * g.BSLW + g.LOFF + r] : NOSLOT;
    const unsigned sl = v ? wk.bsl[(tile - 1) * g.BSLW + g.ROFF + r] : NOSLOT;
    const unsigned sou = __shfl_up_sync(FULL, so, 1), slu = __shfl_up_sync(FULL, sl, 1);
    const unsigned long long SL = S - g.SL;   // the left tile's first slot
    if (v && ((bl >> r) & 1u)) keep(S + so, SL + sl, so != NOSLOT && sl != NOSLOT);
    if (CONN == 8 && v && ((bul >> r) & 1u)) keep(S + so, SL + slu, so != NOSLOT && slu != NOSLOT);
    if (CONN == 8 && v && ((bur >> r) & 1u)) keep(SL + sl, S + sou, sl != NOSLOT && sou != NOSLOT);
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
    union_g(wk, Pi, t.b, (uint32_t)(key >> 32), (uint32_t)key, g, cap, status);
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

// regions per image (offsets are modulo 2^32; a count that int32 cannot
// hold is flagged)
__global__ void k_region_counts(const uint32_t* off, long long chunksPerImage, int batch, int32_t* n_out,
                                int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) {
    const uint32_t n = off[(long long)(b + 1) * chunksPerImage] - off[(long long)b * chunksPerImage];
    if (n > (uint32_t)INT_MAX) raise_flag(status, FLAG_LABEL_RANGE);
    n_out[b] = (int32_t)min(n, (uint32_t)INT_MAX);
  }
}

// label of the region whose root is slot s of image b: 1 + the leaders
// before its run in its chunk + the chunk's offset in its image
__device__ __forceinline__ int label_of_root(const Work& wk, uint32_t s, int b, const Geom& g, int* status) {
  const long long tile = (long long)b * g.tilesPerImage + s / (uint32_t)g.SL;
  const uint32_t e = wk.bls[(long long)b * g.slotsPerImage + s];
  const int q = e & 0xFFF, r = (int)(e >> 12);
  const TileCoord t = tile_coord_of(g, tile);
  const int rb = r == 0 ? 0 : wk.hdr[tile * TH + r - 1];
  const uint32_t* lw = wk.lr + tile * g.LRT;
  if (!((__ldcg(lw + (q >> 5)) >> (q & 31)) & 1u)) raise_flag(status, FLAG_INTERNAL);   // a root leads
  const int rank = range_popc(lw, rb, q);
  const long long img0 = (long long)b * g.H * g.CPR;
  const uint32_t lab = wk.cnt[img0 + (long long)(t.y0 + r) * g.CPR + t.tx] - wk.cnt[img0] + (uint32_t)rank + 1u;
  if (lab > (uint32_t)INT_MAX) raise_flag(status, FLAG_LABEL_RANGE);
  return (int)lab;
}

constexpr int RESOLVE_WARPS = 2;   // tiles (a warp each) per block: small blocks free their slot sooner;
                                   // held to 32 registers so that 32 blocks (64 warps) fit an SM

// The label found for a leader linked across a seam (run q of its tile)
// waits in the labels buffer, inside that tile (q < the tile's pixels), until
// k_number reads it back before it writes the tile.
__device__ __forceinline__ long long parked_label_index(const TileCoord& t, const Geom& g, int q) {
  const int ry = q / t.tw;
  return ((long long)t.b * g.H + t.y0 + ry) * g.W + t.x0 + (q - ry * t.tw);
}

// Collapse + Number for the border leaders linked across seams (a warp per
// tile, a lane per slot): each walks to its region's root and parks the
// root's label for its slot.  After k_seams an entry changes only here, and
// only to carry its region's label: label << 32 | LABEL_MARK (no slot has
// that id: an image has fewer than 2^32 - 1 slots).  The first walker to
// reach a root labels the root, and every walker labels the slot it started
// from, so that later walks stop at the first labelled entry they meet.
constexpr uint32_t LABEL_MARK = 0xFFFFFFFFu;

__global__ void __launch_bounds__(32 * RESOLVE_WARPS, 32) k_resolve(Work wk, int32_t* labels, Geom g,
                                                                long long nTiles, int cap, int* status) {
  const long long tile = (long long)blockIdx.x * RESOLVE_WARPS + (threadIdx.x >> 5);
  if (tile >= nTiles) return;
  const int lane = threadIdx.x & 31;
  const TileCoord t = tile_coord_of(g, tile);
  unsigned long long* Pi = wk.P + (long long)t.b * g.slotsPerImage;
  const uint32_t n = g.slotsPerImage;
  const uint32_t s0 = (uint32_t)((tile - (long long)t.b * g.tilesPerImage) * g.SL);
  const int count = min((int)wk.bcnt[tile], g.SL);
  for (int k = lane; k < count; k += 32) {
    const uint32_t s = s0 + k;
    unsigned long long v = ld_relaxed_gpu(Pi + s);
    // still a leader (maybe labelled by a walker already): k_number labels it
    if ((uint32_t)v == s || (uint32_t)v == LABEL_MARK) continue;
    CCL_COUNT(CCL_CNT_RESOLVE_STEPS);
    const int q = wk.bls[tile * g.SL + k] & 0xFFF;
    uint32_t x = (uint32_t)v;
    int st = 0;
    for (; st < cap; ++st) {   // to the root, or to a node already labelled
      if (x >= n) break;
      v = ld_relaxed_gpu(Pi + x);
      if ((uint32_t)v == LABEL_MARK || (uint32_t)v == x) break;
      x = (uint32_t)v;
    }
    if (st == cap || x >= n) {
      raise_flag(status, st == cap ? FLAG_WALK_CAP : FLAG_INTERNAL);
      continue;
    }
    int lab;
    if ((uint32_t)v == LABEL_MARK) {
      lab = (int)(v >> 32);
    } else {
      lab = label_of_root(wk, x, t.b, g, status);
      atomicCAS(Pi + x, v, ((unsigned long long)(uint32_t)lab << 32) | LABEL_MARK);
    }
    // this slot carries the label from now on: later walks through it stop here
    atomicExch(Pi + s, ((unsigned long long)(uint32_t)lab << 32) | LABEL_MARK);
    labels[parked_label_index(t, g, q)] = lab;
  }
}

// Number: the tile's leaders take 1 + the leaders before them in raster
// order (chunk offset + rank among the chunk's leaders), leaders linked
// across a seam the label k_resolve found; every run takes its leader's
// label and every pixel its run's.
// Number is bound by the latency of each tile's records (loads, then three
// barriers), so its blocks are small: four warps, four rows each, and twelve
// tiles in flight on an SM (shared memory is the limit; eleven in the binary
// mode, whose foreground bits take more).
constexpr int NUM_NT = 128;   // threads of a Number block

template <bool BIN>
__global__ void __launch_bounds__(NUM_NT, NUM_NT == 256 ? 8 : 12) k_number(Work wk, int32_t* labels, Geom g,
                                                                     int* status, long long tile0) {
  __shared__ __align__(16) int runLab[TILE];
  __shared__ uint32_t swS[TH][WPT];
  __shared__ uint32_t fwS[BIN ? TH : 1][WPT];
  __shared__ int spS[TH][WPT];
  __shared__ uint32_t lrS[LRW];
  __shared__ int rbS[TH + 1];
  __shared__ uint32_t offS[TH];
  constexpr int NTN = NUM_NT, RPWN = TH / (NTN / 32);   // rows a warp writes
  constexpr int PRE = 768 / NTN;   // runs a thread prefetches the leader of
  const long long tile = tile0 + blockIdx.x;   // launches may cover a band of tiles
  const TileCoord t = tile_coord_of(g, tile);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, xl = lane * PX;
  const long long rowoff0 = (long long)t.b * g.H;
  const uint16_t* ent = wk.ent + tile * g.ENT;
  // every load of the tile's records is issued before the first barrier
  // (entries past the tile's runs are read but never used): the leaders of
  // the first PRE * NTN runs, and the leader-bit words holding those runs
  const int total = __ldg(wk.hdr + tile * TH + TH - 1);
  int pe[PRE];
  uint32_t pl[PRE];
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int q = tid + i * NTN;
    pe[i] = q < g.ENT ? __ldg(ent + q) : 0;
    pl[i] = q < g.ENT ? __ldg(wk.lr + tile * g.LRT + (q >> 5)) : 0u;
  }
  if (tid < TH * WPT) {   // the rows' start (and foreground) bits, prefix counts per word
    const int r = tid / WPT, m = tid % WPT;
    uint32_t w = 0u, f = 0u;
    if (r < t.th && m * 32 < t.tw) {
      const long long wi = (rowoff0 + t.y0 + r) * g.WPR + t.tx * WPT + m;
      w = __ldg(wk.sm + wi);
      if (BIN) f = __ldg(wk.fm + wi);
    }
    const int pc = __popc(w);
    int inc = pc;
#pragma unroll
    for (int d = 1; d < WPT; d <<= 1) {
      const int v = __shfl_up_sync(FULL, inc, d);
      if ((lane & (WPT - 1)) >= d) inc += v;
    }
    swS[r][m] = w;
    spS[r][m] = inc - pc;
    if (BIN) fwS[r][m] = f;
  }
  // the leader-bit words, run bases and chunk offsets: a thread each (the
  // threads past the rows' words, or all of a block of TH * WPT threads)
  static_assert(NTN == TH * WPT || NTN == 2 * TH * WPT, "loaders of the tile's records");
  if (NTN == TH * WPT || tid >= TH * WPT) {
    const int i = NTN == TH * WPT ? tid : tid - TH * WPT;
    if (i < g.LRT) lrS[i] = __ldg(wk.lr + tile * g.LRT + i);
    if (i < TH) rbS[i + 1] = __ldg(wk.hdr + tile * TH + i);
    if (i == TH) rbS[0] = 0;
    if (i >= 32 && i < 32 + TH) {
      const int r = i - 32;
      const long long img0 = rowoff0 * g.CPR;
      offS[r] = r < t.th ? __ldg(wk.cnt + (rowoff0 + t.y0 + r) * g.CPR + t.tx) - __ldg(wk.cnt + img0) : 0u;
    }
  }
  // leaders linked across a seam (their own leader, out of the leader bits):
  // the label k_resolve parked in the tile
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int q = tid + i * NTN;
    if (q < total && pe[i] == q && !((pl[i] >> (q & 31)) & 1u)) runLab[q] = labels[parked_label_index(t, g, q)];
  }
  for (int q = tid + PRE * NTN; q < total; q += NTN)
    if (__ldg(ent + q) == q && !((__ldg(wk.lr + tile * g.LRT + (q >> 5)) >> (q & 31)) & 1u))
      runLab[q] = labels[parked_label_index(t, g, q)];
  __syncthreads();
  // the leaders still in the leader bits, row by row (each row by one warp):
  // 1 + the chunk's offset + the leaders before them in the row
#pragma unroll
  for (int k = 0; k < RPWN; ++k) {
    const int r = warp * RPWN + k;
    if (r >= t.th) continue;   // warp-uniform
    const int re = rbS[r + 1];
    uint32_t lab = offS[r] + 1u;
    for (int q0 = rbS[r]; q0 < re; q0 += 32) {   // warp-uniform bounds
      const int q = q0 + lane;
      const bool lead = q < re && ((lrS[q >> 5] >> (q & 31)) & 1u);
      const unsigned bal = __ballot_sync(FULL, lead);
      if (lead) {
        const uint32_t v = lab + (uint32_t)__popc(bal & ((1u << lane) - 1u));
        if (v > (uint32_t)INT_MAX) raise_flag(status, FLAG_LABEL_RANGE);
        runLab[q] = (int)v;
      }
      lab += (uint32_t)__popc(bal);
    }
  }
  __syncthreads();
  // every other run: its leader's label (a leader linked across a seam holds
  // the label read back above)
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int q = tid + i * NTN;
    if (q < total && pe[i] != q) runLab[q] = runLab[pe[i]];
  }
  for (int q = tid + PRE * NTN; q < total; q += NTN) {
    const int e = __ldg(ent + q);
    if (e != q) runLab[q] = runLab[e];
  }
  __syncthreads();
  const int nval = max(0, min(PX, t.tw - xl));
  const bool vec = g.vec_out && nval == PX;
#pragma unroll
  for (int k = 0; k < RPWN; ++k) {
    const int r = warp * RPWN + k;
    if (r >= t.th) continue;
    const int m = lane >> 2, sh = 8 * (lane & 3);
    const uint32_t w = swS[r][m];
    // the run of the pixel before this lane's first: runs before the row,
    // before the word and before the lane, less one
    int id = rbS[r] + spS[r][m] + __popc(w & ((1u << sh) - 1u)) - 1;
    const unsigned st = (w >> sh) & 0xFFu;
    const unsigned fg = BIN ? (fwS[r][m] >> sh) & 0xFFu : 0xFFu;
    int out[PX];
#pragma unroll
    for (int j = 0; j < PX; ++j) {
      if ((st >> j) & 1u) ++id;
      out[j] = ((fg >> j) & 1u) ? runLab[id & (TILE - 1)] : 0;
    }
    int32_t* orow = labels + (rowoff0 + t.y0 + r) * (long long)g.W + t.x0 + xl;
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

}  // namespace ccl_dev
