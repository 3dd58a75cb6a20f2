// ccl.cu -- host side of the GB300 connected-component labelling library:
// argument checks, workspace layout, launches and the C ABI of include/ccl.h.
// The kernels and their design notes are in ccl_label_kernels.cuh and
// ccl_stats_kernels.cuh.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "ccl.h"
#include "ccl_label_kernels.cuh"
#include "ccl_stats_kernels.cuh"

namespace {

using namespace ccl_dev;

// ------------------------------------------------------------------ host

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
int* g_status[MAX_DEVICES] = {nullptr};
cudaMemPool_t g_pool[MAX_DEVICES] = {nullptr};
cudaStream_t g_copy[MAX_DEVICES] = {nullptr};   // the host entry point's copy stream
long long g_walk_cap = 0;   // 0: default
std::atomic<long long> g_launches{0};

// ---- optional per-stage CUDA events
constexpr int NSTAGES = 5;
const char* const STAGE_NAMES[NSTAGES] = {"tile_local", "seams", "scan", "resolve", "number"};
struct EventSet {
  int dev;
  cudaEvent_t ev[NSTAGES + 1];
};
bool g_stage_events = false;
std::vector<EventSet> g_free_sets, g_pending_sets;

// Returns an event set to record into, or false when timing is off.
bool take_event_set(EventSet* out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_stage_events) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  for (size_t k = 0; k < g_free_sets.size(); ++k) {
    if (g_free_sets[k].dev == dev) {
      *out = g_free_sets[k];
      g_free_sets.erase(g_free_sets.begin() + k);
      return true;
    }
  }
  out->dev = dev;
  for (int k = 0; k <= NSTAGES; ++k)
    if (cudaEventCreate(&out->ev[k]) != cudaSuccess) return false;
  return true;
}

void keep_event_set(const EventSet& e) {
  std::lock_guard<std::mutex> lk(g_mutex);
  g_pending_sets.push_back(e);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  Geom g;
  long long nTiles;
  long long nChunks;     // batch * H * CPR
  int nScanBlocks;
  size_t offSm, offFm, offCnt, offBsum, offHdr, offEnt, offLr, offBsl, offBls, offBcnt, offSj, offP, total;
};

// exact division by d (1 <= d < 2^31) for dividends below 2^31 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// l = ceil(log2 d), magic = ceil(2^(32+l) / d), n / d = (n * magic) >> (32 + l).
// The magic has at most 33 bits, so the product stays below 2^64.
void magic_divisor(long long d, unsigned long long* magic, int* shift) {
  int l = 0;
  while ((1ll << l) < d) ++l;
  *shift = 32 + l;
  *magic = ((1ull << (32 + l)) + (unsigned long long)d - 1ull) / (unsigned long long)d;
}

// Largest image the labelling accepts: keys (raster indices inside an image)
// are 32-bit, so H*W < 2^32.
constexpr long long MAX_IMAGE_PIXELS = (1ll << 32) - 1;

// `fg`: the ignoring modes, which keep foreground bits too
int make_layout(int batch, int H, int W, bool fg, Layout* L) {
  Geom& g = L->g;
  g.H = H;
  g.W = W;
  // (in 64 bits: W or H may be as large as 2^31 - 1)
  g.tilesX = (int)(((long long)W + TW - 1) / TW);
  g.tilesY = (int)(((long long)H + TH - 1) / TH);
  g.WPR = (int)(((long long)W + 31) / 32);
  g.CPR = g.tilesX;
  g.HW = (long long)H * W;
  g.tilesPerImage = (long long)g.tilesX * g.tilesY;
  L->nTiles = g.tilesPerImage * batch;
  L->nChunks = (long long)batch * H * g.CPR;
  // per-tile records, sized by the full tile of this image shape
  const int twf = W < TW ? W : TW, thf = H < TH ? H : TH;
  const int tw8 = (twf + 7) / 8 * 8;
  g.ENT = twf * thf;
  g.LRT = (g.ENT + 31) / 32;
  g.SL = twf * thf - (twf > 2 ? twf - 2 : 0) * (thf > 2 ? thf - 2 : 0);   // border pixels
  g.BOFF = thf > 1 ? tw8 : 0;            // a one-row tile's last row is its first
  g.LOFF = g.BOFF + tw8;
  g.ROFF = g.LOFF + thf;
  g.BSLW = (g.ROFF + thf + 7) / 8 * 8;   // 16-byte rows
  g.SJL = (twf + PX - 1) / PX;           // a word per lane with pixels, then the first column's 3
  g.SJW = g.SJL + 3;
  const long long spi = g.tilesPerImage * g.SL;
  const long long nsb = (L->nChunks + SCAN_BLOCK - 1) / SCAN_BLOCK;
  // tile indices below 2^31; slot ids inside an image below 2^32
  if (nsb > (1ll << 30) || L->nTiles > (1ll << 31) - 1 || spi >= (1ll << 32)) return CCL_ERR_TOO_LARGE;
  g.slotsPerImage = (unsigned)spi;
  L->nScanBlocks = (int)nsb;
  magic_divisor(W, &g.wmagic, &g.wshift);
  magic_divisor(g.tilesPerImage, &g.tmagic, &g.tshift);
  magic_divisor(g.tilesX, &g.xmagic, &g.xshift);
  g.vec_img = 0;
  g.vec_out = 0;
  g.bgval = 0u;
  const size_t rows = (size_t)batch * H, nt = (size_t)L->nTiles;
  size_t o = 0;
  auto take = [&](size_t* off, size_t bytes) {
    *off = o;
    o = align_up(o + bytes, 256);
  };
  take(&L->offSm, rows * g.WPR * sizeof(uint32_t));
  take(&L->offFm, fg ? rows * g.WPR * sizeof(uint32_t) : 0);
  take(&L->offCnt, (size_t)(L->nChunks + 1) * sizeof(uint32_t));
  take(&L->offBsum, (size_t)(L->nScanBlocks + 1) * sizeof(uint32_t));
  take(&L->offHdr, nt * TH * sizeof(uint16_t));
  take(&L->offEnt, nt * g.ENT * sizeof(uint16_t));
  take(&L->offLr, nt * g.LRT * sizeof(uint32_t));
  take(&L->offBsl, nt * g.BSLW * sizeof(uint16_t));
  take(&L->offBls, nt * g.SL * sizeof(uint16_t));
  take(&L->offBcnt, nt * sizeof(uint32_t));
  take(&L->offSj, nt * g.SJW * sizeof(uint32_t));
  take(&L->offP, nt * g.SL * sizeof(unsigned long long));
  L->total = o;
  return CCL_OK;
}

int validate(const void* img, int batch, int H, int W, int pb, int conn, int mode,
             const int32_t* labels, const int32_t* n_out, bool* empty) {
  *empty = false;
  if (batch < 0 || H < 0 || W < 0) return CCL_ERR_INVALID_ARG;
  if (pb < 1 || pb > 4) return CCL_ERR_INVALID_ARG;
  if (conn != 4 && conn != 8) return CCL_ERR_INVALID_ARG;
  if (mode != CCL_MODE_ALL && mode != CCL_MODE_BINARY) return CCL_ERR_INVALID_ARG;
  if ((long long)H * W > MAX_IMAGE_PIXELS) return CCL_ERR_TOO_LARGE;
  if (n_out && ((uintptr_t)n_out & 3)) return CCL_ERR_INVALID_ARG;
  if (batch == 0 || H == 0 || W == 0) {
    *empty = true;
    return CCL_OK;
  }
  if (!img || !labels) return CCL_ERR_INVALID_ARG;
  // pixels align to their size; 3-byte RGB pixels need no alignment
  if ((pb != 3 && (uintptr_t)img % (uintptr_t)pb) || ((uintptr_t)labels & 3)) return CCL_ERR_INVALID_ARG;
  const uintptr_t n = (uintptr_t)batch * (uintptr_t)H * (uintptr_t)W;
  const uintptr_t ia = (uintptr_t)img, ib = ia + n * (uintptr_t)pb;
  const uintptr_t la = (uintptr_t)labels, lb = la + n * 4;
  if (ia < lb && la < ib) return CCL_ERR_INVALID_ARG;   // overlapping buffers
  if (n_out) {   // the counts are written before the labels: they may share no byte
    const uintptr_t na = (uintptr_t)n_out, nb = na + (uintptr_t)batch * 4;
    if (na < lb && la < nb) return CCL_ERR_INVALID_ARG;
  }
  return CCL_OK;
}

// A caller's workspace must not share bytes with the image, the labels or
// the counts: the kernels write all of it.
bool workspace_overlaps(const void* ws, size_t wsBytes, const void* img, int batch, int H, int W,
                        int pb, const int32_t* labels, const int32_t* n_out) {
  const uintptr_t wa = (uintptr_t)ws, wb = wa + wsBytes;
  const uintptr_t n = (uintptr_t)batch * (uintptr_t)H * (uintptr_t)W;
  auto hit = [&](uintptr_t a, uintptr_t bytes) { return a < wb && wa < a + bytes; };
  return hit((uintptr_t)img, n * (uintptr_t)pb) || hit((uintptr_t)labels, n * 4) ||
         (n_out && hit((uintptr_t)n_out, (uintptr_t)batch * 4));
}

// the current device's copy stream (created once, non-blocking)
int device_copy_stream(cudaStream_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return CCL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_copy[dev]) {
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return CCL_ERR_CUDA;
    g_copy[dev] = s;
  }
  *out = g_copy[dev];
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

// Kernel templates are instantiated for every pixel width (1, 2, 3, 4 bytes),
// connectivity (4, 8) and mode (all, ignoring one value).
#define CCL_DISPATCH(KERNEL, GRID, BLOCK, ...)                                                        \
  do {                                                                                   \
    const unsigned grid_ = (unsigned)(GRID);                                             \
    const unsigned block_ = (unsigned)(BLOCK);                                           \
    const bool bin_ = mode == CCL_MODE_BINARY;                                           \
    if (pb == 1) {                                                                       \
      if (conn == 8) { if (bin_) KERNEL<uint8_t, 8, true><<<grid_, block_, 0, st>>>((const uint8_t*)img, __VA_ARGS__); \
                       else KERNEL<uint8_t, 8, false><<<grid_, block_, 0, st>>>((const uint8_t*)img, __VA_ARGS__); } \
      else { if (bin_) KERNEL<uint8_t, 4, true><<<grid_, block_, 0, st>>>((const uint8_t*)img, __VA_ARGS__); \
             else KERNEL<uint8_t, 4, false><<<grid_, block_, 0, st>>>((const uint8_t*)img, __VA_ARGS__); } \
    } else if (pb == 3) {                                                                \
      if (conn == 8) { if (bin_) KERNEL<Rgb24, 8, true><<<grid_, block_, 0, st>>>((const Rgb24*)img, __VA_ARGS__); \
                       else KERNEL<Rgb24, 8, false><<<grid_, block_, 0, st>>>((const Rgb24*)img, __VA_ARGS__); } \
      else { if (bin_) KERNEL<Rgb24, 4, true><<<grid_, block_, 0, st>>>((const Rgb24*)img, __VA_ARGS__); \
             else KERNEL<Rgb24, 4, false><<<grid_, block_, 0, st>>>((const Rgb24*)img, __VA_ARGS__); } \
    } else if (pb == 2) {                                                                \
      if (conn == 8) { if (bin_) KERNEL<uint16_t, 8, true><<<grid_, block_, 0, st>>>((const uint16_t*)img, __VA_ARGS__); \
                       else KERNEL<uint16_t, 8, false><<<grid_, block_, 0, st>>>((const uint16_t*)img, __VA_ARGS__); } \
      else { if (bin_) KERNEL<uint16_t, 4, true><<<grid_, block_, 0, st>>>((const uint16_t*)img, __VA_ARGS__); \
             else KERNEL<uint16_t, 4, false><<<grid_, block_, 0, st>>>((const uint16_t*)img, __VA_ARGS__); } \
    } else {                                                                             \
      if (conn == 8) { if (bin_) KERNEL<uint32_t, 8, true><<<grid_, block_, 0, st>>>((const uint32_t*)img, __VA_ARGS__); \
                       else KERNEL<uint32_t, 8, false><<<grid_, block_, 0, st>>>((const uint32_t*)img, __VA_ARGS__); } \
      else { if (bin_) KERNEL<uint32_t, 4, true><<<grid_, block_, 0, st>>>((const uint32_t*)img, __VA_ARGS__); \
             else KERNEL<uint32_t, 4, false><<<grid_, block_, 0, st>>>((const uint32_t*)img, __VA_ARGS__); } \
    }                                                                                    \
  } while (0)

// The pipeline's pieces on `st`: `ws` is the workspace (layout L), `status`
// the device word the kernels flag limits in.
struct Pipe {
  const void* img;
  int batch, H, W, pb, conn, mode;
  int32_t* labels;
  int32_t* n_out;
  const Layout* L;
  Work wk;
  uint32_t* bsum;
  Geom g;
  int capTile, capImg;
  int* status;
  cudaStream_t st;
};

Pipe make_pipe(const void* img, int batch, int H, int W, int pb, int conn, int mode, uint32_t bgval,
               int32_t* labels, int32_t* n_out, const Layout& L, void* ws, int* status,
               cudaStream_t st) {
  Pipe q;
  q.img = img;
  q.batch = batch;
  q.H = H;
  q.W = W;
  q.pb = pb;
  q.conn = conn;
  q.mode = mode;
  q.labels = labels;
  q.n_out = n_out;
  q.L = &L;
  char* base = (char*)ws;
  q.wk.sm = (uint32_t*)(base + L.offSm);
  q.wk.fm = (uint32_t*)(base + L.offFm);
  q.wk.cnt = (uint32_t*)(base + L.offCnt);
  q.wk.hdr = (uint16_t*)(base + L.offHdr);
  q.wk.ent = (uint16_t*)(base + L.offEnt);
  q.wk.lr = (uint32_t*)(base + L.offLr);
  q.wk.bsl = (uint16_t*)(base + L.offBsl);
  q.wk.bls = (uint16_t*)(base + L.offBls);
  q.wk.bcnt = (uint32_t*)(base + L.offBcnt);
  q.wk.sj = (uint32_t*)(base + L.offSj);
  q.wk.P = (unsigned long long*)(base + L.offP);
  q.bsum = (uint32_t*)(base + L.offBsum);
  // walk caps: the nodes a walk can visit (runs of a tile; slots of the call)
  long long capT = TILE + 1, capI = (long long)L.g.slotsPerImage + 1;
  const long long user = g_walk_cap;
  if (user > 0) {
    capT = capT < user ? capT : user;
    capI = capI < user ? capI : user;
  }
  q.capTile = (int)capT;
  q.capImg = (int)(capI > INT32_MAX ? INT32_MAX : capI);
  // vector access when every row start keeps the needed alignment
  q.g = L.g;
  q.g.bgval = bgval;
  const uintptr_t ia = (uintptr_t)img;
  if (pb == 1) q.g.vec_img = (W % 8 == 0) && (ia % 8 == 0);
  else if (pb == 2) q.g.vec_img = (W % 8 == 0) && (ia % 16 == 0);
  else if (pb == 3) q.g.vec_img = (W % 8 == 0) && (ia % 8 == 0);   // 24-byte lanes on 8-byte boundaries
  else q.g.vec_img = (W % 4 == 0) && (ia % 16 == 0);
  q.g.vec_out = (W % 8 == 0) && ((uintptr_t)labels % 16 == 0);
  q.status = status;
  q.st = st;
  return q;
}

// Start + Connect + Collapse for tiles [tile0, tile0 + ntiles)
void launch_tile_local(const Pipe& q, long long tile0, long long ntiles) {
  const int pb = q.pb, conn = q.conn, mode = q.mode;
  const void* img = q.img;
  cudaStream_t st = q.st;
  CCL_DISPATCH(k_tile_local, ntiles, NT, q.wk, q.g, q.capTile, q.status, tile0);
}
void launch_seams(const Pipe& q) {
  const unsigned grid = (unsigned)((q.L->nTiles + SEAM_WARPS - 1) / SEAM_WARPS);
  if (q.conn == 8)
    k_seams<8><<<grid, 32 * SEAM_WARPS, 0, q.st>>>(q.wk, q.g, q.L->nTiles, q.capImg, q.status);
  else
    k_seams<4><<<grid, 32 * SEAM_WARPS, 0, q.st>>>(q.wk, q.g, q.L->nTiles, q.capImg, q.status);
}
void launch_scan(const Pipe& q) {
  const Layout& L = *q.L;
  k_scan_reduce<<<L.nScanBlocks, NT, 0, q.st>>>(q.wk.cnt, L.nChunks, q.bsum);
  k_scan_top<<<1, NT, 0, q.st>>>(q.bsum, L.nScanBlocks);
  k_scan_down<<<L.nScanBlocks, NT, 0, q.st>>>(q.wk.cnt, L.nChunks, q.bsum);
  if (q.n_out)
    k_region_counts<<<(q.batch + 255) / 256, 256, 0, q.st>>>(q.wk.cnt, (long long)q.H * L.g.CPR, q.batch,
                                                             q.n_out, q.status);
}
void launch_resolve(const Pipe& q) {
  const Layout& L = *q.L;
  k_resolve<<<(unsigned)((L.nTiles + RESOLVE_WARPS - 1) / RESOLVE_WARPS), 32 * RESOLVE_WARPS, 0, q.st>>>(
      q.wk, q.labels, q.g, L.nTiles, q.capImg, q.status);
}
// Number for tiles [tile0, tile0 + ntiles)
void launch_number(const Pipe& q, long long tile0, long long ntiles) {
  if (q.mode == CCL_MODE_BINARY)
    k_number<true><<<(unsigned)ntiles, NUM_NT, 0, q.st>>>(q.wk, q.labels, q.g, q.status, tile0);
  else
    k_number<false><<<(unsigned)ntiles, NUM_NT, 0, q.st>>>(q.wk, q.labels, q.g, q.status, tile0);
}

// The whole labelling pipeline on `st`; `events` whether the optional
// per-stage events may be recorded.
int run_pipeline(const void* img, int batch, int H, int W, int pb, int conn, int mode,
                 uint32_t bgval, int32_t* labels, int32_t* n_out, const Layout& L, void* ws,
                 int* status, bool events, cudaStream_t st) {
  const Pipe q = make_pipe(img, batch, H, W, pb, conn, mode, bgval, labels, n_out, L, ws, status, st);
  EventSet es;
  const bool timed = events && take_event_set(&es);
  auto mark = [&](int k) {
    if (timed) cudaEventRecord(es.ev[k], st);
  };
  mark(0);
  launch_tile_local(q, 0, L.nTiles);
  mark(1);
  launch_seams(q);
  mark(2);
  launch_scan(q);
  mark(3);
  launch_resolve(q);
  mark(4);
  launch_number(q, 0, L.nTiles);
  mark(5);
  if (timed) keep_event_set(es);
  g_launches += n_out ? 8 : 7;
  return cudaPeekAtLastError() == cudaSuccess ? CCL_OK : CCL_ERR_CUDA;
}

// The host entry point's pipeline.  The image goes up and the labels come
// down in HOST_BANDS bands of whole tile rows on a copy stream `cs`: Start,
// Connect and Collapse of a band run while the next band is copied in, and a
// band's labels are copied out as soon as Number has written them (Number of
// a tile reads and writes only that tile's part of the labels).  Seams, scan
// and resolve need the whole image and run in between.
constexpr int HOST_BANDS = 8;

int run_host_banded(const void* img_host, int batch, int H, int W, int pb, int conn, int mode,
                    int32_t* labels_host, int32_t* n_host, void* dImg, int32_t* dLab, int32_t* dN,
                    const Layout& L, void* ws, int* status, cudaStream_t st, cudaStream_t cs) {
  const Pipe q = make_pipe(dImg, batch, H, W, pb, conn, mode, 0u, dLab, dN, L, ws, status, st);
  const long long tilesY = L.g.tilesY, tilesX = L.g.tilesX;
  const long long tileRows = (long long)batch * tilesY;
  const int K = (int)(tileRows < HOST_BANDS ? tileRows : HOST_BANDS);
  cudaEvent_t ev[2 * HOST_BANDS + 2];
  int made = 0;
  int rc = CCL_OK;
  for (; made < 2 * K + 2; ++made)
    if (cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) != cudaSuccess) {
      rc = CCL_ERR_CUDA;
      break;
    }
  // image rows (counted across the batch) of tile row tr: [first, end)
  auto firstRow = [&](long long tr) {
    const long long b = tr / tilesY, ty = tr - b * tilesY;
    return b * H + ty * TH;
  };
  auto endRow = [&](long long tr) {
    const long long b = tr / tilesY, ty = tr - b * tilesY;
    return b * H + ((ty + 1) * TH < H ? (ty + 1) * TH : H);
  };
  auto bandRows = [&](int k, long long* tr0, long long* tr1) {
    *tr0 = tileRows * k / K;
    *tr1 = tileRows * (k + 1) / K;
  };
  if (rc == CCL_OK) {
    const size_t rowBytes = (size_t)W * pb;
    // the copy stream touches the buffers only after their allocation
    cudaEventRecord(ev[2 * K], st);
    cudaStreamWaitEvent(cs, ev[2 * K], 0);
    for (int k = 0; k < K && rc == CCL_OK; ++k) {
      long long tr0, tr1;
      bandRows(k, &tr0, &tr1);
      const long long r0 = firstRow(tr0), r1 = endRow(tr1 - 1);
      if (cudaMemcpyAsync((char*)dImg + r0 * rowBytes, (const char*)img_host + r0 * rowBytes,
                          (size_t)(r1 - r0) * rowBytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
          cudaEventRecord(ev[k], cs) != cudaSuccess)
        rc = CCL_ERR_CUDA;
    }
    for (int k = 0; k < K && rc == CCL_OK; ++k) {
      long long tr0, tr1;
      bandRows(k, &tr0, &tr1);
      cudaStreamWaitEvent(st, ev[k], 0);
      launch_tile_local(q, tr0 * tilesX, (tr1 - tr0) * tilesX);
    }
    if (rc == CCL_OK) {
      launch_seams(q);
      launch_scan(q);
      launch_resolve(q);
    }
    for (int k = 0; k < K && rc == CCL_OK; ++k) {
      long long tr0, tr1;
      bandRows(k, &tr0, &tr1);
      launch_number(q, tr0 * tilesX, (tr1 - tr0) * tilesX);
      const long long r0 = firstRow(tr0), r1 = endRow(tr1 - 1);
      if (cudaEventRecord(ev[K + k], st) != cudaSuccess || cudaStreamWaitEvent(cs, ev[K + k], 0) != cudaSuccess ||
          cudaMemcpyAsync(labels_host + r0 * W, dLab + r0 * W, (size_t)(r1 - r0) * W * sizeof(int32_t),
                          cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        rc = CCL_ERR_CUDA;
    }
    if (rc == CCL_OK && n_host &&
        cudaMemcpyAsync(n_host, dN, (size_t)batch * sizeof(int32_t), cudaMemcpyDeviceToHost, cs) !=
            cudaSuccess)
      rc = CCL_ERR_CUDA;
    // the buffers are freed on `st` after the last copy
    cudaEventRecord(ev[2 * K + 1], cs);
    cudaStreamWaitEvent(st, ev[2 * K + 1], 0);
    g_launches += 2 * K + 6;   // K tile_local, seams, 3 scans, region counts, resolve, K number
  }
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  if (rc == CCL_OK && cudaPeekAtLastError() != cudaSuccess) rc = CCL_ERR_CUDA;
  return rc;
}

int run(const void* img, int batch, int H, int W, int pb, int conn, int mode, int32_t* labels,
        int32_t* n_out, const Layout& L, void* ws, cudaStream_t st, uint32_t bgval = 0u) {
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != CCL_OK) return rc;
  if (bgval != 0u)
    return run_pipeline(img, batch, H, W, pb, conn, mode, bgval, labels, n_out, L, ws, status,
                        true, st);
  return run_pipeline(img, batch, H, W, pb, conn, mode, 0u, labels, n_out, L, ws, status, true, st);
}

// the ccl_status a device status word stands for
int status_of_flags(int h) {
  if (h & (FLAG_WALK_CAP | FLAG_INTERNAL)) return CCL_ERR_DEVICE_LIMIT;
  if (h & FLAG_LABEL_RANGE) return CCL_ERR_TOO_LARGE;
  if (h & FLAG_STATS_CAP) return CCL_ERR_NO_MEMORY;
  if (h & FLAG_BAD_LABEL) return CCL_ERR_INVALID_ARG;
  return CCL_OK;
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
  std::lock_guard<std::mutex> lk(g_mutex);
  if (option == CCL_OPT_WALK_CAP) {
    g_walk_cap = value > 0 ? value : 0;
    return CCL_OK;
  }
  if (option == CCL_OPT_STAGE_EVENTS) {
    g_stage_events = value != 0;
    return CCL_OK;
  }
  return CCL_ERR_INVALID_ARG;
}

const char* ccl_stage_name(int stage) {
  return (stage >= 0 && stage < NSTAGES) ? STAGE_NAMES[stage] : "";
}

long long ccl_kernel_launches(void) { return g_launches.load(); }

int ccl_stage_times(double* ms_sum, int max_stages, int* n_calls) {
  std::vector<EventSet> sets;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    sets.swap(g_pending_sets);
  }
  double acc[NSTAGES] = {0};
  int rc = NSTAGES;
  for (const EventSet& e : sets) {
    if (cudaEventSynchronize(e.ev[NSTAGES]) != cudaSuccess) rc = -CCL_ERR_CUDA;
    for (int k = 0; k < NSTAGES && rc > 0; ++k) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, e.ev[k], e.ev[k + 1]) != cudaSuccess) rc = -CCL_ERR_CUDA;
      acc[k] += ms;
    }
  }
  if (rc < 0) cudaGetLastError();
  for (int k = 0; k < NSTAGES && k < max_stages && ms_sum; ++k) ms_sum[k] = acc[k];
  if (n_calls) *n_calls = (int)sets.size();
  std::lock_guard<std::mutex> lk(g_mutex);
  for (const EventSet& e : sets) g_free_sets.push_back(e);
  return rc;
}

size_t ccl_workspace_bytes(int batch, int H, int W, int pixel_bytes, int connectivity, int mode) {
  if (batch <= 0 || H <= 0 || W <= 0) return 0;
  if (pixel_bytes < 1 || pixel_bytes > 4) return 0;
  if (connectivity != 4 && connectivity != 8) return 0;
  if (mode != CCL_MODE_ALL && mode != CCL_MODE_BINARY) return 0;
  if ((long long)H * W > MAX_IMAGE_PIXELS) return 0;
  Layout L;
  if (make_layout(batch, H, W, mode == CCL_MODE_BINARY, &L) != CCL_OK) return 0;
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
  rc = make_layout(batch, H, W, mode == CCL_MODE_BINARY, &L);
  if (rc != CCL_OK) return rc;
  if (!workspace || ((uintptr_t)workspace & 255)) return CCL_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return CCL_ERR_NO_MEMORY;
  if (workspace_overlaps(workspace, L.total, img, batch, H, W, pixel_bytes, labels_i32, n_regions_out))
    return CCL_ERR_INVALID_ARG;
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
  rc = make_layout(batch, H, W, mode == CCL_MODE_BINARY, &L);
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

int ccl_label_ignore(const void* img, int batch, int H, int W, int pixel_bytes, int connectivity,
                     uint32_t ignore_value, int32_t* labels_i32, int32_t* n_regions_out,
                     void* workspace, size_t workspace_bytes, ccl_stream_t stream) {
  bool empty = false;
  int rc = validate(img, batch, H, W, pixel_bytes, connectivity, CCL_MODE_BINARY, labels_i32,
                    n_regions_out, &empty);
  if (rc != CCL_OK) return rc;
  if (pixel_bytes < 4 && (ignore_value >> (8 * pixel_bytes)) != 0u) return CCL_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (empty) return empty_call(batch, n_regions_out, st);
  Layout L;
  rc = make_layout(batch, H, W, true, &L);
  if (rc != CCL_OK) return rc;
  if (workspace) {
    if ((uintptr_t)workspace & 255) return CCL_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return CCL_ERR_NO_MEMORY;
    if (workspace_overlaps(workspace, L.total, img, batch, H, W, pixel_bytes, labels_i32,
                           n_regions_out))
      return CCL_ERR_INVALID_ARG;
    int* status = nullptr;
    rc = device_status_ptr(&status);
    if (rc != CCL_OK) return rc;
    return run_pipeline(img, batch, H, W, pixel_bytes, connectivity, CCL_MODE_BINARY, ignore_value,
                        labels_i32, n_regions_out, L, workspace, status, true, st);
  }
  cudaMemPool_t pool;
  rc = device_pool(&pool);
  if (rc != CCL_OK) return rc;
  void* ws = nullptr;
  if (cudaMallocFromPoolAsync(&ws, L.total, pool, st) != cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_NO_MEMORY;
  }
  int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc == CCL_OK)
    rc = run_pipeline(img, batch, H, W, pixel_bytes, connectivity, CCL_MODE_BINARY, ignore_value,
                      labels_i32, n_regions_out, L, ws, status, true, st);
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
  rc = make_layout(batch, H, W, mode == CCL_MODE_BINARY, &L);
  if (rc != CCL_OK) return rc;
  cudaMemPool_t pool;
  rc = device_pool(&pool);
  if (rc != CCL_OK) return rc;
  const size_t npx = (size_t)batch * H * W;
  const size_t imgBytes = align_up(npx * pixel_bytes, 256);
  const size_t labBytes = align_up(npx * 4, 256);
  const size_t nBytes = align_up((size_t)batch * 4, 256);
  constexpr size_t statusBytes = 256;
  char* buf = nullptr;
  if (cudaMallocFromPoolAsync((void**)&buf, imgBytes + labBytes + nBytes + statusBytes + L.total, pool, st) !=
      cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_NO_MEMORY;
  }
  void* dImg = buf;
  int32_t* dLab = (int32_t*)(buf + imgBytes);
  int32_t* dN = (int32_t*)(buf + imgBytes + labBytes);
  // this call's own status word: limits tripped by calls on other streams
  // stay in the device's sticky word for ccl_last_status
  int* status = (int*)(buf + imgBytes + labBytes + nBytes);
  void* ws = buf + imgBytes + labBytes + nBytes + statusBytes;
  cudaStream_t cs = nullptr;
  rc = cudaMemsetAsync(status, 0, sizeof(int), st) == cudaSuccess ? CCL_OK : CCL_ERR_CUDA;
  if (rc == CCL_OK) rc = device_copy_stream(&cs);
  if (rc == CCL_OK)
    rc = run_host_banded(img_host, batch, H, W, pixel_bytes, connectivity, mode, labels_host,
                         n_regions_host, dImg, dLab, dN, L, ws, status, st, cs);
  int h = 0;
  if (rc == CCL_OK && cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    rc = CCL_ERR_CUDA;
  cudaFreeAsync(buf, st);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_CUDA;
  }
  return rc != CCL_OK ? rc : status_of_flags(h);
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
  return status_of_flags(h);
}

int ccl_debug_counters(unsigned long long* out, int n, int reset) {
#ifdef CCL_COUNTERS
  if (!out || n < 0) return CCL_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return CCL_ERR_CUDA;
  unsigned long long h[CCL_NCOUNTERS];
  if (cudaMemcpyFromSymbol(h, g_counters, sizeof(h)) != cudaSuccess) return CCL_ERR_CUDA;
  for (int i = 0; i < n && i < CCL_NCOUNTERS; ++i) out[i] = h[i];
  if (reset) {
    const unsigned long long z[CCL_NCOUNTERS] = {0};
    if (cudaMemcpyToSymbol(g_counters, z, sizeof(z)) != cudaSuccess) return CCL_ERR_CUDA;
  }
  return CCL_OK;
#else
  (void)out;
  (void)n;
  (void)reset;
  return CCL_ERR_INVALID_ARG;   // not the counters build
#endif
}

size_t ccl_region_stats_workspace_bytes(int batch) {
  if (batch < 0) return 0;
  return align_up((size_t)(batch + 1) * sizeof(long long), 256);
}

int ccl_region_stats(const int32_t* labels_i32, int batch, int H, int W, const int32_t* n_regions,
                     ccl_region_stat* stats, int64_t capacity, void* workspace,
                     size_t workspace_bytes, ccl_stream_t stream) {
  if (batch < 0 || H < 0 || W < 0 || capacity < 0) return CCL_ERR_INVALID_ARG;
  if ((long long)H * W >= (1ll << 31)) return CCL_ERR_TOO_LARGE;
  if (batch == 0 || H == 0 || W == 0) return CCL_OK;
  if (!labels_i32 || !n_regions || ((uintptr_t)labels_i32 & 3) || ((uintptr_t)n_regions & 3))
    return CCL_ERR_INVALID_ARG;
  if (capacity > 0 && (!stats || ((uintptr_t)stats & 7))) return CCL_ERR_INVALID_ARG;
  const size_t need = ccl_region_stats_workspace_bytes(batch);
  if (workspace) {
    if ((uintptr_t)workspace & 255) return CCL_ERR_INVALID_ARG;
    if (workspace_bytes < need) return CCL_ERR_NO_MEMORY;
  }
  Layout L;
  int rc = make_layout(batch, H, W, false, &L);
  if (rc != CCL_OK) return rc;
  Geom g = L.g;
  g.vec_out = (W % 8 == 0) && ((uintptr_t)labels_i32 % 16 == 0);
  int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc != CCL_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  void* ws = workspace;
  cudaMemPool_t pool = nullptr;
  if (!ws) {
    rc = device_pool(&pool);
    if (rc != CCL_OK) return rc;
    if (cudaMallocFromPoolAsync(&ws, need, pool, st) != cudaSuccess) {
      cudaGetLastError();
      return CCL_ERR_NO_MEMORY;
    }
  }
  long long* off = (long long*)ws;
  k_stats_offsets<<<1, NT, 0, st>>>(n_regions, batch, off, status);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  k_stats_init<<<(unsigned)(sms * 8), NT, 0, st>>>(stats, (long long)capacity, off, batch, status);
  const int stripsX = (int)(((long long)W + STRIP_W - 1) / STRIP_W);
  const long long strips = (long long)batch * (((long long)H + SR - 1) / SR) * stripsX;
  k_region_stats<<<(unsigned)strips, STATS_NT, 0, st>>>(labels_i32, n_regions, off, stats,
                                                  (long long)capacity, g, stripsX, status);
  g_launches += 3;
  rc = cudaPeekAtLastError() == cudaSuccess ? CCL_OK : CCL_ERR_CUDA;
  if (!workspace && cudaFreeAsync(ws, st) != cudaSuccess && rc == CCL_OK) rc = CCL_ERR_CUDA;
  return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Labelling without any device allocation.
//
// Some callers may not allocate device memory at all: a host application or
// framework that owns the whole GPU memory budget (a fixed arena handed out
// by its own allocator), or a latency-critical loop that cannot afford the
// device-wide synchronisation cudaMalloc / cudaFree may imply.  For them
// ccl_label_noalloc runs the same kernels as ccl_label with its scratch in a
// fixed array that is part of this library's device image: every GPU that
// loads the library holds CCL_NOALLOC_SCRATCH_BYTES for it until the process
// exits.  Its first 256 bytes hold the call's device status word, the rest
// the workspace that ccl_workspace_bytes() sizes.

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CCL_NOALLOC_SCRATCH_BYTES];

constexpr size_t NOALLOC_STATUS_BYTES = 256;

// Device address of g_noalloc_scratch on the current device.  The array's
// name in host code is only a host-side stand-in, so the address is asked
// from the runtime once per device (with that device current) and cached.
void* g_noalloc_addr[MAX_DEVICES] = {nullptr};

int noalloc_scratch(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return CCL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CCL_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = (char*)g_noalloc_addr[dev];
  return CCL_OK;
}

// A device-side limit tripped during this call: every count becomes -1.
__global__ void k_noalloc_report(const int* status, int32_t* n_out, int batch) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch && *status != 0) n_out[b] = -1;
}

}  // namespace

extern "C" int ccl_label_noalloc(const void* img, int batch, int H, int W, int pixel_bytes,
                                 int connectivity, int mode, int32_t* labels_i32,
                                 int32_t* n_regions_out, ccl_stream_t stream) {
  bool empty = false;
  int rc = validate(img, batch, H, W, pixel_bytes, connectivity, mode, labels_i32, n_regions_out,
                    &empty);
  if (rc != CCL_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (empty) return empty_call(batch, n_regions_out, st);
  Layout L;
  rc = make_layout(batch, H, W, mode == CCL_MODE_BINARY, &L);
  if (rc != CCL_OK) return rc;
  if (L.total > (size_t)CCL_NOALLOC_SCRATCH_BYTES - NOALLOC_STATUS_BYTES) return CCL_ERR_TOO_LARGE;
  char* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != CCL_OK) return rc;
  int* status = (int*)scratch;
  // the array keeps the previous call's contents: the status word must start
  // at zero; every workspace word the kernels read is written earlier in the
  // same call
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) {
    cudaGetLastError();
    return CCL_ERR_CUDA;
  }
  rc = run_pipeline(img, batch, H, W, pixel_bytes, connectivity, mode, 0u, labels_i32,
                    n_regions_out, L, scratch + NOALLOC_STATUS_BYTES, status, false, st);
  if (rc == CCL_OK && n_regions_out) {
    k_noalloc_report<<<(batch + 255) / 256, 256, 0, st>>>(status, n_regions_out, batch);
    g_launches += 1;
    if (cudaPeekAtLastError() != cudaSuccess) rc = CCL_ERR_CUDA;
  }
  return rc;
}
