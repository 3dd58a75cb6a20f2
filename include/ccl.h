/*
 * ccl.h -- C ABI of the GB300 connected-component labelling library
 * (libccl.so).
 *
 * The operation ("every-colour", blogs.fablnx.com, ch. 01 "The job" and
 * ch. 02 "Regions"): two pixels belong to the same region exactly when a path
 * of neighbouring pixels of exactly equal value joins them; 8-connectivity
 * counts corner-sharing neighbours, 4-connectivity only edge-sharing ones
 * ("About Connected Components Labeling on GPU", bendabir.com, Prologue).
 * Regions are numbered 1..n in the raster order of their first pixel
 * ("every-colour", ch. 04 "Point at a leader" -- the leader is the first
 * pixel in reading order -- and ch. 11 "How we know it is right").  In
 * binary mode value 0 is background: it keeps label 0 and joins nothing
 * ("every-colour", ch. 08 switch 4 "Ignore the paper"; bendabir.com, "The
 * basic approach", labels + 1 keep 0 for background).
 *
 * The library runs the four stages of "every-colour" ch. 05 (Start,
 * Connect, Collapse, Number) as CUDA kernels for sm_103a.  There is no CPU
 * fallback: every entry point that computes needs a CUDA device.
 *
 * Conventions for every entry point:
 *  - Images are contiguous and row-major: pixel (b, y, x) sits at byte
 *    ((b*H + y)*W + x) * pixel_bytes of `img`; labels likewise at element
 *    (b*H + y)*W + x of `labels_i32`.  `img` must be aligned to pixel_bytes
 *    (3-byte pixels: no alignment), `labels_i32` and `n_regions_out` to 4
 *    bytes.
 *  - pixel_bytes 3 is packed 24-bit RGB, three bytes a pixel: the form
 *    "every-colour" reads its drawings in (ch. 08 "Tried and dropped": a
 *    packed 32-bit copy of the picture was slower and twice the memory).
 *  - Pixel equality compares all pixel_bytes bytes (RGBA: alpha included).
 *  - Labels are canonical per image: numbering restarts at 1 in every image.
 *  - H*W must be below 2^32 (CCL_ERR_TOO_LARGE otherwise; "every-colour"
 *    ch. 11 names images of more than 2^31 pixels as the case it never ran):
 *    raster indices inside an image are 32-bit.  Also refused: an image whose
 *    256 x 16 tiles would hold 2^32 or more border slots (only images of one
 *    or two rows close to that size), and a grid of 2^31 or more tiles.
 *    batch*H*W may exceed 2^32.  Labels stay int32: an image with more than
 *    2^31 - 1 regions completes with its counts clamped and the device status
 *    CCL_ERR_TOO_LARGE (ccl_last_status).
 *  - batch == 0, H == 0 or W == 0 is a valid empty call (n_regions_out, if
 *    given, is set to 0 for every image).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  The return value reports argument and launch errors
 *    only; a device-side limit that trips is reported by ccl_last_status().
 *  - `labels_i32` also holds, between two stages of the call, the labels of
 *    regions joined across tile seams (parked inside their tile until the
 *    last stage reads them back), so it must not overlap `img`; the counts
 *    are written before the labels, so `n_regions_out` must not overlap
 *    `labels_i32` either.
 *  - All pointers are owned by the caller; the library frees nothing of theirs.
 */
#ifndef CCL_H_
#define CCL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same layout as cudaStream_t, without pulling in the CUDA headers. */
typedef struct CUstream_st* ccl_stream_t;

typedef enum {
  CCL_OK = 0,
  CCL_ERR_INVALID_ARG = 1,   /* bad pointer, size, enum value or alignment */
  CCL_ERR_TOO_LARGE = 2,     /* H*W >= 2^32 (see the conventions); on the device:
                                more regions than int32 labels hold */
  CCL_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  CCL_ERR_NO_MEMORY = 4,     /* workspace allocation failed / too small */
  CCL_ERR_DEVICE_LIMIT = 5   /* a bounded device loop reached its cap */
} ccl_status;

enum { CCL_MODE_ALL = 0, CCL_MODE_BINARY = 1 };

/*
 * ccl_label -- label `batch` images of H x W pixels.
 *   img            device pointer, batch*H*W pixels of pixel_bytes (1, 2, 3 or 4)
 *   connectivity   4 or 8
 *   mode           CCL_MODE_ALL (every pixel labelled) or CCL_MODE_BINARY
 *                  (all-zero pixels are background, label 0)
 *   labels_i32     device pointer, batch*H*W int32, written completely
 *   n_regions_out  device pointer to batch int32 (region count per image),
 *                  or NULL
 * Scratch (ccl_workspace_bytes(...) bytes, about 3.9 bytes per pixel) comes
 * from a stream-ordered memory pool the library keeps per device.
 * Returns CCL_OK or an error status; nothing is written on an argument error.
 */
int ccl_label(const void* img, int batch, int H, int W, int pixel_bytes,
              int connectivity, int mode, int32_t* labels_i32,
              int32_t* n_regions_out, ccl_stream_t stream);

/* Bytes of device workspace ccl_label_ws needs for these arguments
 * (0 for an empty call or invalid arguments).  Per image row a run-start bit
 * per pixel (and, in binary mode, a foreground bit); per tile of 256 columns
 * x 16 rows a leader for every run it can hold, its leader bits, run bases,
 * seam joins, and for every border pixel a slot record and an 8-byte parent
 * entry; chunk counts for the numbering.  About 3.9 bytes per pixel for
 * images of many whole tiles (4.0 in binary mode); thin images cost more per
 * pixel, since every pixel of a one-row tile is a border pixel (one row of
 * 2^31 - 1 pixels: about 15 bytes per pixel). */
size_t ccl_workspace_bytes(int batch, int H, int W, int pixel_bytes,
                           int connectivity, int mode);

/*
 * ccl_label_ws -- ccl_label with caller-provided scratch: `workspace` is a
 * device pointer to at least ccl_workspace_bytes(...) bytes, 256-byte
 * aligned, owned by the caller and not used by any other call in flight.
 * Returns CCL_ERR_NO_MEMORY if workspace_bytes is too small and
 * CCL_ERR_INVALID_ARG if the workspace it uses shares bytes with the image,
 * the labels or the counts.
 */
int ccl_label_ws(const void* img, int batch, int H, int W, int pixel_bytes,
                 int connectivity, int mode, int32_t* labels_i32,
                 int32_t* n_regions_out, void* workspace,
                 size_t workspace_bytes, ccl_stream_t stream);

/*
 * ccl_label_ignore -- label every pixel except those whose pixel_bytes
 * bytes equal `ignore_value` (little-endian; it must fit in pixel_bytes):
 * those keep label 0 and join nothing ("every-colour", ch. 08 switch 4
 * "Ignore the paper": if the caller names a colour to ignore, its pixels get
 * label 0 in Start and take part in nothing after).  ignore_value 0 is the
 * same as CCL_MODE_BINARY.  The other pixels are labelled as in
 * CCL_MODE_ALL: 1..n by first pixel in raster order.
 * `workspace` as in ccl_label_ws, sized by ccl_workspace_bytes(..., 
 * CCL_MODE_BINARY) (the ignoring pipeline keeps foreground bits), 256-byte
 * aligned; or NULL to take scratch from the library's per-device pool.
 * Returns CCL_ERR_INVALID_ARG if ignore_value does not fit in pixel_bytes.
 */
int ccl_label_ignore(const void* img, int batch, int H, int W,
                     int pixel_bytes, int connectivity, uint32_t ignore_value,
                     int32_t* labels_i32, int32_t* n_regions_out,
                     void* workspace, size_t workspace_bytes,
                     ccl_stream_t stream);

/*
 * ccl_label_host -- the whole call from host memory: copies `img_host` to
 * the device, labels it and copies the labels (and counts) back into
 * `labels_host` / `n_regions_host` (host pointers; page-locked memory is
 * fastest).  The copies run in bands of 16-row tile rows on a copy stream of
 * the library's, overlapped with the kernels (a band is labelled inside its
 * tiles while the next is copied in; a band's labels are copied out once
 * numbered).  Device buffers come from the library's pool.  Returns after the
 * results are in host memory (the stream is synchronised); a device-side
 * finding of this call (a tripped limit: CCL_ERR_DEVICE_LIMIT; more regions
 * than int32 labels: CCL_ERR_TOO_LARGE) is returned directly.  The call keeps
 * a status word of its own: findings of other calls stay in the device's word
 * for ccl_last_status, and this call's do not go there.
 */
int ccl_label_host(const void* img_host, int batch, int H, int W,
                   int pixel_bytes, int connectivity, int mode,
                   int32_t* labels_host, int32_t* n_regions_host,
                   ccl_stream_t stream);

/*
 * ccl_last_status -- synchronises `stream`, then returns and clears the
 * current device's sticky device-side status: CCL_ERR_DEVICE_LIMIT if a
 * bounded loop (a union-find walk or a union retry) reached its cap in any
 * call since the last check, CCL_ERR_TOO_LARGE if an image had more regions
 * than int32 labels hold, CCL_ERR_NO_MEMORY / CCL_ERR_INVALID_ARG for the
 * device-side findings of ccl_region_stats (see there), CCL_ERR_CUDA if the
 * stream reports an error, else CCL_OK.  Every labelling call except
 * ccl_label_host and ccl_label_noalloc reports into this word.  The caps are far above any
 * legitimate walk; tripping one means the labels of that call are not valid.
 */
int ccl_last_status(ccl_stream_t stream);

/* Human-readable name of a status value (static string). */
const char* ccl_status_string(int status);

/*
 * Debug / test options (process-wide):
 *   CCL_OPT_WALK_CAP  cap on every union-find walk and union retry loop
 *                     (value <= 0 restores the default, the number of pixels
 *                     the walk can visit); lowering it lets a test make the
 *                     device report CCL_ERR_DEVICE_LIMIT without any hang.
 *   CCL_OPT_STAGE_EVENTS  non-zero: record per-stage CUDA events in every
 *                     call (see ccl_stage_times); 0: stop recording.
 * Returns CCL_OK or CCL_ERR_INVALID_ARG for an unknown option.
 */
enum { CCL_OPT_WALK_CAP = 1, CCL_OPT_STAGE_EVENTS = 2 };
int ccl_set_option(int option, long long value);

/*
 * Per-stage device timing.  While option CCL_OPT_STAGE_EVENTS is non-zero
 * every labelling call records a CUDA event on its own stream before its
 * first kernel and after each stage (the stages are named by
 * ccl_stage_name: 0 tile_local, 1 seams, 2 scan, 3 resolve, 4 number).
 * ccl_stage_times waits for those events, writes the summed milliseconds of
 * each stage over all recorded calls into ms_sum[0..max_stages) and the call
 * count into *n_calls (either pointer may be NULL), forgets the recorded
 * calls and returns the number of stages (or a negative ccl_status).
 */
int ccl_stage_times(double* ms_sum, int max_stages, int* n_calls);
const char* ccl_stage_name(int stage);

/* Number of CUDA kernels this library has launched in this process. */
long long ccl_kernel_launches(void);

/*
 * ccl_label_noalloc -- ccl_label for callers that may not allocate device
 * memory: a program whose device memory is owned and budgeted by someone
 * else (a framework arena, a fixed-size pool), or a latency-critical loop
 * that must not pay for the device-wide synchronisation cudaMalloc and
 * cudaFree can cause.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.  The pages this library follows have no counterpart of
 * this entry point; it exists only for such callers.
 *
 * Arguments, layout, results and ownership are those of ccl_label; the
 * caller still provides img, labels_i32 and n_regions_out.  The scratch is a
 * fixed array of CCL_NOALLOC_SCRATCH_BYTES inside the library's device image,
 * held by every GPU that loads the library until the process exits; 256
 * bytes of it are a status word and the rest must be at least
 * ccl_workspace_bytes(...) for these arguments, else the call returns
 * CCL_ERR_TOO_LARGE without doing anything (about 3.9 bytes per pixel:
 * roughly 8.5 million pixels per call).
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array: calls whose work overlaps
 *    on the GPU (other streams, or other threads) race and give wrong labels.
 *    Serialise them, e.g. by using one stream.
 *  - A device-side limit tripped during the call (see ccl_last_status) is
 *    reported by writing -1 to every n_regions_out entry (pass
 *    n_regions_out to be told); ccl_last_status does not see it.
 */
#define CCL_NOALLOC_SCRATCH_BYTES (32u << 20)
int ccl_label_noalloc(const void* img, int batch, int H, int W,
                      int pixel_bytes, int connectivity, int mode,
                      int32_t* labels_i32, int32_t* n_regions_out,
                      ccl_stream_t stream);

/*
 * Region statistics, the step after labelling: regions are labelled so that
 * their area and position can be measured (CUDA image segmentation, lpnh.cn,
 * §1.1); statistics on every labelled region are the next image-processing
 * step ("GPU Connected Component Labeling", mcclanahoochie.com, closing
 * section); each area's bounding box (bendabir.com, Prologue).  Per region:
 *   area            number of pixels carrying the label;
 *   y_min .. x_max  inclusive bounding box (rows, columns);
 *   first           raster index y*W + x, inside its image, of the region's
 *                   first pixel in reading order (its leader);
 *   sum_y, sum_x    sums of the rows and of the columns of its pixels (the
 *                   centroid is sum / area).
 * A label that no pixel carries keeps area 0, box (INT32_MAX, INT32_MAX,
 * -1, -1), first INT32_MAX and zero sums.
 */
typedef struct ccl_region_stat {
  int32_t area, y_min, x_min, y_max, x_max, first;
  int64_t sum_y, sum_x;
} ccl_region_stat; /* 40 bytes */

/*
 * ccl_region_stats_workspace_bytes -- scratch bytes ccl_region_stats needs
 * for `batch` images ((batch + 1) int64 offsets, rounded up to 256); 0 for
 * batch < 0.
 */
size_t ccl_region_stats_workspace_bytes(int batch);

/*
 * ccl_region_stats -- statistics of every region of `labels_i32` (device,
 * [batch][H][W] int32, as written by ccl_label / ccl_label_ws /
 * ccl_label_ignore: 0 is background and counted nowhere, 1..n_regions[b] in
 * image b).  `n_regions` (device, int32[batch]) holds the region counts of
 * the same call.  `stats` (device, 8-byte aligned, room for `capacity`
 * entries): the entry of label l of image b is at index
 * n_regions[0] + ... + n_regions[b-1] + l - 1, and every entry below that
 * total is written.  `workspace`: ccl_region_stats_workspace_bytes(batch)
 * bytes, 256-byte aligned, or NULL to take it from the library's pool.  All
 * buffers are the caller's; the call only reads labels_i32 and n_regions.
 * Asynchronous on `stream`.  Host-side errors are returned (bad pointer,
 * alignment or size: CCL_ERR_INVALID_ARG; H*W >= 2^31, whose raster indices
 * the int32 `first` field cannot hold: CCL_ERR_TOO_LARGE;
 * workspace too small: CCL_ERR_NO_MEMORY).  Device-side findings go to
 * ccl_last_status: CCL_ERR_NO_MEMORY if the regions outnumber `capacity`
 * (entries at and beyond it are skipped), CCL_ERR_INVALID_ARG if a label lies
 * outside 0..n_regions of its image or a count is negative (skipped).
 */
int ccl_region_stats(const int32_t* labels_i32, int batch, int H, int W,
                     const int32_t* n_regions, ccl_region_stat* stats,
                     int64_t capacity, void* workspace, size_t workspace_bytes,
                     ccl_stream_t stream);

/*
 * Event counters of the labelling kernels, for measuring the method rather
 * than using it: in-tile walks, their steps and links (shared memory),
 * global walks, their steps and links (the parent array across tiles), seam
 * leader pairs kept, resolve walk steps (indices CCL_CNT_*).  They exist only
 * in the counters build of the library (compiled with -DCCL_COUNTERS, one
 * global atomic per event, slow); the normal build returns
 * CCL_ERR_INVALID_ARG.  ccl_debug_counters synchronises the device, copies
 * min(n, CCL_NCOUNTERS) counters to `out` (host) and, if `reset`, zeroes them.
 */
#define CCL_NCOUNTERS 8
enum {
  CCL_CNT_TILE_WALKS = 0, CCL_CNT_TILE_STEPS = 1, CCL_CNT_TILE_LINKS = 2,
  CCL_CNT_GLOBAL_WALKS = 3, CCL_CNT_GLOBAL_STEPS = 4, CCL_CNT_GLOBAL_LINKS = 5,
  CCL_CNT_SEAM_PAIRS = 6, CCL_CNT_RESOLVE_STEPS = 7
};
int ccl_debug_counters(unsigned long long* out, int n, int reset);

/* Library version, as major*10000 + minor*100 + patch. */
int ccl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCL_H_ */
