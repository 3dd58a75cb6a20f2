/*
 * ccl_oracle.c -- the oracle: plain, slow, single-threaded CPU labelling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file; it shares no code with the CUDA library.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes is the plain definition of the result, not the GPU method:
 *
 *   "every-colour" (blogs.fablnx.com), ch. 01 "The job" and ch. 02 "Regions":
 *     two pixels share a number exactly when one can walk from one to the
 *     other, one neighbour at a time, without changing colour; anti-aliased
 *     shades are colours of their own; a pixel has eight neighbours (or four,
 *     "About Connected Components Labeling on GPU", bendabir.com, Prologue).
 *   "every-colour", ch. 04 "Point at a leader" and ch. 11 "How we know it is
 *     right": a region's leader is its first pixel in reading order, and the
 *     regions are numbered 1, 2, 3 ... in the reading order of their leaders.
 *   "every-colour", ch. 08 switch 4 "Ignore the paper": pixels of the ignored
 *     value get label 0 and join nothing.  Binary mode ignores value 0
 *     (bendabir.com, "The basic approach": background keeps 0).
 *
 * Algorithm: for every image, scan the pixels in raster order; every pixel
 * that is neither labelled nor ignored starts a new region with the next
 * number and a breadth-first flood fill (explicit FIFO queue, no recursion)
 * spreads that number over every pixel reachable through equal-valued
 * neighbours.  Because the seeds are taken in raster order, the first pixel
 * of every region is its seed, and the numbering is the canonical one.
 *
 * Equality compares all pixel_bytes bytes of a pixel (RGBA: alpha included).
 */
#include <stdint.h>
#include <stdlib.h>
#include <limits.h>
#include <string.h>

/* Return codes mirror the library's status numbers where they overlap. */
#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_TOO_LARGE 2   /* H*W >= 2^32, or more regions than int32 labels hold */
#define ORACLE_ERR_NO_MEMORY 4

enum { ORACLE_MODE_ALL = 0, ORACLE_MODE_BINARY = 1 };

static int same_value(const uint8_t* a, const uint8_t* b, int pb) {
  return memcmp(a, b, (size_t)pb) == 0;
}

static int is_zero(const uint8_t* a, int pb) {
  for (int k = 0; k < pb; ++k)
    if (a[k] != 0) return 0;
  return 1;
}

/*
 * Label one image.  img: H*W pixels of pb bytes, row-major.  labels: H*W
 * int32, written completely.  queue: scratch of H*W int64.  Returns the
 * number of regions, or -1 if they outnumber what int32 labels hold.
 */
static int64_t label_one(const uint8_t* img, int64_t H, int64_t W, int pb,
                         int conn, int mode, const uint8_t* ign,
                         int32_t* labels, int64_t* queue) {
  const int64_t N = H * W;
  /* neighbour offsets: 4-connectivity uses the first four (edge-sharing),
   * 8-connectivity adds the four corner-sharing ones */
  static const int dr[8] = {-1, 0, 0, 1, -1, -1, 1, 1};
  static const int dc[8] = {0, -1, 1, 0, -1, 1, -1, 1};
  const int nn = (conn == 8) ? 8 : 4;

  for (int64_t i = 0; i < N; ++i) labels[i] = 0;
  /* pixels still to visit are marked -1; ignored pixels keep 0 */
  for (int64_t i = 0; i < N; ++i) {
    const uint8_t* v = img + i * pb;
    if (mode == ORACLE_MODE_BINARY && is_zero(v, pb))
      labels[i] = 0;
    else if (ign && same_value(v, ign, pb))
      labels[i] = 0;   /* the ignored value: background */
    else
      labels[i] = -1;
  }

  int64_t n = 0;
  for (int64_t seed = 0; seed < N; ++seed) {
    if (labels[seed] != -1) continue;
    if (n == INT32_MAX) return -1;   /* one more region than int32 labels hold */
    ++n;
    labels[seed] = (int32_t)n;
    int64_t head = 0, tail = 0;
    queue[tail++] = seed;
    while (head < tail) {
      const int64_t p = queue[head++];
      const int64_t r = p / W, c = p % W;
      const uint8_t* pv = img + p * pb;
      for (int k = 0; k < nn; ++k) {
        const int64_t rr = r + dr[k], cc = c + dc[k];
        if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue; /* no wrap */
        const int64_t q = rr * W + cc;
        if (labels[q] != -1) continue;
        if (!same_value(pv, img + q * pb, pb)) continue;
        labels[q] = (int32_t)n;
        queue[tail++] = q;
      }
    }
  }
  return n;
}

/*
 * oracle_label: label `batch` images of H x W pixels of `pixel_bytes` bytes,
 * stored contiguously; image b starts at byte b*H*W*pixel_bytes and its labels
 * at element b*H*W.  n_out[b] receives the number of regions of image b.
 * Host pointers only.  Images of up to 2^32 - 1 pixels (64-bit indices
 * throughout).  Returns ORACLE_OK, ORACLE_ERR_INVALID_ARG,
 * ORACLE_ERR_NO_MEMORY, or ORACLE_ERR_TOO_LARGE (H*W >= 2^32, or an image
 * with more regions than int32 labels hold: its count is -1).
 */
static int label_all(const void* img, int64_t batch, int64_t H, int64_t W,
                     int pixel_bytes, int connectivity, int mode,
                     const uint8_t* ign, int32_t* labels, int32_t* n_out);

int oracle_label(const void* img, int64_t batch, int64_t H, int64_t W,
                 int pixel_bytes, int connectivity, int mode,
                 int32_t* labels, int32_t* n_out) {
  return label_all(img, batch, H, W, pixel_bytes, connectivity, mode, NULL,
                   labels, n_out);
}

/*
 * oracle_label_ignore: as oracle_label in the all-pixels mode, except that
 * pixels whose pixel_bytes bytes equal ignore_value (host pointer to
 * pixel_bytes bytes) are background: label 0, joining nothing
 * ("every-colour", ch. 08 switch 4 "Ignore the paper": the named colour
 * gets label 0 and takes part in nothing after).
 */
int oracle_label_ignore(const void* img, int64_t batch, int64_t H, int64_t W,
                        int pixel_bytes, int connectivity,
                        const void* ignore_value, int32_t* labels,
                        int32_t* n_out) {
  if (!ignore_value) return ORACLE_ERR_INVALID_ARG;
  return label_all(img, batch, H, W, pixel_bytes, connectivity, ORACLE_MODE_ALL,
                   (const uint8_t*)ignore_value, labels, n_out);
}

static int label_all(const void* img, int64_t batch, int64_t H, int64_t W,
                     int pixel_bytes, int connectivity, int mode,
                     const uint8_t* ign, int32_t* labels, int32_t* n_out) {
  if (batch < 0 || H < 0 || W < 0) return ORACLE_ERR_INVALID_ARG;
  if (pixel_bytes < 1 || pixel_bytes > 16) return ORACLE_ERR_INVALID_ARG;
  if (connectivity != 4 && connectivity != 8) return ORACLE_ERR_INVALID_ARG;
  if (mode != ORACLE_MODE_ALL && mode != ORACLE_MODE_BINARY)
    return ORACLE_ERR_INVALID_ARG;
  const int64_t N = H * W;
  if (batch == 0 || N == 0) {
    for (int64_t b = 0; b < batch; ++b) n_out[b] = 0;
    return ORACLE_OK;
  }
  if (!img || !labels || !n_out) return ORACLE_ERR_INVALID_ARG;
  /* the library's bound: raster indices inside an image fit 32 bits */
  if (N >= ((int64_t)1 << 32)) return ORACLE_ERR_TOO_LARGE;
  int64_t* queue = (int64_t*)malloc((size_t)N * sizeof(int64_t));
  if (!queue) return ORACLE_ERR_NO_MEMORY;
  const uint8_t* base = (const uint8_t*)img;
  int rc = ORACLE_OK;
  for (int64_t b = 0; b < batch; ++b) {
    const int64_t n = label_one(base + b * N * pixel_bytes, H, W, pixel_bytes,
                                connectivity, mode, ign, labels + b * N, queue);
    if (n < 0) rc = ORACLE_ERR_TOO_LARGE;
    n_out[b] = n < 0 ? -1 : (int32_t)n;
  }
  free(queue);
  return rc;
}

/*
 * Region statistics: the step that usually follows labelling.  The lpnh.cn
 * page (CUDA image segmentation, §1.1) labels the regions so that their
 * area and position can be measured next; "GPU Connected Component Labeling"
 * (mcclanahoochie.com, closing section) names statistics on every labelled
 * region as the next image-processing step; bendabir.com (Prologue) uses the
 * labels to cut out each area's bounding box.  The pages define no formula
 * beyond the names, so the plain definitions are taken:
 *
 *   area         number of pixels carrying the label;
 *   y_min .. x_max  the smallest and largest row and column among them
 *                (inclusive bounding box);
 *   first        raster index y*W + x, inside the image, of the first of them
 *                in reading order;
 *   sum_y, sum_x sums of their row and column indices (the centroid is
 *                sum / area).
 *
 * Layout (40 bytes): six int32 (area, y_min, x_min, y_max, x_max, first),
 * then two int64 (sum_y, sum_x).  The entry of label l (1..n_regions[b]) of
 * image b is at index n_regions[0] + ... + n_regions[b-1] + l - 1.  A label
 * that no pixel carries keeps area 0, box (INT32_MAX, INT32_MAX, -1, -1),
 * first INT32_MAX and zero sums.  Labels must lie in 0..n_regions[b]
 * (0 = background, counted nowhere); any other value gives
 * ORACLE_ERR_INVALID_ARG.  Host pointers only.
 */
typedef struct {
  int32_t area, y_min, x_min, y_max, x_max, first;
  int64_t sum_y, sum_x;
} oracle_region_stat;

int oracle_region_stats(const int32_t* labels, int64_t batch, int64_t H,
                        int64_t W, const int32_t* n_regions,
                        oracle_region_stat* out, int64_t capacity) {
  if (batch < 0 || H < 0 || W < 0 || capacity < 0) return ORACLE_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int64_t b = 0; b < batch; ++b) {
    if (n_regions[b] < 0) return ORACLE_ERR_INVALID_ARG;
    total += n_regions[b];
  }
  if (total > capacity) return ORACLE_ERR_NO_MEMORY;
  for (int64_t e = 0; e < total; ++e) {
    out[e].area = 0;
    out[e].y_min = INT32_MAX;
    out[e].x_min = INT32_MAX;
    out[e].y_max = -1;
    out[e].x_max = -1;
    out[e].first = INT32_MAX;
    out[e].sum_y = 0;
    out[e].sum_x = 0;
  }
  int64_t base = 0;
  for (int64_t b = 0; b < batch; ++b) {
    const int32_t* lab = labels + b * H * W;
    for (int64_t y = 0; y < H; ++y) {
      for (int64_t x = 0; x < W; ++x) {
        const int32_t l = lab[y * W + x];
        if (l == 0) continue;
        if (l < 0 || l > n_regions[b]) return ORACLE_ERR_INVALID_ARG;
        oracle_region_stat* s = &out[base + l - 1];
        if (s->area == 0) s->first = (int32_t)(y * W + x);   /* reading order */
        s->area += 1;
        if (y < s->y_min) s->y_min = (int32_t)y;
        if (x < s->x_min) s->x_min = (int32_t)x;
        if (y > s->y_max) s->y_max = (int32_t)y;
        if (x > s->x_max) s->x_max = (int32_t)x;
        s->sum_y += y;
        s->sum_x += x;
      }
    }
    base += n_regions[b];
  }
  return ORACLE_OK;
}
