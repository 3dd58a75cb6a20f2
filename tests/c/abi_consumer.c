/* A plain C99 consumer of include/ccl.h: it links against libccl.so and calls
 * only entry points that answer on the host (no device is touched), so it
 * runs without a GPU.  Exit status 0 when every check holds; otherwise the
 * number of the first failed check. */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ccl.h"

/* the statistics entry is 40 bytes: six int32 fields then two int64 sums */
typedef char stat_is_40_bytes[sizeof(ccl_region_stat) == 40 ? 1 : -1];
typedef char sum_y_at_24[offsetof(ccl_region_stat, sum_y) == 24 ? 1 : -1];

int main(void) {
  const void* fake = (const void*)(uintptr_t)(1u << 20);   /* never dereferenced */
  int32_t* labels = (int32_t*)(uintptr_t)(1u << 26);
  if (ccl_version() <= 0) return 1;
  if (strcmp(ccl_status_string(CCL_OK), "CCL_OK") != 0) return 2;
  if (strcmp(ccl_status_string(CCL_ERR_TOO_LARGE), "CCL_ERR_TOO_LARGE") != 0) return 3;
  if (ccl_workspace_bytes(1, 1024, 1024, 4, 8, CCL_MODE_ALL) == 0) return 4;
  if (ccl_workspace_bytes(1, 1024, 1024, 5, 8, CCL_MODE_ALL) != 0) return 5;
  /* argument errors are found on the host, before any device call */
  if (ccl_label(fake, 1, 64, 64, 4, 6, CCL_MODE_ALL, labels, NULL, NULL) != CCL_ERR_INVALID_ARG) return 6;
  if (ccl_label(fake, 1, 65536, 65536, 1, 8, CCL_MODE_ALL, labels, NULL, NULL) != CCL_ERR_TOO_LARGE) return 7;
  if (ccl_label(fake, 1, 64, 64, 4, 8, CCL_MODE_ALL, (int32_t*)fake, NULL, NULL) != CCL_ERR_INVALID_ARG) return 8;
  /* an empty call succeeds without work */
  if (ccl_label(NULL, 0, 64, 64, 1, 8, CCL_MODE_BINARY, NULL, NULL, NULL) != CCL_OK) return 9;
  if (ccl_set_option(CCL_OPT_WALK_CAP, 0) != CCL_OK) return 10;
  if (ccl_set_option(99, 0) != CCL_ERR_INVALID_ARG) return 11;
  if (strcmp(ccl_stage_name(0), "tile_local") != 0) return 12;
  printf("C consumer ok\n");
  return 0;
}
