/* A plain C99 program against include/flce.h and libflce.so: the header is C,
 * and the host-side entry points (sizes, validation, status strings) work
 * without a GPU.  Prints "ok" and exits 0 on success. */
#include <stdio.h>
#include <string.h>

#include "flce.h"

int main(void) {
  flce_problem_t p;
  memset(&p, 0, sizeof p);
  p.n = 8192;
  p.h = 2048;
  p.v = 32000;
  p.ignore_index = -100;
  p.reduction = FLCE_REDUCTION_MEAN;
  size_t full = flce_workspace_bytes(&p);
  size_t rowchunk = flce_workspace_bytes_rowchunk(&p);
  p.v = 4 * 32000;
  size_t full_wide = flce_workspace_bytes(&p);
  p.v = 32000;
  if (full == 0 || rowchunk == 0 || full != full_wide) {
    printf("bad workspace sizes %zu %zu %zu\n", full, rowchunk, full_wide);
    return 1;
  }
  p.h = 12; /* not a multiple of 8 */
  if (flce_workspace_bytes(&p) != 0) {
    printf("h = 12 accepted\n");
    return 1;
  }
  p.h = 2048;
  /* a null X is rejected before any device call */
  if (flce_forward(&p, NULL, (const void*)0x2000, (const int32_t*)0x3000, (float*)0x4000, (float*)0x5000,
                   (void*)0x100000, full, NULL) != FLCE_ERR_INVALID_ARGUMENT) {
    printf("null X accepted\n");
    return 1;
  }
  if (strlen(flce_status_string(FLCE_ERR_TIMEOUT)) == 0) {
    printf("empty status string\n");
    return 1;
  }
  printf("ok %zu %zu\n", full, rowchunk);
  return 0;
}
