/* A C99 consumer of the library's public headers: it must compile as plain
 * C (no C++), link against the shared library, and get synchronous answers
 * from the calls that need no GPU.  Prints the sizes of the tuning structs
 * so that the Python binding's layouts can be compared with C's. */
#include <stdio.h>

#include "fa.h"
#include "fa_diag.h"

int main(void) {
  int failures = 0;
  /* argument errors come back before anything touches the device */
  if (fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 2, 128, 128, 128, 0, 0.125f, NULL, NULL) != FA_ERR_INVALID_ARG) {
    fprintf(stderr, "fa_fwd(NULL ...) did not return FA_ERR_INVALID_ARG\n");
    ++failures;
  }
  if (fa_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 2, 2, 128, 128, 128, 0, 0.125f, NULL, 0,
             NULL, 0, NULL) != FA_ERR_INVALID_ARG) {
    fprintf(stderr, "fa_bwd(NULL ...) did not return FA_ERR_INVALID_ARG\n");
    ++failures;
  }
  /* the workspace size is pure host arithmetic: accumulator + two row-term
   * arrays + the scheduler's counter slot */
  {
    const size_t n = fa_bwd_workspace_size(1, 2, 2, 128, 128, 128, NULL, 0, 0);
    const size_t want = (size_t)128 * 2 * 128 * 4 + 2 * ((size_t)2 * 128 * 4) + 256;
    if (n != want) {
      fprintf(stderr, "fa_bwd_workspace_size: %zu, expected %zu\n", n, want);
      ++failures;
    }
    if (fa_bwd_workspace_size(1, 2, 2, 128, 128, 80, NULL, 0, 0) != 0) {
      fprintf(stderr, "fa_bwd_workspace_size accepted D = 80\n");
      ++failures;
    }
  }
  {
    const fa_bwd_tuning t = fa_bwd_default_tuning();
    if (t.paired != 0 || t.schedule != -1) {
      fprintf(stderr, "unexpected backward defaults\n");
      ++failures;
    }
  }
  printf("status %s\n", fa_status_string(FA_ERR_WORKSPACE));
  printf("sizeof fa_fwd_tuning %zu\n", sizeof(fa_fwd_tuning));
  printf("sizeof fa_bwd_tuning %zu\n", sizeof(fa_bwd_tuning));
  return failures ? 1 : 0;
}
