/* A plain C client of libfused_ce_tvd.so: the header and the library used
 * without Python.  Calls only entry points that need no GPU (version, status
 * strings, size queries, argument errors reported before any launch). */
#include <stdio.h>
#include <string.h>

#include "fused_ce_tvd.h"

int main(void) {
  if (fct_version() < 100) return 1;
  if (strcmp(fct_status_string(FCT_OK), fct_status_string(FCT_ERR_INVALID_ARG)) == 0) return 2;
  if (fused_ce_tvd_signs_row_bytes(151936, FCT_BF16) != 4 + 18992) return 3;
  /* logit blocks, then 2 x rows x 594 log-sum-exp states of 8 bytes */
  if (fused_linear_ce_tvd_workspace_size(151936, 2, FCT_F32) !=
      (size_t)2 * 151936 * 12 + (size_t)2 * 2 * 594 * 8)
    return 4;
  if (fused_linear_ce_tvd_workspace_size(151936, 2, FCT_BF16) !=
      (size_t)2 * 151936 * 6 + (size_t)2 * 2 * 594 * 8)
    return 4;
  if (fused_linear_ce_tvd_workspace_size(151936, 2, (fct_dtype)7) != 0) return 4;
  /* empty batch: a no-op */
  if (fused_ce_tvd_forward(NULL, 0, NULL, 0, FCT_BF16, NULL, 0, 8, -100, NULL, NULL, NULL,
                           NULL, NULL, NULL, NULL) != FCT_OK)
    return 5;
  /* negative batch and missing pointers: argument errors before any launch */
  if (ce_forward(NULL, 8, FCT_BF16, NULL, -1, 8, -100, NULL, NULL, NULL, NULL) !=
      FCT_ERR_INVALID_ARG)
    return 6;
  if (ce_forward_backward(NULL, 8, FCT_F32, NULL, 4, 8, -100, NULL, 1, NULL, NULL, NULL, 8,
                          NULL, NULL) != FCT_ERR_INVALID_ARG)
    return 7;
  printf("ok %d\n", fct_version());
  return 0;
}
