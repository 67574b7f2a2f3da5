/* A plain C99 consumer of the C ABI: includes the header, links libdmoe.so and
 * calls the entry points that need no GPU (queries and host-side argument
 * validation).  Built and run by the CPU tests; prints "ok" on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dmoe.h"

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s\n", what);
  return 1;
}

int main(void) {
  if (dmoe_version() <= 0) return fail("version");
  if (strlen(dmoe_status_string(DMOE_OK)) == 0) return fail("status string");
  if (dmoe_workspace_bytes(8192, 22, 512) < DMOE_WS_STATUS_BYTES) return fail("workspace bytes");
  if (dmoe_fingerprint_num_chunks((size_t)3 << 20, (size_t)1 << 20) != 3) return fail("chunks");
  dmoe_launch launch = {0, 0};
  /* null operands: rejected on the host before any device work */
  if (moe_grouped_gemm_fwd(NULL, NULL, NULL, 512, 4, 128, 256, NULL, &launch, NULL, 0, NULL) !=
      DMOE_ERR_INVALID_ARG)
    return fail("null operands");
  printf("ok\n");
  return 0;
}
