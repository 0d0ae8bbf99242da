/* Plain C99 use of the C ABI (include/ipttt.h), host-only calls: no GPU is needed.
 * Prints one line per check; the exit status is the number of failed checks. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ipttt.h"

static int failures = 0;

static void check(int ok, const char* what) {
  printf("%s %s\n", ok ? "ok" : "FAIL", what);
  if (!ok) ++failures;
}

int main(void) {
  size_t bytes = 0, train = 0;
  check(ipttt_version() != NULL && strlen(ipttt_version()) > 0, "version string");
  check(strcmp(ipttt_status_string(IPTTT_OK), "IPTTT_OK") == 0, "status string of OK");
  /* the 4B-shaped 32k-token layer */
  check(ipttt_workspace_size(1, 32768, 2560, 9728, 1024, 4, IPTTT_BF16, &bytes) == IPTTT_OK && bytes > 0,
        "workspace size of the 4B-shaped layer");
  printf("workspace %zu\n", bytes);
  check(ipttt_saved_size(1, 32768, 2560, 9728, 1024, 4, IPTTT_BF16, &train) == IPTTT_OK && train > 0,
        "saved-activation size of the 4B-shaped layer");
  printf("saved %zu\n", train);
  check(ipttt_workspace_size(1, 32768, 2560, 9728, 1000, 4, IPTTT_BF16, &bytes) == IPTTT_ERR_UNSUPPORTED,
        "bf16 chunk size not a multiple of 128 is unsupported");
  check(ipttt_workspace_size(1, 64, 64, 128, 16, 4, IPTTT_F32, NULL) == IPTTT_ERR_INVALID_ARG,
        "NULL size pointer is an invalid argument");
  check(ipttt_create(NULL, 0, NULL) == IPTTT_ERR_INVALID_ARG, "create without an output pointer");
  check(ipttt_layer_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 8, 8, 1, 1, 1.0f, IPTTT_F32, NULL,
                            NULL, NULL, 0) == IPTTT_ERR_INVALID_ARG,
        "layer call without a context");
  check(ipttt_decode_step(NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 8, 8, IPTTT_F32, NULL, NULL, NULL, NULL, 0, 0) ==
            IPTTT_ERR_INVALID_ARG,
        "decode step without a context");
  ipttt_destroy(NULL);
  check(1, "destroy(NULL) is a no-op");
  return failures;
}
