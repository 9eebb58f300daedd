/* A plain C program against include/vca.h and libvca.so: the header compiles
 * as C99, the entry points link, and the calls that need no GPU behave as the
 * header documents (status strings, version, workspace sizes, synchronous
 * rejection of bad arguments).  Prints one line per check and returns the
 * number of failures. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "vca.h"

static int failures = 0;

static void check(int ok, const char *what) {
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok) failures++;
}

int main(void) {
    uint8_t *fake8 = (uint8_t *)(uintptr_t)0x10000;   /* aligned, never dereferenced */
    float *fakef = (float *)(uintptr_t)0x10000;
    uint16_t *fake16 = (uint16_t *)(uintptr_t)0x10000;
    int32_t *fake32 = (int32_t *)(uintptr_t)0x10000;

    check(strcmp(vca_status_string(VCA_OK), "ok") == 0, "status string of VCA_OK");
    check(strcmp(vca_status_string(VCA_ERR_WORKSPACE), "workspace missing or too small") == 0,
          "status string of VCA_ERR_WORKSPACE");
    check(vca_version() >= 100, "version");
    check(vca_workspace_bytes(VCA_OP_GROUP, 1, 40, 70656, 128, 64, VCA_V_E4M3) > 0, "group workspace at 1x40x70656");
    check(vca_workspace_bytes(VCA_OP_PREP, 1, 40, 70656, 128, 1, VCA_V_NVFP4) > 0, "prep workspace at 1x40x70656");
    check(vca_workspace_bytes(VCA_OP_PREP, 1, 40, 1000, 128, 1, VCA_V_E4M3) == 0, "no workspace for a ragged N");
    check(vca_attention(fake8, fakef, fake8, fakef, fake8, NULL, fakef, fake16, 1, 2, 1024, 128, 0.0f, 1,
                        VCA_V_E4M3, NULL, NULL, NULL) == VCA_ERR_INVALID_ARG,
          "attention without an output pointer");
    check(vca_attention(fake8, fakef, fake8, fakef, fake8, fake8, fakef, fake16, 1, 2, 1024, 128, 0.0f, 1,
                        VCA_V_NVFP4, fake16, NULL, NULL) == VCA_ERR_UNSUPPORTED,
          "ExpCast with NVFP4 V");
    check(vca_group(fake16, 1, 2, 1024, 128, 8, 4, fake32, fake32, NULL, NULL, NULL, 0, NULL, NULL)
              == VCA_ERR_WORKSPACE,
          "group without a workspace");
    check(vca_prep_quant_ex(fake16, fake16, fake16, fake32, 1, 2, 1024, 128, VCA_V_E4M3, 4u, fake8, fakef, fake8,
                            fakef, fake8, NULL, fakef, fake16, fake8, 1u << 30, NULL) == VCA_ERR_INVALID_ARG,
          "prep with an undefined flag");
    return failures;
}
