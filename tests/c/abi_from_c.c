/* The carbon_gemm C ABI used from plain C (C99): the public headers compile
 * as C, and the library's validation and status paths answer without a
 * GPU.  No compute call reaches a device: every call below fails its
 * argument checks or is failed by host-side fault injection first.
 * Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "carbon_gemm.h"
#include "carbon_gemm_debug.h"

#define CHECK(cond)                                                     \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                                   \
        }                                                               \
    } while (0)

int main(void)
{
    void *fake = (void *)0x1000; /* never dereferenced */
    CHECK(carbon_abi_version() == CARBON_ABI_VERSION);
    CHECK((carbon_abi_version() >> 16) == 1 && (carbon_abi_version() & 0xffff) >= 2);
    CHECK(strcmp(carbon_status_string(CARBON_OK), "CARBON_OK") == 0);
    CHECK(strcmp(carbon_status_string(CARBON_ERR_MISALIGNED), "CARBON_ERR_MISALIGNED") == 0);
    /* argument errors come back before any device work */
    CHECK(carbon_gemm_fwd(fake, fake, fake, NULL, -1, 8, 8, CARBON_BF16, CARBON_TIER_EXACT, NULL)
          == CARBON_ERR_INVALID_ARG);
    CHECK(carbon_gemm_dx(fake, NULL, fake, 8, 8, 8, CARBON_F16, CARBON_TIER_EXACT, NULL)
          == CARBON_ERR_INVALID_ARG);
    CHECK(carbon_gemm_dw(fake, fake, fake, 8, 8, 8, CARBON_F32, CARBON_TIER_TC, NULL)
          == CARBON_ERR_UNSUPPORTED);
    CHECK(carbon_gemm_dw_f32((float *)fake, fake, fake, 8, 8, 8, (carbon_tier_t)7, NULL)
          == CARBON_ERR_INVALID_ARG);
    /* an empty output is a successful no-op */
    CHECK(carbon_gemm_fwd(fake, fake, fake, NULL, 0, 8, 8, CARBON_BF16, CARBON_TIER_EXACT, NULL)
          == CARBON_OK);
    /* host-side fault injection: the call fails as a launch would */
    setenv("CARBON_FAULT", "launch", 1);
    CHECK(carbon_gemm_fwd(fake, fake, fake, NULL, 8, 8, 8, CARBON_BF16, CARBON_TIER_TC, NULL)
          == CARBON_ERR_CUDA);
    CHECK(strstr(carbon_last_cuda_error(), "injected launch failure") != NULL);
    unsetenv("CARBON_FAULT");
    printf("ok\n");
    return 0;
}
