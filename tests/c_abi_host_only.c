/* A plain C caller of libcca.so (no Python, no torch): the ABI version, the status strings,
 * the workspace sizes, and argument checks that reject bad calls on the host before any
 * CUDA call.  It touches no GPU, so it runs anywhere the library loads.  Exit status 0 on
 * success; the failing check's line number otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "cca.h"

#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
            return __LINE__;                                       \
        }                                                          \
    } while (0)

int main(void) {
    cca_params_t p;
    memset(&p, 0, sizeof p);
    p.B = 1;
    p.Hq = 4;
    p.Hkv = 2;
    p.N = 1024;
    p.d = 128;
    p.g = 16;
    p.w = 256;
    p.dtype = CCA_BF16;
    CHECK(cca_abi_version() == CCA_ABI_VERSION);
    CHECK(strlen(cca_status_string(CCA_OK)) > 0);
    CHECK(strlen(cca_status_string(CCA_ERR_INVALID_ARG)) > 0);
    CHECK(strlen(cca_status_string(12345)) > 0);
    /* partials of B * Hq rows, MAX_SPLITS = 64 splits, d + 2 floats each */
    CHECK(cca_decode_workspace_size(&p) == (uint64_t)1 * 4 * 64 * 130 * 4);
    CHECK(cca_prefill_bwd_workspace_size(&p) > 0);
    /* fake, 16-byte aligned pointers: every call below is rejected before they are used */
    char *f = (char *)0x10000;
    cca_params_t bad = p;
    bad.N = 1000; /* not a multiple of g */
    CHECK(cca_pool(f, f, f, f, f, &bad, NULL) == CCA_ERR_INVALID_ARG);
    CHECK(cca_attn_fwd(f, f, f, f, f, f, (float *)f, &bad, NULL) == CCA_ERR_INVALID_ARG);
    CHECK(cca_decode_workspace_size(&bad) == 0);
    CHECK(cca_attn_fwd(f, f, f, f, f, f + 1, (float *)f, &p, NULL) == CCA_ERR_INVALID_ARG); /* misaligned O */
    CHECK(cca_attn_fwd_rows(f, f, f, f, f, f, (float *)f, 500, 10, 402, 108, &p, NULL) == CCA_ERR_INVALID_ARG);
    CHECK(cca_decode_kernels(&p, p.N) == CCA_ERR_INVALID_ARG);
    bad = p;
    bad.pool_mode = 3;
    bad.Hq = 18;
    bad.Hkv = 2; /* nine query heads per KV head: more than pool_mode 3 supports */
    CHECK(cca_pool(f, f, f, f, f, &bad, NULL) == CCA_ERR_UNSUPPORTED);
    printf("c abi ok\n");
    return 0;
}
