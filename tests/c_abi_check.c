/* Plain-C user of the library: compiles against include/ar_fusion.h with a C
 * compiler (C99, no C++), links libarfusion.so, and exercises the entry
 * points that need no GPU (size queries and argument checks). */
#include <stdio.h>
#include <string.h>

#include "ar_fusion.h"

static int failures = 0;

static void expect(int got, int want, const char* what)
{
    if (got != want) {
        printf("%s: got %d want %d (%s)\n", what, got, want, ar_fusion_last_error());
        ++failures;
    }
}

int main(void)
{
    size_t bytes = 0;
    const size_t up = 255;
    const size_t buf = (size_t)8 * 8192 * 7168 * 2;
    const size_t flags = (size_t)8 * AR_BARRIER_FLAG_COUNT * 4;
    size_t want;
    ar_fusion_ws* ws = NULL;
    const void* bufs[2] = {(const void*)16, (const void*)32};
    ar_fusion_ws_info info;
    ar_fusion_state st;

    expect(ar_fusion_version(), 10000, "version");
    expect(ar_fusion_workspace_bytes(8, 8192, 7168, AR_DT_BF16, &bytes), AR_OK, "bytes bf16");
    /* [buffer | flags | 3 Lamport slots | state], regions 256-byte aligned */
    want = (((buf + up) & ~up) + flags + up) & ~up;          /* Lamport region offset */
    want = (want + 3 * buf + up) & ~up;                      /* state offset */
    want = (want + sizeof(ar_fusion_state) + up) & ~up;
    if (bytes != want) {
        printf("workspace bytes %zu, expected %zu\n", bytes, want);
        ++failures;
    }
    expect(ar_fusion_workspace_bytes(8, 128, 4096, AR_DT_FP32, &bytes), AR_OK, "bytes fp32");
    expect(ar_fusion_workspace_bytes(0, 16, 512, AR_DT_BF16, &bytes), AR_ERR_UNSUPPORTED, "0 ranks");
    expect(ar_fusion_workspace_bytes(2, 16, 500, AR_DT_BF16, &bytes), AR_ERR_INVALID, "hidden 500");
    expect(ar_fusion_workspace_bytes(2, 16, 512, 9, &bytes), AR_ERR_UNSUPPORTED, "dtype 9");
    if (strlen(ar_fusion_last_error()) == 0) {
        printf("no error text after a failure\n");
        ++failures;
    }
    expect(ar_fusion_workspace_create(2, 16, 12, AR_DT_BF16, NULL, 0, NULL, &ws), AR_ERR_INVALID,
           "create hidden 12");
    expect(ar_fusion_workspace_info(NULL, &info), AR_ERR_INVALID, "info NULL");
    expect(ar_fusion_workspace_copy_state(NULL, NULL, &st), AR_ERR_INVALID, "copy_state NULL");
    expect(ar_fusion_run(NULL, NULL, 2, 16, 512, AR_DT_BF16, NULL, NULL, 1e-6f,
                         AR_RESIDUAL_OUT | AR_NORM_OUT, NULL, NULL, NULL, NULL, NULL, NULL),
           AR_ERR_INVALID, "run without workspace");
    expect(ar_fusion_sum(bufs, 2, 0, AR_DT_FP16, (void*)64, NULL), AR_OK, "empty sum");
    expect(ar_fusion_sum_ex(bufs, 2, 10, AR_DT_FP16, 7, (void*)64, NULL), AR_ERR_INVALID,
           "sum accumulate 7");
    expect(ar_fusion_run_noalloc(bufs, 17, 1, 64, AR_DT_BF16, (void*)16, (void*)16, 1e-5f,
                                 AR_RESIDUAL_OUT | AR_NORM_OUT, (void*)16, (void*)16, NULL, NULL,
                                 NULL, NULL),
           AR_ERR_UNSUPPORTED, "noalloc 17 ranks");
    expect(ar_fusion_workspace_destroy(NULL), AR_OK, "destroy NULL");
    printf("%d failures\n", failures);
    return failures != 0;
}
