/*
 * A plain C program against the library's C ABI (include/fp8fg.h, linked with
 * libfp8fg.so): every entry point called with arguments that break its documented rules
 * must return FP8FG_ERR_ARG with a message, before touching any device, and empty
 * problems must return FP8FG_OK without launching. Needs no GPU: nothing here reaches
 * a CUDA call. Prints the number of checks and exits 0 when all hold.
 */
#include <stdio.h>
#include <stdint.h>
#include <string.h>

#include "fp8fg.h"

static int checks = 0, failures = 0;

static void expect(int got, int want, const char *what, const char *needle) {
    ++checks;
    const char *msg = fp8fg_last_error();
    if (got != want || (needle && !strstr(msg, needle))) {
        ++failures;
        fprintf(stderr, "FAIL %s: got %d (want %d), message \"%s\"\n", what, got, want, msg);
    }
}

int main(void) {
    /* a 16-byte aligned, never dereferenced address and a misaligned one */
    void *p = (void *)(uintptr_t)0x10000;
    void *odd = (void *)(uintptr_t)0x10008;
    const uint16_t *x = (const uint16_t *)p;
    uint8_t *q = (uint8_t *)p;
    float *s = (float *)p;

    expect(fp8fg_version() > 0 ? FP8FG_OK : -1, FP8FG_OK, "version", NULL);

    expect(fp8_quant_act_1x128(x, 4, 100, 104, 0, q, s, NULL), FP8FG_ERR_ARG, "act K % 128", "of 128");
    expect(fp8_quant_act_1x128(x, 100, 256, 256, 1, q, s, NULL), FP8FG_ERR_ARG, "act transposed M % 128", "of 128");
    expect(fp8_quant_act_1x128((const uint16_t *)odd, 4, 256, 256, 0, q, s, NULL), FP8FG_ERR_ARG, "act misaligned", "aligned");
    expect(fp8_quant_act_1x128(NULL, 0, 256, 256, 0, NULL, NULL, NULL), FP8FG_OK, "act empty", NULL);

    expect(fp8_quant_act_1x128_transposed_pair(x, 256, 256, q, s, x, 512, 512, q, s, 100, NULL), FP8FG_ERR_ARG,
           "pair M % 128", "of 128");
    expect(fp8_quant_act_1x128_transposed_pair(x, 256, 256, q, s, NULL, 512, 512, q, s, 128, NULL), FP8FG_ERR_ARG,
           "pair null", "null");

    expect(fp8_quant_w_128x128(x, 100, 256, 256, q, s, NULL), FP8FG_ERR_ARG, "weight N % 128", "of 128");
    expect(fp8_quant_w_128x128_dual(x, 128, 256, 200, q, s, q, s, NULL), FP8FG_ERR_ARG, "weight dual ldw", "ldw");
    expect(fp8_quant_act_1x128_dual(x, 100, 256, 256, q, s, q, s, NULL), FP8FG_ERR_ARG, "act dual M % 128",
           "of 128");

    expect(fp8_quant_act_delayed(x, 4, 256, 256, s, 0, q, s, NULL), FP8FG_ERR_ARG, "delayed H", "history");

    expect(fp8_blockscaled_gemm(q, s, q, s, 2, p, FP8FG_OUT_BF16, 128, 256, 256, NULL), FP8FG_ERR_ARG,
           "gemm sb_kind", "sb_kind");
    expect(fp8_blockscaled_gemm(q, s, q, s, FP8FG_SB_BLOCK_128x128, p, 7, 128, 256, 256, NULL), FP8FG_ERR_ARG,
           "gemm c_dtype", "c_dtype");
    expect(fp8_blockscaled_gemm(q, s, q, s, FP8FG_SB_BLOCK_128x128, p, FP8FG_OUT_F32, 128, 200, 256, NULL),
           FP8FG_ERR_ARG, "gemm N % 128", "of 128");
    expect(fp8_blockscaled_gemm(q, s, q, s, FP8FG_SB_BLOCK_128x128, p, FP8FG_OUT_F32, 0, 256, 256, NULL), FP8FG_OK,
           "gemm empty", NULL);
    expect(fp8_blockscaled_gemm_ws(q, s, q, s, FP8FG_SB_BLOCK_128x128, p, FP8FG_OUT_F32, 128, 256, 256, NULL, 0, NULL),
           FP8FG_ERR_ARG, "gemm_ws null workspace", "workspace");
    expect(fp8_blockscaled_gemm_e4m3(q, s, q, s, FP8FG_SB_BLOCK_128x128, q, s, 128, 200, 256, NULL), FP8FG_ERR_ARG,
           "gemm_e4m3 N % 128", "of 128");
    expect(fp8_grouped_gemm(q, s, q, s, (const int32_t *)p, 0, 128, p, FP8FG_OUT_BF16, 256, 256, NULL),
           FP8FG_ERR_ARG, "grouped E", "E=");
    expect(fp8_grouped_gemm(q, s, q, s, (const int32_t *)p, 2, 100, p, FP8FG_OUT_BF16, 256, 256, NULL),
           FP8FG_ERR_ARG, "grouped Mtot % 128", "of 128");

    printf("%d %d\n", checks, failures);
    return failures != 0;
}
