/* A plain C11 client of include/nvfp4.h: the library is usable without Python or C++.
 * Built and run by tests/test_c_abi_client.py on the CPU: it exercises the calls that need
 * no GPU (sizes, status strings, host argument checks, which launch nothing). */
#include <stdio.h>
#include <string.h>

#include "nvfp4.h"

int main(void) {
    int fails = 0;
#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond);   \
            ++fails;                                                 \
        }                                                            \
    } while (0)
    CHECK(strcmp(nvfp4_status_string(NVFP4_OK), "ok") == 0);
    CHECK(nvfp4_scales_mma_bytes(128, 256) == 2048);
    CHECK(nvfp4_mx_scales_mma_bytes(128, 256) == 1024);
    CHECK(nvfp4_sqrelu_maxima_bytes(-1) == 0);      /* sized per device: no such device */
    CHECK(nvfp4_gemm_workspace_bytes(-1) == 0);

    nvfp4_qparams p;
    memset(&p, 0, sizeof p);
    p.block = NVFP4_BLOCK_1X16_ROW;
    p.round = NVFP4_ROUND_RNE;
    float s_dec_dummy;
    nvfp4_qtensor q;
    memset(&q, 0, sizeof q);
    q.codes = (uint8_t*)0x1000;
    q.scales = (uint8_t*)0x1000;
    q.s_dec = &s_dec_dummy;
    q.rows = 32;
    q.cols = 40;                                     /* 40 % 16 != 0: rejected on the host */
    CHECK(nvfp4_quantize((const void*)0x1000, NVFP4_BF16, 32, 40, 40, &p, &q, (void*)0x2000, 1 << 16, NULL, NULL) ==
          NVFP4_ERR_SHAPE);
    q.cols = 64;
    p.rht = 1;                                       /* the RHT needs column blocks */
    CHECK(nvfp4_quantize((const void*)0x1000, NVFP4_BF16, 32, 64, 64, &p, &q, (void*)0x2000, 1 << 16, NULL, NULL) ==
          NVFP4_ERR_INVALID_ARG);
    nvfp4_qtensor a, b;
    memset(&a, 0, sizeof a);
    memset(&b, 0, sizeof b);
    a.codes = b.codes = (uint8_t*)0x1000;
    a.scales_mma = b.scales_mma = (uint8_t*)0x1000;
    a.s_dec = b.s_dec = &s_dec_dummy;
    a.rows = 128; a.cols = 256;
    b.rows = 256; b.cols = 128;                      /* K mismatch */
    CHECK(nvfp4_gemm(&a, &b, (void*)0x4000, NVFP4_BF16, 256, NULL, NULL) == NVFP4_ERR_SHAPE);
    CHECK(nvfp4_gemm_ws(&a, &b, (void*)0x4000, NVFP4_BF16, 256, NULL, 0, NULL, NULL) == NVFP4_ERR_SHAPE);
    CHECK(nvfp4_mx_gemm(&a, &b, (void*)0x4000, NVFP4_F32, 256, NULL, NULL) == NVFP4_ERR_UNSUPPORTED);
    printf("%s %d\n", fails ? "failed" : "ok", fails);
    return fails != 0;
}
