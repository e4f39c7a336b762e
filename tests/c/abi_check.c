/* Compiled as C99 against include/igemm.h and linked with libigemm.so by
 * tests/test_c_header.py: the header is valid C and the argument checks and
 * host-only queries answer as documented, with no GPU needed. */
#include <stdio.h>
#include <string.h>
#include "igemm.h"

#define EXPECT(cond)                                                  \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "line %d: %s\n", __LINE__, #cond);        \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main(void)
{
    const uint8_t *fake = (const uint8_t *)(uintptr_t)0x10000;
    int32_t *c = (int32_t *)(uintptr_t)0x20000;
    int plan[4] = {0, 0, 0, 0};

    EXPECT(i4i4_gemm(fake, fake, c, -1, 8, 64, 0) == IGEMM_INVALID_ARGUMENT);
    EXPECT(i4i4_gemm(fake, fake, c, 8, 8, 48, 0) == IGEMM_UNSUPPORTED_SHAPE);
    EXPECT(i4i4_gemm(fake, fake, c, 8, 8, 33554432, 0) == IGEMM_OVERFLOW_BOUND);
    EXPECT(w4a8_gemm((const int8_t *)fake, fake, c, 8, 8, 2097152, 0) == IGEMM_OVERFLOW_BOUND);
    EXPECT(w4a8_gemm((const int8_t *)fake, fake, c + 1, 8, 8, 64, 0) == IGEMM_MISALIGNED);
    EXPECT(w4a8_gemm(NULL, NULL, NULL, 0, 8, 64, 0) == IGEMM_OK);
    EXPECT(i4i4_gemm_host(fake, fake, NULL, 8, 8, 64, 0) == IGEMM_INVALID_ARGUMENT);
    EXPECT(fp8_gemm(fake, fake, (float *)c, 8, 8, 24, 0) == IGEMM_UNSUPPORTED_SHAPE);
    EXPECT(pack_int4(NULL, NULL, 4, 7, 0) == IGEMM_UNSUPPORTED_SHAPE);
    EXPECT(igemm_strerror(IGEMM_MISALIGNED) != NULL && strlen(igemm_strerror(IGEMM_MISALIGNED)) > 0);

    /* the decode shape on a 152-SM part with room for 76 pairs and 36 quads */
    EXPECT(igemm_skinny_plan(1, 16, 28672, 8192, 152, 76, 36, plan) == IGEMM_OK);
    EXPECT(plan[0] >= 1 && plan[1] > 0 && plan[1] % 256 == 0 && plan[2] >= 1 && plan[2] <= 152);
    EXPECT(plan[3] == 1 || plan[3] == 2 || plan[3] == 4);
    EXPECT(igemm_skinny_plan(1, 65, 28672, 8192, 152, 76, 36, plan) == IGEMM_INVALID_ARGUMENT);
    {
        int ss[7] = {0};
        /* W4A8 4096^3 on 76 pairs: 512 tiles, the last 56 dealt out as ranges of k blocks */
        EXPECT(igemm_ss_plan(1, 4096, 4096, 4096, 76, ss) == IGEMM_OK);
        EXPECT(ss[0] == 1 && ss[3] == 56 && ss[4] > 0 && ss[4] < 32 && ss[5] == 76 && ss[6] == 1);
        EXPECT(igemm_ss_plan(2, 4096, 4096, 4096, 76, ss) == IGEMM_INVALID_ARGUMENT);
        /* W4A8 decode: skinny; 256 activations against 28672 x 8192 weights: packed weights */
        EXPECT(igemm_route(1, 16, 28672, 8192, 152, 76, 36, ss) == IGEMM_OK && ss[0] == 0);
        EXPECT(igemm_route(1, 256, 28672, 8192, 152, 76, 36, ss) == IGEMM_OK && ss[0] == 4);
        EXPECT(igemm_route(0, 8192, 8192, 8192, 152, 76, 36, ss) == IGEMM_OK && ss[0] == 2);
        EXPECT(igemm_route(0, 8, 8, 48, 152, 76, 36, ss) == IGEMM_INVALID_ARGUMENT);
    }
    printf("c abi ok: split %d, slice %d, ctas %d, cluster %d\n", plan[0], plan[1], plan[2], plan[3]);
    return 0;
}
