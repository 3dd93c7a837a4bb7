/* A plain C consumer of the library's header: compiled with gcc -std=c11
 * (no C++), linked against libqmm.so, and run without a GPU. It exercises the
 * host-side contract only: sizes, version, and argument rejection with the
 * documented status codes before anything touches the device. */
#include <stdio.h>
#include <string.h>

#include "qmm.h"

static int fails = 0;
#define EXPECT(cond)                                                        \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "line %d: %s (last error: %s)\n", __LINE__, #cond, \
                    qmm_last_error());                                      \
            ++fails;                                                        \
        }                                                                   \
    } while (0)

int main(void) {
    EXPECT(qmm_version() > 0);
    /* byte sizes: (k/32)*18, (k/256)*144, (k/256)*210, 2k per row */
    EXPECT(qmm_weight_bytes(QMM_Q4_0, 4096, 3) == (size_t)(4096 / 32) * 18 * 3);
    EXPECT(qmm_weight_bytes(QMM_Q4_K, 4096, 3) == (size_t)(4096 / 256) * 144 * 3);
    EXPECT(qmm_weight_bytes(QMM_Q6_K, 2560, 3) == (size_t)(2560 / 256) * 210 * 3);
    EXPECT(qmm_weight_bytes(QMM_BF16, 4096, 3) == (size_t)2 * 4096 * 3);
    EXPECT(qmm_weight_bytes(QMM_Q4_K, 300, 1) == 0);
    EXPECT(qmm_weight_bytes(QMM_AFFINE4, 128, 2) == 128);

    /* the plain seven-argument call with invalid shapes: rejected on the host */
    float dummy[4];
    EXPECT(qmm_matmul(QMM_Q4_K, dummy, dummy, 300, 8, 1, dummy) == QMM_ERR_SHAPE);
    EXPECT(qmm_matmul(99, dummy, dummy, 256, 8, 1, dummy) == QMM_ERR_FORMAT);
    EXPECT(qmm_matmul(QMM_Q4_K, dummy, dummy, 256, 8, 0, dummy) == QMM_ERR_SHAPE);
    EXPECT(strlen(qmm_last_error()) > 0);

    qmm_args a;
    memset(&a, 0, sizeof a);
    a.fmt = QMM_Q4_K;
    a.w = dummy;
    a.x = dummy;
    a.y = dummy;
    a.k = 256;
    a.n = 8;
    a.n_tokens = 1;
    a.w_len = 10;
    EXPECT(qmm_matmul_ex(&a) == QMM_ERR_SIZE);
    a.w_len = 0;
    a.j_start = 5;
    a.j_end = 3;
    EXPECT(qmm_matmul_ex(&a) == QMM_ERR_RANGE);
    a.j_start = a.j_end = 4; /* empty tile: OK, nothing launched */
    EXPECT(qmm_matmul_ex(&a) == QMM_OK);
    a.j_start = a.j_end = 0;
    a.y = NULL;
    EXPECT(qmm_matmul_ex(&a) == QMM_ERR_NULL);
    a.y = dummy;
    a.fmt = QMM_AFFINE4;
    a.k = 128;
    EXPECT(qmm_matmul_ex(&a) == QMM_ERR_FORMAT); /* affine weights need qmm_matmul_affine */
    EXPECT(qmm_matmul_glu(&a, dummy, QMM_ACT_SWIGLU) == QMM_ERR_FORMAT);
    a.fmt = QMM_Q4_K;
    a.k = 256;
    EXPECT(qmm_matmul_glu(&a, dummy, 7) == QMM_ERR_FORMAT);
    int32_t ids[2] = {0, 0};
    EXPECT(qmm_matmul_experts(&a, ids, 0, 1) == QMM_ERR_SHAPE);
    EXPECT(qmm_dequant(QMM_Q4_K, dummy, 100, 1, dummy, NULL) == QMM_ERR_SHAPE);

    if (fails) {
        fprintf(stderr, "%d check(s) failed\n", fails);
        return 1;
    }
    printf("c abi consumer: all checks passed\n");
    return 0;
}
