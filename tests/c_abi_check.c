/* A plain C99 caller of the W12 C ABI, compiled and run by the CPU test-suite: the header must
 * compile as C, the library must link from C, and the host-only calls (shapes, status names)
 * must answer without a GPU. */
#include <stdio.h>

#include "w12.h"

int main(void) {
    w12_tensor t;
    size_t records = 0, bases = 0;
    if (w12_tensor_shape(17408, 5120, &t, &records, &bases) != W12_OK) return 1;
    w12_q8_head h;
    size_t codes8 = 0, rows8 = 0;
    if (w12_q8_shape(151936, 5120, &h, &codes8, &rows8) != W12_OK) return 2;
    w12_q6_copy c;
    size_t codes6 = 0, rows6 = 0;
    if (w12_q6_shape(151936, 5120, &c, &codes6, &rows6) != W12_OK) return 3;
    if (w12_tensor_shape(16, 12, &t, NULL, NULL) != W12_ERR_UNSUPPORTED_SHAPE) return 4;
    if (w12_gemm(NULL, NULL, 1, NULL, W12_OUT_F32, NULL, 0, NULL) != W12_ERR_INVALID_ARG) return 5;
    w12_tensor_shape(17408, 5120, &t, NULL, NULL);
    printf("%d %d %zu %zu %zu %zu %s\n", t.n_tiles, t.k_tiles, records, bases, codes8, codes6,
           w12_status_str(W12_ERR_TIMEOUT));
    return 0;
}
