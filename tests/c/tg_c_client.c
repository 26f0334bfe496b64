/*
 * A plain C client of include/tg_sgemm.h (no Python, no CUDA runtime calls of
 * its own): host buffers go through tg_sgemm_host, so the program links only
 * libtg_sgemm.so, plus the oracle library to check the results.
 *
 *   tg_c_client cpu   argument checks and planning (no GPU needed)
 *   tg_c_client gpu   products on the current GPU, bit-exact on integer data
 *
 * Prints "C ABI OK" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tg_sgemm.h"

int tg_oracle_sgemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                    int64_t ldb, float* C, int64_t ldc);
int tg_oracle_sgemm_general(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                            float* C, int64_t ldc);

static uint32_t lcg_state = 12345u;
static int small_int(void) { /* uniform on {-2, ..., 2} */
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return (int)((lcg_state >> 16) % 5u) - 2;
}

#define CHECK(cond, what)                                  \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "FAILED: %s (line %d)\n", what, __LINE__); \
            return 1;                                      \
        }                                                  \
    } while (0)

static int cpu_checks(void) {
    float x[16];
    tg_plan_info info;
    CHECK(tg_sgemm(-1, 4, 4, x, 4, x, 4, x, 4, NULL) == TG_ERR_INVALID_VALUE, "negative M");
    CHECK(tg_sgemm(4, 4, 8, x, 7, x, 4, x, 4, NULL) == TG_ERR_INVALID_VALUE, "lda < K");
    CHECK(tg_sgemm(0, 4, 4, NULL, 4, NULL, 4, NULL, 4, NULL) == TG_OK, "empty output is a no-op");
    CHECK(tg_sgemm_general(2, 0, 4, 4, 4, 1.0f, x, 4, x, 4, 0.0f, x, 4, NULL, NULL) == TG_ERR_INVALID_VALUE,
          "bad op");
    CHECK(tg_sgemm_plan(8192, 8192, 8192, NULL, 8192, NULL, 8192, NULL, 8192, TG_PATH_AUTO, 0, 152, &info) ==
              TG_OK, "plan");
    CHECK(info.path == TG_PATH_TF32X3 && info.tiles_m == 64 && info.tiles_n == 32 && info.grid == 152,
          "plan fields");
    CHECK(strncmp(tg_status_string(TG_ERR_TIMEOUT), "TG_ERR_TIMEOUT", 14) == 0, "status string");
    CHECK(tg_sgemm_version() == 103, "version");
    return 0;
}

static int gpu_checks(void) {
    const int M = 300, N = 260, K = 700;
    float* A = malloc(sizeof(float) * M * K);
    float* B = malloc(sizeof(float) * K * N);
    float* At = malloc(sizeof(float) * K * M);
    float* C = malloc(sizeof(float) * M * N);
    float* R = malloc(sizeof(float) * M * N);
    CHECK(A && B && At && C && R, "host allocation");
    for (int i = 0; i < M * K; ++i) A[i] = (float)small_int();
    for (int i = 0; i < K * N; ++i) B[i] = (float)small_int();
    for (int i = 0; i < M; ++i)
        for (int k = 0; k < K; ++k) At[(size_t)k * M + i] = A[(size_t)i * K + k];
    CHECK(tg_oracle_sgemm(M, N, K, A, K, B, N, R, N) == 0, "oracle");
    for (int path = TG_PATH_FFMA; path <= TG_PATH_TF32_BF16; ++path) {
        tg_sgemm_opts o;
        memset(&o, 0, sizeof o);
        o.path = path;
        memset(C, 0xFF, sizeof(float) * M * N);
        CHECK(tg_sgemm_host(M, N, K, A, K, B, N, C, N, NULL, &o) == TG_OK, "tg_sgemm_host");
        CHECK(memcmp(C, R, sizeof(float) * M * N) == 0, "host product is bit-exact on integers");
    }
    CHECK(tg_sgemm_sync_status(NULL) == TG_OK, "no timeout recorded");
    /* the oracle's general form with A stored transposed gives the same bits */
    CHECK(tg_oracle_sgemm_general(1, 0, M, N, K, 1.0f, At, M, B, N, 0.0f, C, N) == 0, "oracle general");
    CHECK(memcmp(C, R, sizeof(float) * M * N) == 0, "oracle general agrees");
    free(A); free(B); free(At); free(C); free(R);
    return 0;
}

int main(int argc, char** argv) {
    const int gpu = argc > 1 && strcmp(argv[1], "gpu") == 0;
    if (cpu_checks() != 0) return 1;
    if (gpu && gpu_checks() != 0) return 1;
    printf("C ABI OK\n");
    return 0;
}
