/* A plain C program against the C ABI of include/shmm.h, with no Python in
 * between.  It plans the worked example of "Sharded matrix multiplication and
 * result ownership" (Engineering example: two ranks split the contracted dim,
 * the result is reduce-scattered by rows) and checks the planner's answers
 * and its argument errors.  Built with -DSHMM_C_GPU and run with --gpu, it
 * also runs an integer-valued sharded matmul on the device, through shmm_run
 * and through shmm_run_host, and compares every output element with a host
 * triple loop; integers are exact in bf16 and fp32, so the comparison is
 * exact.  Prints "OK" and exits 0 when every check passes. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "shmm.h"

#ifdef SHMM_C_GPU
#include <cuda_runtime.h>
#endif

static int fails = 0;
#define CHECK(cond, ...)                                              \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__);      \
            fprintf(stderr, __VA_ARGS__);                             \
            fprintf(stderr, " (%s)\n", shmm_last_error());            \
            ++fails;                                                  \
        }                                                             \
    } while (0)

static shmm_mesh_t make_mesh(int naxes, const char *const *names, const int *sizes) {
    shmm_mesh_t m;
    memset(&m, 0, sizeof m);
    m.naxes = naxes;
    for (int a = 0; a < naxes; ++a) {
        strncpy(m.name[a], names[a], SHMM_AXIS_NAME_LEN - 1);
        m.size[a] = sizes[a];
    }
    return m;
}

/* rows split by mesh axis r (-1: not split), columns by c */
static shmm_spec_t make_spec(int r, int c) {
    shmm_spec_t s;
    memset(&s, 0, sizeof s);
    if (r >= 0) s.axes[0][s.naxes[0]++] = r;
    if (c >= 0) s.axes[1][s.naxes[1]++] = c;
    return s;
}

static void check_planner(void) {
    const char *y[] = {"Y"};
    const int two[] = {2};
    const shmm_mesh_t m = make_mesh(1, y, two);
    const shmm_spec_t sA = make_spec(-1, 0), sB = make_spec(0, -1), sC = make_spec(0, -1);
    shmm_plan_t *p = NULL;
    shmm_status_t st = shmm_plan(&m, &sA, &sB, &sC, 2, 2, 2, SHMM_F32, SHMM_F32, 0, &p);
    CHECK(st == SHMM_OK && p, "plan of the worked example: %s", shmm_status_string(st));
    if (!p) return;
    shmm_plan_info_t info;
    CHECK(shmm_plan_query(p, &info) == SHMM_OK, "query");
    CHECK(info.case_id == 3, "case %d, want 3", info.case_id);
    CHECK(info.collective == SHMM_COLL_REDUCE_SCATTER && info.scatter_dim == 0, "reduce-scatter over rows");
    CHECK(info.nranks == 2 && info.group_size == 2 && info.ngroups == 1, "one group of two ranks");
    CHECK(info.payload_reduce_scatter == 8, "reduce-scatter payload %lld B per rank, the page prints 8",
          (long long)info.payload_reduce_scatter);
    for (int r = 0; r < 2; ++r) {
        int64_t off[2], ext[2];
        CHECK(shmm_plan_rank_box(p, SHMM_TENSOR_C, r, off, ext) == SHMM_OK, "C box");
        CHECK(off[0] == r && off[1] == 0 && ext[0] == 1 && ext[1] == 2, "rank %d owns row %d", r, r);
        CHECK(shmm_plan_rank_box(p, SHMM_TENSOR_A, r, off, ext) == SHMM_OK, "A box");
        CHECK(off[0] == 0 && off[1] == r && ext[0] == 2 && ext[1] == 1, "rank %d holds column %d of A", r, r);
    }
    CHECK(shmm_plan_rank_box(p, SHMM_TENSOR_C, 2, (int64_t[2]){0}, (int64_t[2]){0}) == SHMM_ERR_SHAPE,
          "rank out of range");
    CHECK(shmm_plan_destroy(p) == SHMM_OK, "destroy");

    /* errors: an uneven split, an output split twice by one axis, NULLs */
    p = NULL;
    CHECK(shmm_plan(&m, &sA, &sB, &sC, 3, 2, 2, SHMM_F32, SHMM_F32, 0, &p) == SHMM_ERR_SHAPE && !p,
          "I = 3 over 2 ranks");
    const shmm_spec_t bad = make_spec(0, 0);
    CHECK(shmm_plan(&m, &sA, &sB, &bad, 2, 2, 2, SHMM_F32, SHMM_F32, 0, &p) != SHMM_OK && !p,
          "C[I_Y,K_Y] rejected");
    CHECK(shmm_plan(NULL, &sA, &sB, &sC, 2, 2, 2, SHMM_F32, SHMM_F32, 0, &p) == SHMM_ERR_NULL, "NULL mesh");
    CHECK(shmm_run(NULL, NULL, NULL, NULL, NULL, 0, NULL) == SHMM_ERR_NULL, "NULL plan");
    CHECK(strcmp(shmm_status_string(SHMM_OK), "SHMM_OK") == 0, "status string");
    CHECK(shmm_version() == 100, "version");
}

#ifdef SHMM_C_GPU
/* bf16 bits of a small integer (exact: the low 16 bits of its fp32 are 0) */
static uint16_t bf16_of(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

static void check_gpu(void) {
    /* {X:2,Y:2}, A[I_X,J_Y], B[J_Y,K], C[I_X,K]: the all-reduce over Y fused
     * into the tensor-core GEMM, bf16 in, fp32 out */
    const int64_t I = 256, J = 512, K = 384;
    const char *xy[] = {"X", "Y"};
    const int sizes[] = {2, 2};
    const shmm_mesh_t m = make_mesh(2, xy, sizes);
    const shmm_spec_t sA = make_spec(0, 1), sB = make_spec(1, -1), sC = make_spec(0, -1);
    shmm_plan_t *p = NULL;
    CHECK(shmm_plan(&m, &sA, &sB, &sC, I, J, K, SHMM_BF16, SHMM_F32, SHMM_FLAG_FUSED, &p) == SHMM_OK, "plan");
    if (!p) return;
    shmm_plan_info_t info;
    shmm_plan_query(p, &info);
    CHECK(info.tensor_core == 1 && info.fused == 1, "tensor cores, fused");

    float *A = malloc(sizeof(float) * I * J), *B = malloc(sizeof(float) * J * K);
    uint16_t *Ah = malloc(2 * I * J), *Bh = malloc(2 * J * K);
    float *C = malloc(sizeof(float) * I * K), *Ch = malloc(sizeof(float) * I * K);
    uint32_t s = 12345u;
    for (int64_t i = 0; i < I * J; ++i) {
        s = s * 1664525u + 1013904223u;
        A[i] = (float)((int)(s >> 24) % 9 - 4);
        Ah[i] = bf16_of(A[i]);
    }
    for (int64_t i = 0; i < J * K; ++i) {
        s = s * 1664525u + 1013904223u;
        B[i] = (float)((int)(s >> 24) % 9 - 4);
        Bh[i] = bf16_of(B[i]);
    }
    for (int64_t i = 0; i < I; ++i)
        for (int64_t k = 0; k < K; ++k) {
            int64_t acc = 0;
            for (int64_t j = 0; j < J; ++j) acc += (int64_t)A[i * J + j] * (int64_t)B[j * K + k];
            C[i * K + k] = (float)acc;
        }

    void *A_r[4], *B_r[4], *C_r[4];
    for (int r = 0; r < 4; ++r) {
        int64_t off[2], ext[2];
        shmm_plan_rank_box(p, SHMM_TENSOR_A, r, off, ext);
        cudaMalloc(&A_r[r], 2 * ext[0] * ext[1]);
        cudaMemcpy2D(A_r[r], 2 * ext[1], Ah + off[0] * J + off[1], 2 * J, 2 * ext[1], ext[0], cudaMemcpyHostToDevice);
        shmm_plan_rank_box(p, SHMM_TENSOR_B, r, off, ext);
        cudaMalloc(&B_r[r], 2 * ext[0] * ext[1]);
        cudaMemcpy2D(B_r[r], 2 * ext[1], Bh + off[0] * K + off[1], 2 * K, 2 * ext[1], ext[0], cudaMemcpyHostToDevice);
        shmm_plan_rank_box(p, SHMM_TENSOR_C, r, off, ext);
        cudaMalloc(&C_r[r], 4 * ext[0] * ext[1]);
    }
    size_t ws_bytes = 0;
    shmm_workspace_size(p, &ws_bytes);
    void *ws = NULL;
    if (ws_bytes) cudaMalloc(&ws, ws_bytes);
    CHECK(shmm_run(p, (const void *const *)A_r, (const void *const *)B_r, C_r, ws, ws_bytes, NULL) == SHMM_OK,
          "shmm_run");
    CHECK(shmm_sync_status(NULL) == SHMM_OK, "device status");
    for (int r = 0; r < 4; ++r) {
        int64_t off[2], ext[2];
        shmm_plan_rank_box(p, SHMM_TENSOR_C, r, off, ext);
        float *got = malloc(4 * ext[0] * ext[1]);
        cudaMemcpy(got, C_r[r], 4 * ext[0] * ext[1], cudaMemcpyDeviceToHost);
        int bad = 0;
        for (int64_t i = 0; i < ext[0]; ++i)
            for (int64_t k = 0; k < ext[1]; ++k) bad += got[i * ext[1] + k] != C[(off[0] + i) * K + off[1] + k];
        CHECK(bad == 0, "rank %d: %d elements differ from the host triple loop", r, bad);
        free(got);
        cudaMemset(C_r[r], 0, 4 * ext[0] * ext[1]);
    }
    /* the same from host memory: global A, B in, global C out */
    memset(Ch, 0, sizeof(float) * I * K);
    CHECK(shmm_run_host(p, Ah, Bh, Ch, A_r, B_r, C_r, ws, ws_bytes, NULL) == SHMM_OK, "shmm_run_host");
    CHECK(shmm_sync_status(NULL) == SHMM_OK, "device status");
    int bad = 0;
    for (int64_t i = 0; i < I * K; ++i) bad += Ch[i] != C[i];
    CHECK(bad == 0, "shmm_run_host: %d elements differ", bad);
    for (int r = 0; r < 4; ++r) {
        cudaFree(A_r[r]);
        cudaFree(B_r[r]);
        cudaFree(C_r[r]);
    }
    if (ws) cudaFree(ws);
    free(A); free(B); free(Ah); free(Bh); free(C); free(Ch);
    shmm_plan_destroy(p);
}
#endif

int main(int argc, char **argv) {
    check_planner();
#ifdef SHMM_C_GPU
    if (argc > 1 && strcmp(argv[1], "--gpu") == 0) check_gpu();
#else
    (void)argc;
    (void)argv;
#endif
    if (fails) {
        fprintf(stderr, "%d check(s) failed\n", fails);
        return 1;
    }
    printf("OK\n");
    return 0;
}
