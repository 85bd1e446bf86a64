/*
 * A plain C client of libtstgemm.so, built by the tests with gcc against
 * include/tstgemm.h (no Python, no torch): the boundary is usable as a C ABI.
 *
 *   c_abi_client map M N K kind group P   host-only plan: print F(i) for every task,
 *                                         then unit 0's work list
 *   c_abi_client run M N K                on the GPU: C = A x B for small-integer
 *                                         BF16 inputs made here, checked element by
 *                                         element against an integer product
 *
 * Exit status 0 on success; 1 with a message otherwise.
 */
#include <dlfcn.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tstgemm.h"

/* the few CUDA runtime calls the GPU mode needs, resolved at run time so that the
   map mode runs on a machine without the CUDA runtime's development files */
typedef int (*malloc_fn)(void **, size_t);
typedef int (*free_fn)(void *);
typedef int (*memcpy_fn)(void *, const void *, size_t, int);
typedef int (*sync_fn)(void);

static uint16_t bf16_of_int(int v) {  /* small integers are exact in BF16 */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static int map_mode(int argc, char **argv) {
    if (argc < 8) return 1;
    int64_t M = atoll(argv[2]), N = atoll(argv[3]), K = atoll(argv[4]);
    tst_mapping mapping = {atoi(argv[5]), atoi(argv[6])};
    tst_epilogue epi = {TST_OUT_F32, 1.0f, 0, 0, 0};
    tst_plan_options opts;
    memset(&opts, 0, sizeof opts);
    opts.host_only = 1;
    opts.num_sms = atoi(argv[7]);
    opts.cta_group = 1;
    opts.bn = 128;
    tst_plan *plan = NULL;
    tst_status st = gemm_plan_create_ex(&plan, M, N, K, TST_BF16, TST_LAYOUT_A_ROW_B_NK, mapping, TST_PERSISTENT,
                                        &epi, &opts);
    if (st != TST_OK) {
        fprintf(stderr, "gemm_plan_create_ex: %s\n", gemm_status_string(st));
        return 1;
    }
    tst_plan_info info;
    gemm_plan_get_info(plan, &info);
    printf("tiles %lld grid %d\n", (long long)info.tiles, info.grid);
    for (int64_t i = 0; i < info.tiles; ++i) {
        int32_t m, n;
        if (gemm_tile_map(plan, i, &m, &n) != TST_OK) return 1;
        printf("%d %d\n", m, n);
    }
    tst_work_item items[4096];
    int64_t count = 0;
    if (gemm_work_items(plan, 0, items, 4096, &count) != TST_OK) return 1;
    printf("unit0 %lld\n", (long long)count);
    for (int64_t j = 0; j < count && j < 4096; ++j) printf("%d\n", items[j].tile);
    return gemm_plan_destroy(plan) == TST_OK ? 0 : 1;
}

static int run_mode(int argc, char **argv) {
    if (argc < 5) return 1;
    const int64_t M = atoll(argv[2]), N = atoll(argv[3]), K = atoll(argv[4]);
    const char *path = getenv("CUDART_PATH");
    void *rt = path ? dlopen(path, RTLD_NOW) : NULL;
    if (!rt) rt = dlopen("libcudart.so", RTLD_NOW);
    if (!rt) rt = dlopen("libcudart.so.13", RTLD_NOW);
    if (!rt) rt = dlopen("libcudart.so.12", RTLD_NOW);
    if (!rt) {
        fprintf(stderr, "no CUDA runtime\n");
        return 1;
    }
    malloc_fn cmalloc = (malloc_fn)dlsym(rt, "cudaMalloc");
    free_fn cfree = (free_fn)dlsym(rt, "cudaFree");
    memcpy_fn cmemcpy = (memcpy_fn)dlsym(rt, "cudaMemcpy");
    sync_fn csync = (sync_fn)dlsym(rt, "cudaDeviceSynchronize");
    if (!cmalloc || !cfree || !cmemcpy || !csync) return 1;

    uint16_t *A = malloc(sizeof(uint16_t) * M * K), *B = malloc(sizeof(uint16_t) * N * K);
    int *ai = malloc(sizeof(int) * M * K), *bi = malloc(sizeof(int) * N * K);
    float *C = malloc(sizeof(float) * M * N);
    uint64_t x = 12345;
    for (int64_t i = 0; i < M * K; ++i) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        ai[i] = (int)((x >> 33) % 9) - 4;
        A[i] = bf16_of_int(ai[i]);
    }
    for (int64_t i = 0; i < N * K; ++i) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        bi[i] = (int)((x >> 33) % 9) - 4;
        B[i] = bf16_of_int(bi[i]);
    }
    void *dA, *dB, *dC;
    if (cmalloc(&dA, sizeof(uint16_t) * M * K) || cmalloc(&dB, sizeof(uint16_t) * N * K) ||
        cmalloc(&dC, sizeof(float) * M * N))
        return 1;
    cmemcpy(dA, A, sizeof(uint16_t) * M * K, 1 /* host to device */);
    cmemcpy(dB, B, sizeof(uint16_t) * N * K, 1);

    tst_mapping mapping = {TST_MAP_GROUPED_M, 8};
    tst_epilogue epi = {TST_OUT_F32, 1.0f, 0, 0, 0};
    tst_plan *plan = NULL;
    tst_status st = gemm_plan_create(&plan, M, N, K, TST_BF16, TST_LAYOUT_A_ROW_B_NK, mapping, TST_PERSISTENT, &epi);
    if (st != TST_OK) {
        fprintf(stderr, "gemm_plan_create: %s\n", gemm_status_string(st));
        return 1;
    }
    st = gemm_run(plan, dA, dB, dC, NULL, NULL, NULL);
    if (st == TST_OK) st = gemm_status_query(plan, NULL);
    if (st != TST_OK) {
        fprintf(stderr, "run: %s\n", gemm_status_string(st));
        return 1;
    }
    csync();
    cmemcpy(C, dC, sizeof(float) * M * N, 2 /* device to host */);
    int64_t bad = 0;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            long s = 0;
            for (int64_t k = 0; k < K; ++k) s += (long)ai[i * K + k] * bi[j * K + k];
            if ((float)s != C[i * N + j]) ++bad;
        }
    gemm_plan_destroy(plan);
    cfree(dA);
    cfree(dB);
    cfree(dC);
    printf("mismatches %lld of %lld\n", (long long)bad, (long long)(M * N));
    return bad == 0 ? 0 : 1;
}

int main(int argc, char **argv) {
    if (argc >= 2 && strcmp(argv[1], "map") == 0) return map_mode(argc, argv);
    if (argc >= 2 && strcmp(argv[1], "run") == 0) return run_mode(argc, argv);
    fprintf(stderr, "usage: c_abi_client map M N K kind group P | run M N K\n");
    return 1;
}
