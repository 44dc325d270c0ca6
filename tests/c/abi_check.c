/*
 * The C ABI used from plain C, with no Python and no torch.
 *
 *   abi_check cpu   host-side validation: every bad argument gets its
 *                   documented status and a message, and nothing is launched.
 *   abi_check gpu   cudaMalloc'd inputs and caches, kvpub_store_mla_fp8 into
 *                   three replicas, then every byte of every replica (guard
 *                   bytes included) compared with the CPU oracle, which is
 *                   linked in alongside as test infrastructure.
 *
 * Exit status 0 on success.  Built and run by tests/test_c_abi.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvpub.h"

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAILED: " __VA_ARGS__);      \
            fprintf(stderr, "\n");                        \
            return 1;                                     \
        }                                                 \
    } while (0)

static int cpu_checks(void) {
    void *a = (void *)(uintptr_t)0x10000; /* placeholder, never dereferenced */
    void *caches[2] = {(void *)(uintptr_t)0x200000, (void *)(uintptr_t)0x400000};
    kvpub_status st;
    st = kvpub_store_mla_fp8(a, 512, a, 64, a, 128, (const int64_t *)a, 16, caches, caches, 0,
                             4, 64, NULL, NULL);
    CHECK(st == KVPUB_ERR_INVALID_ARG, "R = 0 gave %d", st);
    CHECK(strlen(kvpub_last_error()) > 0, "no message for R = 0");
    st = kvpub_store_mla_fp8(a, 512, a, 64, a, 128, (const int64_t *)a, 16, caches, caches, 9,
                             4, 64, NULL, NULL);
    CHECK(st == KVPUB_ERR_TOO_MANY_REPLICAS, "R = 9 gave %d", st);
    st = kvpub_store_mla_fp8((char *)a + 2, 512, a, 64, a, 128, (const int64_t *)a, 16, caches,
                             caches, 2, 4, 64, NULL, NULL);
    CHECK(st == KVPUB_ERR_ALIGNMENT, "misaligned latent gave %d", st);
    st = kvpub_store_mla_bf16(a, 512, a, 64, a, 128, (const int64_t *)a, 16, caches, caches, 2,
                              4, 32, NULL, NULL);
    CHECK(st == KVPUB_ERR_INVALID_ARG, "block_size 32 gave %d", st);
    st = kvpub_gather_insert(a, 512, a, 64, a, 128, (const int64_t *)a, 16, caches, caches, 2, 4,
                             64, NULL, a, 100, NULL);
    CHECK(st == KVPUB_ERR_WORKSPACE, "small workspace gave %d", st);
    CHECK(kvpub_gather_workspace_bytes(10) == 14080, "workspace bytes");
    st = kvpub_epoch_wait((const unsigned long long *)a, 1, 0, (unsigned int *)a, NULL);
    CHECK(st == KVPUB_ERR_INVALID_ARG, "max_polls 0 gave %d", st);
    printf("cpu checks ok\n");
    return 0;
}

#ifdef KVPUB_ABI_CHECK_GPU
#include <cuda_runtime.h>

int64_t kvo_store_mla_fp8(const uint16_t *, int64_t, const uint16_t *, int64_t,
                          const uint16_t *, int64_t, const int64_t *, int64_t,
                          uint8_t *const *, uint8_t *const *, int, int64_t, int64_t *);

static uint32_t lcg(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return *s;
}

/* A bf16 value from the generator: random sign, exponent 100..140, mantissa. */
static uint16_t bf16_value(uint32_t *s) {
    uint32_t r = lcg(s);
    uint32_t sign = (r >> 31) << 15;
    uint32_t exp = 100u + (r >> 8) % 41u;
    return (uint16_t)(sign | (exp << 7) | (r & 0x7Fu));
}

static int gpu_checks(void) {
    const int T = 777, R = 3;
    const int64_t nb = 24, slots_total = nb * 64;
    const size_t main_bytes = (size_t)nb * 64 * KVPUB_MAIN_SLOT_BYTES;
    const size_t idx_bytes = (size_t)nb * KVPUB_INDEXER_BLOCK_BYTES;
    uint32_t seed = 12345u;

    uint16_t *lat = malloc((size_t)T * 512 * 2), *rope = malloc((size_t)T * 64 * 2),
             *idx = malloc((size_t)T * 128 * 2);
    int64_t *slots = malloc((size_t)T * 8);
    int64_t *perm = malloc((size_t)slots_total * 8);
    CHECK(lat && rope && idx && slots && perm, "host malloc");
    for (int64_t i = 0; i < (int64_t)T * 512; ++i) lat[i] = bf16_value(&seed);
    for (int64_t i = 0; i < (int64_t)T * 64; ++i) rope[i] = bf16_value(&seed);
    for (int64_t i = 0; i < (int64_t)T * 128; ++i) idx[i] = bf16_value(&seed);
    for (int64_t i = 0; i < slots_total; ++i) perm[i] = i;
    for (int64_t i = slots_total - 1; i > 0; --i) {
        int64_t j = lcg(&seed) % (uint32_t)(i + 1);
        int64_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    for (int t = 0; t < T; ++t) slots[t] = (t % 11 == 5) ? -1 : perm[t];

    void *d_lat, *d_rope, *d_idx, *d_slots, *d_main[3], *d_ixc[3];
    CHECK(cudaMalloc(&d_lat, (size_t)T * 512 * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_rope, (size_t)T * 64 * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_idx, (size_t)T * 128 * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_slots, (size_t)T * 8) == cudaSuccess, "cudaMalloc");
    cudaMemcpy(d_lat, lat, (size_t)T * 512 * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d_rope, rope, (size_t)T * 64 * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d_idx, idx, (size_t)T * 128 * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d_slots, slots, (size_t)T * 8, cudaMemcpyHostToDevice);
    uint8_t *want_main[3], *want_ixc[3];
    for (int r = 0; r < R; ++r) {
        CHECK(cudaMalloc(&d_main[r], main_bytes) == cudaSuccess, "cudaMalloc");
        CHECK(cudaMalloc(&d_ixc[r], idx_bytes) == cudaSuccess, "cudaMalloc");
        cudaMemset(d_main[r], 0xA5, main_bytes);
        cudaMemset(d_ixc[r], 0xA5, idx_bytes);
        want_main[r] = malloc(main_bytes);
        want_ixc[r] = malloc(idx_bytes);
        memset(want_main[r], 0xA5, main_bytes);
        memset(want_ixc[r], 0xA5, idx_bytes);
    }
    cudaDeviceSynchronize();

    kvpub_status st = kvpub_store_mla_fp8(d_lat, 512, d_rope, 64, d_idx, 128, d_slots, T, d_main,
                                          d_ixc, R, nb, KVPUB_BLOCK_SIZE, NULL, NULL);
    CHECK(st == KVPUB_OK, "store: %s", kvpub_last_error());
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "synchronize");

    int64_t invalid = -1;
    int64_t n = kvo_store_mla_fp8(lat, 512, rope, 64, idx, 128, slots, T, want_main, want_ixc, R,
                                  nb, &invalid);
    CHECK(invalid == 0, "oracle invalid count");
    uint8_t *got = malloc(main_bytes > idx_bytes ? main_bytes : idx_bytes);
    for (int r = 0; r < R; ++r) {
        cudaMemcpy(got, d_main[r], main_bytes, cudaMemcpyDeviceToHost);
        CHECK(memcmp(got, want_main[r], main_bytes) == 0, "Main cache %d differs", r);
        cudaMemcpy(got, d_ixc[r], idx_bytes, cudaMemcpyDeviceToHost);
        CHECK(memcmp(got, want_ixc[r], idx_bytes) == 0, "Indexer cache %d differs", r);
    }
    printf("gpu checks ok: %lld rows x %d replicas byte-exact\n", (long long)n, R);
    return 0;
}
#endif

int main(int argc, char **argv) {
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
#ifdef KVPUB_ABI_CHECK_GPU
        return gpu_checks();
#else
        fprintf(stderr, "built without the GPU part\n");
        return 2;
#endif
    }
    return cpu_checks();
}
