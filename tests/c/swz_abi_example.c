/*
 * swz_abi_example.c -- a plain C99 caller of the library's C ABI (swz.h).
 *
 * Without arguments it exercises the host entry points only.  With --gpu it
 * also allocates device memory through the CUDA runtime, runs a forward and an
 * inverse relayout of 256 tiles of 64 x 64 16-bit elements under
 * Swizzle<3,3,3>, and checks dst[sw(i)] == src[i] per tile and the round trip.
 * Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "swz.h"

static int fail(const char *what) {
    fprintf(stderr, "FAIL: %s\n", what);
    return 1;
}

static int host_checks(void) {
    uint64_t c = 0;
    char text[256];
    int64_t n;
    if (swz_apply(673, 5, 0, 6) != 683) return fail("swz_apply");
    if (swz_slice_collision(0x3f, 2, 0, 2, &c) != SWZ_OK) return fail("swz_slice_collision status");
    if (c != (0x3f & ~swz_apply(0x3f, 2, 0, 2))) return fail("swz_slice_collision value");
    if (swz_slice_collision(1, 3, 0, 0, &c) != SWZ_ERR_PARAM) return fail("S = 0 rejected");
    n = swz_layout_text(text, (int64_t)sizeof text, 2, 4, 4, 2, 0, 2);
    if (n <= 0 || (int64_t)strlen(text) != n) return fail("swz_layout_text");
    if (strncmp(swz_status_string(SWZ_ERR_ALIAS), "SWZ_ERR_ALIAS", 13) != 0) return fail("swz_status_string");
    if (swz_version() < 100) return fail("swz_version");
    return 0;
}

static int gpu_checks(void) {
    enum { TILES = 256, ROWS = 64, COLS = 64, TE = ROWS * COLS, N = TILES * TE };
    uint16_t *h_src = malloc(N * sizeof(uint16_t)), *h_phys = malloc(N * sizeof(uint16_t));
    uint16_t *h_back = malloc(N * sizeof(uint16_t));
    void *d_src = NULL, *d_phys = NULL, *d_back = NULL;
    int64_t t, i;
    int rc = 0;
    if (!h_src || !h_phys || !h_back) return fail("host allocation");
    for (i = 0; i < N; ++i) h_src[i] = (uint16_t)(i * 2654435761u >> 7);
    if (cudaMalloc(&d_src, N * 2) != cudaSuccess || cudaMalloc(&d_phys, N * 2) != cudaSuccess ||
        cudaMalloc(&d_back, N * 2) != cudaSuccess)
        return fail("cudaMalloc");
    cudaMemcpy(d_src, h_src, N * 2, cudaMemcpyHostToDevice);
    if (swz_relayout(d_phys, d_src, TILES, ROWS, COLS, 2, 3, 3, 3, 0, NULL) != SWZ_OK) rc = fail("forward");
    if (swz_relayout(d_back, d_phys, TILES, ROWS, COLS, 2, 3, 3, 3, 1, NULL) != SWZ_OK) rc = fail("inverse");
    if (cudaDeviceSynchronize() != cudaSuccess) rc = fail("synchronize");
    cudaMemcpy(h_phys, d_phys, N * 2, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_back, d_back, N * 2, cudaMemcpyDeviceToHost);
    for (t = 0; t < TILES && !rc; ++t)
        for (i = 0; i < TE; ++i)
            if (h_phys[t * TE + (int64_t)swz_apply((uint64_t)i, 3, 3, 3)] != h_src[t * TE + i]) {
                rc = fail("forward placement");
                break;
            }
    if (!rc && memcmp(h_back, h_src, N * 2) != 0) rc = fail("round trip");
    cudaFree(d_src);
    cudaFree(d_phys);
    cudaFree(d_back);
    free(h_src);
    free(h_phys);
    free(h_back);
    return rc;
}

int main(int argc, char **argv) {
    int rc = host_checks();
    if (!rc && argc > 1 && strcmp(argv[1], "--gpu") == 0) rc = gpu_checks();
    if (!rc) printf("swz_abi_example: ok\n");
    return rc;
}
