/*
 * Plain C use of the relayout library, without PyTorch: allocate with the
 * CUDA runtime, pack a [T][3][H][D] tensor, unpack it again through the
 * single-rank (P = 1) exchange identity, and compare on the host.  Also
 * checks that a rejected call returns the documented status.  Built and run
 * by tests/test_gpu_c_driver.py; exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "vf_relayout.h"

#define CHECK(x)                                                              \
    do {                                                                      \
        if (!(x)) {                                                           \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #x);  \
            return 1;                                                         \
        }                                                                     \
    } while (0)

int main(void) {
    const int64_t T = 37, H = 6, D = 16, P = 1, C = 3;
    const int64_t n = 3 * T * H * D;
    const int64_t st[4] = {3 * H * D, H * D, D, 1};
    uint16_t *h_src = malloc(n * 2), *h_out = malloc(n * 2);
    CHECK(h_src && h_out);
    for (int64_t i = 0; i < n; ++i) h_src[i] = (uint16_t)(i * 2654435761u >> 7);

    void *d_src = NULL, *d_packed = NULL, *d_q = NULL, *d_k = NULL, *d_v = NULL;
    CHECK(cudaMalloc(&d_src, n * 2) == cudaSuccess);
    CHECK(cudaMalloc(&d_packed, n * 2) == cudaSuccess);
    CHECK(cudaMalloc(&d_q, n * 2 / 3) == cudaSuccess);
    CHECK(cudaMalloc(&d_k, n * 2 / 3) == cudaSuccess);
    CHECK(cudaMalloc(&d_v, n * 2 / 3) == cudaSuccess);
    CHECK(cudaMemcpy(d_src, h_src, n * 2, cudaMemcpyHostToDevice) == cudaSuccess);

    CHECK(vf_packed_elems(VF_OP_QKV_PACK, T, H, D, P, C) == n);
    CHECK(vf_qkv_pack(d_src, st, T, H, D, P, C, d_packed, NULL) == VF_OK);
    /* with one rank the received buffer is the packed one */
    CHECK(vf_qkv_unpack(d_packed, T, H, D, P, C, d_q, d_k, d_v, NULL, NULL) == VF_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);

    /* Q, K, V must be the three slabs of the source */
    for (int s = 0; s < 3; ++s) {
        void *d = s == 0 ? d_q : s == 1 ? d_k : d_v;
        CHECK(cudaMemcpy(h_out, d, n * 2 / 3, cudaMemcpyDeviceToHost) == cudaSuccess);
        for (int64_t t = 0; t < T; ++t)
            for (int64_t x = 0; x < H * D; ++x)
                CHECK(h_out[t * H * D + x] == h_src[t * 3 * H * D + s * H * D + x]);
    }

    /* rejected before any launch: H % P != 0 */
    CHECK(vf_qkv_pack(d_src, st, T, H, D, 4, C, d_packed, NULL) == VF_ERR_ARG);
    CHECK(strlen(vf_status_string(VF_ERR_ARG)) > 0);

    cudaFree(d_src);
    cudaFree(d_packed);
    cudaFree(d_q);
    cudaFree(d_k);
    cudaFree(d_v);
    free(h_src);
    free(h_out);
    printf("c driver ok\n");
    return 0;
}
