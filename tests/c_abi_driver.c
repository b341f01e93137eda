/*
 * Plain C use of the relayout library, without PyTorch: allocate with the
 * CUDA runtime, pack a [T][3][H][D] tensor, unpack it again through the
 * single-rank (P = 1) exchange identity, and compare on the host; the same
 * through the opt-in INT8 and E4M3 transport on exactly quantisable rows.
 * Also checks that a rejected call returns the documented status.  Built and run
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

    /* the descriptor entry: P = 2 destinations in both block orders; the
     * slot-major buffer must hold the chunk-major blocks at the offsets the
     * two piece tables give */
    {
        const int64_t P2 = 2;
        void *d_cm = NULL, *d_sm = NULL;
        CHECK(cudaMalloc(&d_cm, n * 2) == cudaSuccess);
        CHECK(cudaMalloc(&d_sm, n * 2) == cudaSuccess);
        vf_relayout_desc desc;
        memset(&desc, 0, sizeof(desc));
        desc.op = VF_OP_QKV_PACK;
        desc.T = T; desc.H = H; desc.D = D; desc.P = P2; desc.C = C;
        desc.c_begin = 0; desc.c_count = C;
        for (int s = 0; s < 3; ++s) desc.strided[s] = (char *)d_src + 2 * s * H * D;
        desc.strides[0] = 3 * H * D; desc.strides[1] = D; desc.strides[2] = 1;
        desc.order = VF_ORDER_CHUNK_MAJOR;
        desc.packed = d_cm;
        CHECK(vf_relayout(&desc, NULL) == VF_OK);
        desc.order = VF_ORDER_SLOT_MAJOR;
        desc.packed = d_sm;
        CHECK(vf_relayout(&desc, NULL) == VF_OK);
        desc.order = 7;
        CHECK(vf_relayout(&desc, NULL) == VF_ERR_ARG);
        CHECK(cudaDeviceSynchronize() == cudaSuccess);

        uint16_t *h_cm = malloc(n * 2), *h_sm = malloc(n * 2);
        CHECK(h_cm && h_sm);
        CHECK(cudaMemcpy(h_cm, d_cm, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
        CHECK(cudaMemcpy(h_sm, d_sm, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
        int64_t ts[8], tl[8], off_cm[8], off_sm[8];
        CHECK(vf_piece_table_ex(VF_OP_QKV_PACK, VF_ORDER_CHUNK_MAJOR, T, H, D, P2, C,
                                ts, tl, off_cm, 8) == P2 * C);
        CHECK(vf_piece_table_ex(VF_OP_QKV_PACK, VF_ORDER_SLOT_MAJOR, T, H, D, P2, C,
                                ts, tl, off_sm, 8) == P2 * C);
        for (int64_t e = 0; e < P2 * C; ++e) {
            const int64_t len = tl[e] * 3 * (H / P2) * D;
            CHECK(memcmp(h_cm + off_cm[e], h_sm + off_sm[e], len * 2) == 0);
        }
        free(h_cm);
        free(h_sm);
        cudaFree(d_cm);
        cudaFree(d_sm);
    }

    /* the opt-in lossy transport on rows whose quantisation is exact: every
     * head row holds integers in [-127, 127] with 127 present (INT8: inv = 1,
     * scale = 1) or E4M3 grid values with 448 present (inv = 1, scale = 1),
     * so pack -> unpack and split -> merge must reproduce the bf16 bits */
    {
        uint16_t *h_x = malloc(n * 2), *h_y = malloc(n * 2);
        float *h_s = malloc(n / D * sizeof(float));
        CHECK(h_x && h_y && h_s);
        static const float grid[8] = {448.0f, -1.0f, 0.5f, 2.0f, -0.015625f, 0.0f, 96.0f, -320.0f};
        for (int fmt = 0; fmt < 2; ++fmt) {
            for (int64_t i = 0; i < n; ++i) {
                float v = fmt == 0 ? (float)((int)((i * 37) % 255) - 127) : grid[(i * 5) % 8];
                if (i % D == 0) v = fmt == 0 ? 127.0f : 448.0f;
                uint32_t u;
                memcpy(&u, &v, 4);
                h_x[i] = (uint16_t)(u >> 16);          /* exact: few significant bits */
            }
            void *d_codes = NULL, *d_scales = NULL;
            CHECK(cudaMalloc(&d_codes, n) == cudaSuccess);
            CHECK(cudaMalloc(&d_scales, n / D * sizeof(float)) == cudaSuccess);
            CHECK(cudaMemcpy(d_src, h_x, n * 2, cudaMemcpyHostToDevice) == cudaSuccess);
            CHECK(vf_scale_count(VF_OP_QKV_PACK, T, H, D, P, C) == n / D);
            if (fmt == 0) {
                CHECK(vf_qkv_pack_int8(d_src, st, T, H, D, P, C, d_codes, d_scales, NULL) == VF_OK);
                CHECK(vf_qkv_unpack_int8(d_codes, d_scales, T, H, D, P, C, d_q, d_k, d_v, NULL,
                                         NULL) == VF_OK);
            } else {
                /* the [T][3H][D] view of the same buffer as one attention output */
                const int64_t s3[3] = {3 * H * D, D, 1};
                CHECK(vf_attn_split_fp8(d_src, s3, T, 3 * H, D, P, C, d_codes, d_scales,
                                        NULL) == VF_OK);
                CHECK(vf_head_merge_fp8(d_codes, d_scales, NULL, T, 3 * H, D, P, C, d_packed,
                                        NULL) == VF_OK);
            }
            CHECK(cudaDeviceSynchronize() == cudaSuccess);
            CHECK(cudaMemcpy(h_s, d_scales, n / D * sizeof(float), cudaMemcpyDeviceToHost) ==
                  cudaSuccess);
            for (int64_t r = 0; r < n / D; ++r) CHECK(h_s[r] == 1.0f);
            if (fmt == 0) {
                for (int s = 0; s < 3; ++s) {
                    void *d = s == 0 ? d_q : s == 1 ? d_k : d_v;
                    CHECK(cudaMemcpy(h_y, d, n * 2 / 3, cudaMemcpyDeviceToHost) == cudaSuccess);
                    for (int64_t t = 0; t < T; ++t)
                        for (int64_t x = 0; x < H * D; ++x)
                            CHECK(h_y[t * H * D + x] == h_x[t * 3 * H * D + s * H * D + x]);
                }
            } else {
                CHECK(cudaMemcpy(h_y, d_packed, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
                CHECK(memcmp(h_y, h_x, n * 2) == 0);
                /* a head row holding a NaN and one holding an infinity are lost rows:
                 * each gets the float32 quiet NaN as its scale, and every element of
                 * theirs arrives as the bfloat16 quiet NaN; no other row changes */
                const int64_t rows = n / D, r1 = 5, r2 = rows - 3;   /* [T][3H][D] rows */
                h_x[r1 * D + 7] = 0x7FC1;
                h_x[r2 * D] = 0xFF80;
                CHECK(cudaMemcpy(d_src, h_x, n * 2, cudaMemcpyHostToDevice) == cudaSuccess);
                const int64_t s3[3] = {3 * H * D, D, 1};
                CHECK(vf_attn_split_fp8(d_src, s3, T, 3 * H, D, P, C, d_codes, d_scales,
                                        NULL) == VF_OK);
                CHECK(vf_head_merge_fp8(d_codes, d_scales, NULL, T, 3 * H, D, P, C, d_packed,
                                        NULL) == VF_OK);
                CHECK(cudaDeviceSynchronize() == cudaSuccess);
                CHECK(cudaMemcpy(h_s, d_scales, rows * sizeof(float), cudaMemcpyDeviceToHost) ==
                      cudaSuccess);
                int lost = 0;
                for (int64_t r = 0; r < rows; ++r) {
                    uint32_t b;
                    memcpy(&b, &h_s[r], 4);
                    lost += b == 0x7FC00000u;
                }
                CHECK(lost == 2);
                CHECK(cudaMemcpy(h_y, d_packed, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
                for (int64_t r = 0; r < rows; ++r)
                    for (int64_t d = 0; d < D; ++d)
                        CHECK(h_y[r * D + d] == ((r == r1 || r == r2) ? 0x7FC0 : h_x[r * D + d]));
            }
            cudaFree(d_codes);
            cudaFree(d_scales);
        }
        free(h_x);
        free(h_y);
        free(h_s);
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
