// Shared-memory staged relayout for short head rows on a head-major strided
// side.
//
// The row-block kernel (relayout_kernel.cuh) moves whole D-element head rows,
// which keeps both sides sector-complete while a head row is at least one
// 32-byte DRAM sector.  Below that (D = 8: 16-byte head rows) and with a
// strided side whose consecutive tokens of one head are closer together than
// consecutive heads of one token (an attention buffer [H][T][D] viewed as
// [T][H][D]), the (token, head) interchange does break coalescing: a warp's
// 16-byte pieces land in as many different sectors.  Measured on GB300 with the
// row-block kernel (split, 64 Mi elements, clean L2): 4.68 TB/s at D = 8 and
// 6.24 TB/s at D = 16 against 7.28 TB/s for a token-major source.
//
// Here a block stages a tile of 64 / DV tokens x kTileHeads heads in shared
// memory: the strided side is read (or written) head by head, each head's
// tokens one contiguous run, and the packed side token by token, each token's
// heads one contiguous run; every global access is a 16-byte vector and
// consecutive threads touch consecutive vectors on both sides.  The tile is
// stored in packed order with one head row of padding per token, so that the
// strided-order accesses (eight 16-byte vectors per shared-memory phase, one
// or two per token) fall on distinct banks.
#pragma once

#include <cstdint>

#include "relayout_kernel.cuh"

namespace vf {

constexpr int kTileThreads = 256;
constexpr int kTileHeads = 32;

// DV = 16-byte vectors per head row (D = 8 * DV); a tile holds 64 / DV
// tokens, so every thread moves 8 vectors per tile.
template <int DV> struct TileShape {
    static constexpr int kTok = 64 / DV;
    static constexpr int kVecs = kTok * kTileHeads * DV;          // 2048
    static constexpr int kPitch = kTileHeads * DV + DV;            // vectors per token row
    static constexpr int kPerThread = kVecs / kTileThreads;        // 8
};

struct TiledArgs {
    uint16_t *packed;
    int64_t row_stride;    // strided side, between tokens (elements)
    int64_t head_stride;   // strided side, between heads (elements)
    int32_t heads;         // heads per packed row
    int32_t head_tiles;    // ceil(heads / kTileHeads)
    Piece pieces[kMaxPieces];
};

// Grid: x = token tiles, y = piece, z = head tiles.  Block: kTileThreads.
template <int DV, bool kPackedIsDst>
__global__ void __launch_bounds__(kTileThreads)
relayout_tiled(const __grid_constant__ TiledArgs a) {
    using S = TileShape<DV>;
    __shared__ uint4 tile[S::kTok * S::kPitch];
#if VF_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    const Piece &pc = a.pieces[blockIdx.y];
    const int rows = int(pc.rows);
    const int t0 = int(blockIdx.x) * S::kTok;
    const int h0 = int(blockIdx.z) * kTileHeads;
    if (t0 >= rows) return;                                   // block-uniform
    const int nt = min(S::kTok, rows - t0);
    const int nh = min(kTileHeads, a.heads - h0);
    constexpr int D = 8 * DV;
    const int64_t R = int64_t(a.heads) * D;                   // packed row length
    uint16_t *const packed0 = a.packed + pc.packed_off + int64_t(t0) * R + int64_t(h0) * D;
    uint16_t *const strided0 = pc.strided + int64_t(t0) * a.row_stride +
                               int64_t(h0) * a.head_stride;

    // strided order: v -> (head h, token tk, vector dv), tokens fastest
    // packed order:  v -> (token tk, head h, vector dv), heads fastest
    uint4 v[S::kPerThread];
    if (kPackedIsDst) {
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int h = e / (S::kTok * DV);
            const int r = e - h * (S::kTok * DV);
            const int tk = r / DV, dv = r - tk * DV;
            if (h < nh && tk < nt)
                v[i] = *reinterpret_cast<const uint4 *>(
                    strided0 + int64_t(tk) * a.row_stride + int64_t(h) * a.head_stride + dv * 8);
        }
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int h = e / (S::kTok * DV);
            const int r = e - h * (S::kTok * DV);
            const int tk = r / DV, dv = r - tk * DV;
            if (h < nh && tk < nt) tile[tk * S::kPitch + h * DV + dv] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int tk = e / (kTileHeads * DV);
            const int r = e - tk * (kTileHeads * DV);
            const int h = r / DV, dv = r - h * DV;
            if (h < nh && tk < nt)
                *reinterpret_cast<uint4 *>(packed0 + int64_t(tk) * R + h * D + dv * 8) =
                    tile[tk * S::kPitch + h * DV + dv];
        }
    } else {
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int tk = e / (kTileHeads * DV);
            const int r = e - tk * (kTileHeads * DV);
            const int h = r / DV, dv = r - h * DV;
            if (h < nh && tk < nt)
                v[i] = *reinterpret_cast<const uint4 *>(packed0 + int64_t(tk) * R + h * D +
                                                        dv * 8);
        }
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int tk = e / (kTileHeads * DV);
            const int r = e - tk * (kTileHeads * DV);
            const int h = r / DV, dv = r - h * DV;
            if (h < nh && tk < nt) tile[tk * S::kPitch + h * DV + dv] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < S::kPerThread; ++i) {
            const int e = int(threadIdx.x) + i * kTileThreads;
            const int h = e / (S::kTok * DV);
            const int r = e - h * (S::kTok * DV);
            const int tk = r / DV, dv = r - tk * DV;
            if (h < nh && tk < nt)
                *reinterpret_cast<uint4 *>(strided0 + int64_t(tk) * a.row_stride +
                                           int64_t(h) * a.head_stride + dv * 8) =
                    tile[tk * S::kPitch + h * DV + dv];
        }
    }
}

}  // namespace vf
