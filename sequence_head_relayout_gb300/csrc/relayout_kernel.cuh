// Device side of the relayouts: one row-block copy kernel for every op.
//
// All the operations ("Sol-Engine alignment on SM86 and SM89", section
// "What is enabled": QKV destination pack, attention result split,
// returned-head merge; "速度、显存与质量", section "剖析单次去噪请求": the
// receive-side QKV unpack) move whole token rows between a contiguous
// *packed* side (the exchange buffer, destination-major) and a *strided*
// side (the caller's tensor views).  The host cuts the work into pieces; a
// piece is one (chunk, destination[, q/k/v slab]) block of the packed storage:
//
//   packed  : rows x (heads x D) contiguous elements starting at packed_off;
//   strided : element (row, head, d) at strided
//             + row * row_stride + head * head_stride + d * d_stride.
//
// There is no element-level transpose: the (token, head) interchange between
// the two sides happens at the granularity of whole D-element head rows (256 B
// at D = 128; at least one 32-byte DRAM sector from D = 16 up), so both sides
// stay sector-complete with plain 16-byte loads and stores and no
// shared-memory staging.  (Shorter head rows on a head-major strided side go
// through the shared-memory tile of tiled_kernel.cuh instead.)  The block is a
// 3-D thread array (x: VW-element vector within a head row, y: head, z: row)
// so the address of
// a thread is a sum of products (the only divisions are block-uniform), and a
// warp covers consecutive packed vectors.  Each thread keeps kRowsPerThread
// independent loads in flight before it stores.  Offsets are 64-bit
// throughout; a source view whose span crosses 2^31 elements is addressed
// correctly (the FP8 section of "速度、显存与质量" notes the same
// widen-before-multiplying rule for views past 2^31 elements).
#pragma once

#include <cstdint>

namespace vf {

// Launch-shape constants; the defaults were chosen by measurement on GB300 and
// can be overridden at compile time for tuning sweeps.
#ifndef VF_ROWS_PER_THREAD
#define VF_ROWS_PER_THREAD 2
#endif
#ifndef VF_CACHE_HINT
#define VF_CACHE_HINT 2
#endif
#ifndef VF_PDL
#define VF_PDL 1
#endif


constexpr int kMaxPieces = 128;                    // pieces per launch (parameter space)
constexpr int kRowsPerThread = VF_ROWS_PER_THREAD; // independent loads in flight per thread
constexpr int kMaxThreads = 512;                   // threads per block, upper bound

struct Piece {
    int64_t packed_off;    // element offset of the block in packed storage
    uint16_t *strided;     // the block's first row on the strided side
    int64_t rows;          // tokens in the block
};

// Read-only sides are passed through the same (non-const) pointer fields;
// the kernel only loads from the side it reads.
struct Args {
    uint16_t *packed;      // packed storage
    int64_t row_stride;    // strided side, between consecutive rows (tokens)
    int64_t head_stride;   // strided side, between heads of one row
    int64_t d_stride;      // strided side, along d (1 on every vector path)
    int32_t heads;         // heads per packed row
    int32_t D;             // elements per head row
    int32_t dchunks;       // ceil(D / VW / blockDim.x)
    int32_t z_base;        // first folded z index of this launch (head, d chunks)
    int32_t piece_fastest; // grid x walks pieces and y row groups (else the reverse)
    Piece pieces[kMaxPieces];
};

template <int VW> struct Vec;
template <> struct Vec<8> { using T = uint4; };
template <> struct Vec<4> { using T = uint2; };
template <> struct Vec<2> { using T = unsigned int; };
template <> struct Vec<1> { using T = unsigned short; };

// Every element is touched exactly once.  Hint 0: streaming loads and
// stores (evict-first, `.cs`); 1: read-only path loads (`.nc`), plain stores;
// 2: plain loads and stores.  Measured on GB300 over the pages', ragged and
// large workloads, 2 is fastest (by about 1%: the streaming hints cost a
// little and buy nothing when no byte is reused; an L2 256-byte prefetch hint
// on the loads was no faster either).
template <typename V>
__device__ __forceinline__ V load_once(const uint16_t *p) {
#if VF_CACHE_HINT == 0
    return __ldcs(reinterpret_cast<const V *>(p));
#elif VF_CACHE_HINT == 1
    return __ldg(reinterpret_cast<const V *>(p));
#else
    return *reinterpret_cast<const V *>(p);
#endif
}

template <typename V>
__device__ __forceinline__ void store_once(uint16_t *p, const V &v) {
#if VF_CACHE_HINT == 0
    __stcs(reinterpret_cast<V *>(p), v);
#else
    *reinterpret_cast<V *>(p) = v;
#endif
}

// Grid: x = groups of kRowsPerThread * blockDim.z rows, y = piece (or the
// two swapped when piece_fastest is set), z = (head chunk, d chunk) folded,
// offset by z_base.  Block: x = vector
// within a head row, y = head, z = row.  A thread copies one vector of each of
// its kRowsPerThread rows: all loads first, then all stores.
template <int VW, bool kPackedIsDst>
__global__ void __launch_bounds__(kMaxThreads)
relayout_rows(const __grid_constant__ Args a) {
    using V = typename Vec<VW>::T;
#if VF_PDL
    // Programmatic dependent launch (the host sets the launch attribute): let
    // the next kernel in the stream begin launching now, then wait -- in
    // hardware, not a spin -- until the previous grid in the stream has
    // completed and its writes are visible, before touching any memory.  The
    // order of work in the stream is unchanged; only the launch gap between
    // back-to-back relayouts (e.g. one call per overlap chunk) is hidden:
    // measured 8.5% on four chunk calls of the split at the pages' shape.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    const Piece &pc = a.pieces[a.piece_fastest ? blockIdx.x : blockIdx.y];
    const int group = int(a.piece_fastest ? blockIdx.y : blockIdx.x);
    const int rows = int(pc.rows);
    const int rstep = int(blockDim.z);
    const int row0 = group * (kRowsPerThread * rstep) + int(threadIdx.z);
    const int z = int(blockIdx.z) + a.z_base;
    const int hc = z / a.dchunks;                          // block-uniform
    const int hh = hc * int(blockDim.y) + int(threadIdx.y);
    const int dx = (z - hc * a.dchunks) * int(blockDim.x) + int(threadIdx.x);
    if (row0 >= rows || hh >= a.heads || dx * VW >= a.D) return;

    const int64_t R = int64_t(a.heads) * a.D;              // packed row length
    const int64_t po = pc.packed_off + int64_t(row0) * R + int64_t(hh) * a.D
                     + int64_t(dx) * VW;
    const int64_t so = int64_t(row0) * a.row_stride + int64_t(hh) * a.head_stride
                     + int64_t(dx) * VW * a.d_stride;
    const uint16_t *s = kPackedIsDst ? pc.strided + so : a.packed + po;
    uint16_t *d = kPackedIsDst ? a.packed + po : pc.strided + so;
    const int64_t s_step = int64_t(rstep) * (kPackedIsDst ? a.row_stride : R);
    const int64_t d_step = int64_t(rstep) * (kPackedIsDst ? R : a.row_stride);

    V v[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
        if (row0 + r * rstep < rows) v[r] = load_once<V>(s + r * s_step);
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
        if (row0 + r * rstep < rows) store_once<V>(d + r * d_step, v[r]);
}

}  // namespace vf
