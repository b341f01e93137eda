// Device side of the opt-in lossy transport: the same relayouts as
// relayout_kernel.cuh, quantising each head row to 8-bit codes on the way
// into packed storage (pack, split) or dequantising on the way out (merge,
// unpack).
//
// "Sol-Engine alignment on SM86 and SM89", table "Upstream gap and
// disposition", row "INT8 QKV and FP8 output transport", names the variant
// (INT8 Q/K/V and FP8 attention output across the exchange) and keeps it out
// of the exact default; it gives no format.  The format read here: per head
// row (the D elements of one token and one head) amax = max |x|; a row with
// amax < 2^-96 is sent as scale 0 and all codes 0; otherwise, with top = 127
// (INT8) or 448 (E4M3), inv = top / amax and scale = amax / top (each one
// correctly rounded division), q = x * inv (one rounding), code =
// clamp(round_half_even(q), +-127) for INT8 or the nearest E4M3 value (ties
// to even, saturating at +-448).  Dequantisation: bf16(value(code) * scale),
// the product rounded to float32 and then to bfloat16, both to nearest even.
// Every step is a single IEEE operation with an explicit rounding mode
// (__fdiv_rn, __fmul_rn, __float2int_rn, the cvt.rn.satfinite conversions),
// so the integer decisions are the same on any correctly rounding machine.
//
// Storage: codes use the element layout of the exact ops, one byte per
// element; scales are one float per head row, indexed by the row's position
// in that layout (element offset / D).
//
// Work split: a group of G lanes (G a power of two, at most 32, aligned
// within the warp) owns one head row at a time; lane l holds VW consecutive
// elements.  amax is reduced within the group with xor shuffles on the
// 15-bit magnitudes of the bfloat16 patterns (for non-NaN values the order of
// |x| is the integer order of those bits).  Each group keeps kQuantRows head
// rows' loads in flight.  Blocks are kQuantThreads threads, whole warps, so
// every shuffle runs with all 32 lanes present.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace vf {

#ifndef VF_QUANT_ROWS
#define VF_QUANT_ROWS 2
#endif

constexpr int kQuantThreads = 256;         // threads per block (8 full warps)
constexpr int kQuantRows = VF_QUANT_ROWS;  // head rows per group in flight
constexpr int kMaxQPieces = 128;           // pieces per launch (parameter space)

constexpr int kFmtInt8 = 1;
constexpr int kFmtE4M3 = 2;

struct QPiece {
    int64_t first_row;     // head-row index of the block's first row in packed storage
    uint16_t *strided;     // the block's first token row on the strided side
    int64_t rows;          // tokens in the block
};

struct QArgs {
    uint8_t *codes;        // packed storage, one byte per element
    float *scales;         // one float per packed head row
    int64_t row_stride;    // strided side, between tokens
    int64_t head_stride;   // strided side, between heads
    int64_t d_stride;      // strided side, along d (1 on every vector path)
    int32_t heads;         // heads per packed token row
    int32_t D;             // elements per head row
    int32_t lanes_log2;    // group size G = 1 << lanes_log2
    int32_t nvec;          // ceil(D / VW) vectors per head row
    QPiece pieces[kMaxQPieces];
};

template <int VW> struct QVec;
template <> struct QVec<8> { using B = uint4; using C = uint2; };
template <> struct QVec<4> { using B = uint2; using C = unsigned int; };
template <> struct QVec<2> { using B = unsigned int; using C = unsigned short; };
template <> struct QVec<1> { using B = unsigned short; using C = unsigned char; };

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) {
    return __uint_as_float(h << 16);
}

template <int FMT>
__device__ __forceinline__ float top_code() {
    return FMT == kFmtE4M3 ? 448.0f : 127.0f;
}

// Quantise VW values (bfloat16 patterns h) with the row's inv into codes c.
template <int VW, int FMT>
__device__ __forceinline__ void encode(const uint16_t (&h)[VW], float inv, bool live,
                                       uint8_t (&c)[VW]) {
    if constexpr (FMT == kFmtInt8) {
#pragma unroll
        for (int i = 0; i < VW; ++i) {
            const float q = __fmul_rn(bf16_bits_to_float(h[i]), inv);
            const int r = min(127, max(-127, __float2int_rn(q)));
            c[i] = live ? uint8_t(int8_t(r)) : uint8_t(0);
        }
    } else if constexpr (VW == 1) {
        const float q = __fmul_rn(bf16_bits_to_float(h[0]), inv);
        c[0] = live ? uint8_t(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3)) : uint8_t(0);
    } else {
#pragma unroll
        for (int i = 0; i < VW; i += 2) {
            const float2 q = make_float2(__fmul_rn(bf16_bits_to_float(h[i]), inv),
                                         __fmul_rn(bf16_bits_to_float(h[i + 1]), inv));
            const uint16_t pair = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
            c[i] = live ? uint8_t(pair & 0xFF) : uint8_t(0);       // first element, low byte
            c[i + 1] = live ? uint8_t(pair >> 8) : uint8_t(0);
        }
    }
}

template <int FMT>
__device__ __forceinline__ float code_value(uint8_t c) {
    if constexpr (FMT == kFmtInt8) {
        return float(int8_t(c));
    } else {
        // every E4M3 value is exact in half precision
        const __half_raw hr = __nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(c), __NV_E4M3);
        return __half2float(__half(hr));
    }
}

template <int VW>
__device__ __forceinline__ uint32_t magnitude_max(const uint16_t (&h)[VW]) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < VW; ++i) m = max(m, uint32_t(h[i]) & 0x7FFFu);
    return m;
}

// Position of head row hr of a piece: (token, head) -> strided element offset.
__device__ __forceinline__ int64_t strided_offset(const QArgs &a, uint32_t hr, int64_t e) {
    const uint32_t heads = uint32_t(a.heads);
    const uint32_t t = hr / heads;
    const uint32_t hh = hr - t * heads;
    return int64_t(t) * a.row_stride + int64_t(hh) * a.head_stride + e * a.d_stride;
}

__device__ __forceinline__ void wait_for_previous_grid() {
    // Programmatic dependent launch, as in the exact kernel: the next grid may
    // start launching; this one waits (in hardware) for the previous grid.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Pack or split with quantisation.  Grid: x = blocks of head-row groups
// (grid-stride), y = piece.  kOne: every lane holds at most one vector of a
// head row (nvec <= G), kept in registers between the reduction and the
// encode; otherwise G = 32 and each lane walks the row twice.
template <int VW, int FMT, bool kOne>
__global__ void __launch_bounds__(kQuantThreads)
quantise_rows(const __grid_constant__ QArgs a) {
    using B = typename QVec<VW>::B;
    using CV = typename QVec<VW>::C;
    wait_for_previous_grid();
    const QPiece &pc = a.pieces[blockIdx.y];
    const uint32_t G = 1u << a.lanes_log2;
    const uint32_t lane = threadIdx.x & (G - 1);
    const uint32_t groups = kQuantThreads >> a.lanes_log2;
    const uint32_t group = threadIdx.x >> a.lanes_log2;
    const uint32_t nrows = uint32_t(pc.rows) * uint32_t(a.heads);   // < 2^31, host-checked
    const float top = top_code<FMT>();

    for (uint32_t base = blockIdx.x * groups * kQuantRows; base < nrows;
         base += gridDim.x * groups * kQuantRows) {
        uint16_t h[kQuantRows][VW];
        uint32_t m[kQuantRows];
#pragma unroll
        for (int r = 0; r < kQuantRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            m[r] = 0;
            if (kOne) {
                const bool ok = hr < nrows && int(lane) < a.nvec;
                B v{};
                if (ok) v = *reinterpret_cast<const B *>(
                            pc.strided + strided_offset(a, hr, int64_t(lane) * VW));
                memcpy(h[r], &v, sizeof(v));
                m[r] = magnitude_max<VW>(h[r]);
            } else if (hr < nrows) {
                const uint16_t *row = pc.strided + strided_offset(a, hr, 0);
                for (int v = int(lane); v < a.nvec; v += int(G)) {
                    const B x = *reinterpret_cast<const B *>(row + int64_t(v) * VW * a.d_stride);
                    uint16_t t[VW];
                    memcpy(t, &x, sizeof(x));
                    m[r] = max(m[r], magnitude_max<VW>(t));
                }
            }
        }
        // group-wide amax: all 32 lanes of every warp are here
#pragma unroll
        for (int r = 0; r < kQuantRows; ++r)
            for (uint32_t o = G >> 1; o > 0; o >>= 1)
                m[r] = max(m[r], __shfl_xor_sync(0xFFFFFFFFu, m[r], int(o)));
#pragma unroll
        for (int r = 0; r < kQuantRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            if (hr >= nrows) continue;
            const float amax = bf16_bits_to_float(m[r]);
            const bool live = amax >= 0x1p-96f;
            const float inv = live ? __fdiv_rn(top, amax) : 0.0f;
            const int64_t prow = pc.first_row + hr;               // packed head row
            uint8_t *crow = a.codes + prow * a.D;
            if (lane == 0) a.scales[prow] = live ? __fdiv_rn(amax, top) : 0.0f;
            if (kOne) {
                if (int(lane) >= a.nvec) continue;
                uint8_t c[VW];
                encode<VW, FMT>(h[r], inv, live, c);
                CV out;
                memcpy(&out, c, sizeof(out));
                *reinterpret_cast<CV *>(crow + int64_t(lane) * VW) = out;
            } else {
                const uint16_t *row = pc.strided + strided_offset(a, hr, 0);
                for (int v = int(lane); v < a.nvec; v += int(G)) {
                    const B x = *reinterpret_cast<const B *>(row + int64_t(v) * VW * a.d_stride);
                    uint16_t t[VW];
                    memcpy(t, &x, sizeof(x));
                    uint8_t c[VW];
                    encode<VW, FMT>(t, inv, live, c);
                    CV out;
                    memcpy(&out, c, sizeof(out));
                    *reinterpret_cast<CV *>(crow + int64_t(v) * VW) = out;
                }
            }
        }
    }
}

// Merge or unpack with dequantisation.  Same grid and groups; no reduction.
template <int VW, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
dequantise_rows(const __grid_constant__ QArgs a) {
    using B = typename QVec<VW>::B;
    using CV = typename QVec<VW>::C;
    wait_for_previous_grid();
    const QPiece &pc = a.pieces[blockIdx.y];
    const uint32_t G = 1u << a.lanes_log2;
    const uint32_t lane = threadIdx.x & (G - 1);
    const uint32_t groups = kQuantThreads >> a.lanes_log2;
    const uint32_t group = threadIdx.x >> a.lanes_log2;
    const uint32_t nrows = uint32_t(pc.rows) * uint32_t(a.heads);

    for (uint32_t base = blockIdx.x * groups * kQuantRows; base < nrows;
         base += gridDim.x * groups * kQuantRows) {
        CV cv[kQuantRows];
        float sc[kQuantRows];
        // one vector per lane per row on the fast path; loads first
        if (int(G) * 1 >= a.nvec) {
#pragma unroll
            for (int r = 0; r < kQuantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr < nrows && int(lane) < a.nvec) {
                    const int64_t prow = pc.first_row + hr;
                    cv[r] = *reinterpret_cast<const CV *>(a.codes + prow * a.D +
                                                          int64_t(lane) * VW);
                    sc[r] = a.scales[prow];
                }
            }
#pragma unroll
            for (int r = 0; r < kQuantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr >= nrows || int(lane) >= a.nvec) continue;
                uint8_t c[VW];
                memcpy(c, &cv[r], sizeof(c));
                uint16_t y[VW];
#pragma unroll
                for (int i = 0; i < VW; ++i)
                    y[i] = __bfloat16_as_ushort(
                        __float2bfloat16_rn(__fmul_rn(code_value<FMT>(c[i]), sc[r])));
                B out;
                memcpy(&out, y, sizeof(out));
                *reinterpret_cast<B *>(pc.strided + strided_offset(a, hr, int64_t(lane) * VW)) =
                    out;
            }
        } else {
            for (int r = 0; r < kQuantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr >= nrows) continue;
                const int64_t prow = pc.first_row + hr;
                const float s = a.scales[prow];
                uint16_t *row = pc.strided + strided_offset(a, hr, 0);
                for (int v = int(lane); v < a.nvec; v += int(G)) {
                    const CV x = *reinterpret_cast<const CV *>(a.codes + prow * a.D +
                                                               int64_t(v) * VW);
                    uint8_t c[VW];
                    memcpy(c, &x, sizeof(c));
                    uint16_t y[VW];
#pragma unroll
                    for (int i = 0; i < VW; ++i)
                        y[i] = __bfloat16_as_ushort(
                            __float2bfloat16_rn(__fmul_rn(code_value<FMT>(c[i]), s)));
                    B out;
                    memcpy(&out, y, sizeof(out));
                    *reinterpret_cast<B *>(row + int64_t(v) * VW * a.d_stride) = out;
                }
            }
        }
    }
}

}  // namespace vf
