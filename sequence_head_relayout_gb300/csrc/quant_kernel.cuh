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
// A head row holding a NaN or an infinity is a lost row: scale = the float32
// quiet NaN 0x7FC00000 and every code 0 (its largest 15-bit magnitude is
// 0x7F80 or more, so the amax reduction finds it for free); a row whose scale
// is not finite is dequantised to the bfloat16 quiet NaN 0x7FC0 throughout.
// Every step is a single IEEE operation with an explicit rounding mode
// (__fdiv_rn, __fmul_rn and its packed form mul.rn.f32x2, __float2int_rn, the
// cvt.rn.satfinite conversions), so the integer decisions are the same on any
// correctly rounding machine.
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
// rows' loads in flight when quantising (kQuantRowsShort on the 8-element
// path when a lane holds at most 2 vectors of a row; kDequantRows when
// dequantising).
// Blocks are kQuantThreads (kDequantThreads) threads, whole warps, so every
// shuffle runs with all 32 lanes present.
//
// The kernels are bound by instruction issue before HBM unless every
// per-element step is a single cheap instruction, so the 8-element path
// (quantise_rows8 / dequantise_rows8) uses exact integer tricks in place of
// conversion instructions, each equal to the plain float32 step:
//   * round half to even to an integer: fl(q + 1.5 * 2^23) for |q| < 2^22 is
//     1.5 * 2^23 + rint(q) (the sum's unit in the last place is 1 and the
//     addition itself rounds to nearest even; 1.5 * 2^23 is even), and its
//     low byte is rint(q) as a two's-complement byte.  No clamp is needed:
//     |x| <= amax gives |q| <= 127 (1 + 2^-24)^2 < 127.5, so rint(q) is within
//     +-127 (a clamp there would never act);
//   * int8 code to float: the float with bits 0x4B000000 | (c ^ 0x80) is
//     2^23 + c + 128 exactly; subtracting 2^23 + 128 gives c exactly;
//   * magnitudes: max over |x| in the integer order of the 15 magnitude bits,
//     two at a time with the 16-bit-lane max of sm_90+;
//   * the row index (token, head) of a group: n / heads by a multiply-high
//     and a shift (the round-up method of Granlund and Montgomery, "Division
//     by invariant integers using multiplication", 1994), exact for
//     n < 2^31;
//   * inv = top / amax and scale = amax / top without a division per row:
//     a live amax is a normal bfloat16, M * 2^k with M = 1 + j/128 (j = its 7
//     stored mantissa bits), and scaling by a power of two commutes with
//     float32 rounding while the result stays normal, so
//     fl(top / amax) = fl(top / M) * 2^-k and fl(amax / top) = fl(M / top) * 2^k
//     exactly.  Each block computes the 128 values fl(top / M) and fl(M / top)
//     with the correctly rounded division into shared memory once; a row then
//     takes two table reads and two additions to the exponent field.  For
//     amax in [2^-96, 2^128) both results stay normal (inv within
//     [2^-121, 2^105], scale within [2^-105, 2^121]).  Unlike a division per
//     row, the cost does not depend on the data: with a correctly rounded
//     division per row, rows whose amax is 2^126 or more (1/amax subnormal)
//     took a slower path, and a payload with 40% such rows made the ragged
//     split 7% slower.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace vf {

#ifndef VF_QUANT_ROWS
#define VF_QUANT_ROWS 2
#endif
#ifndef VF_QUANT_ROWS_SHORT
#define VF_QUANT_ROWS_SHORT 4
#endif
#ifndef VF_DEQUANT_ROWS
#define VF_DEQUANT_ROWS 1
#endif
#ifndef VF_QUANT_THREADS
#define VF_QUANT_THREADS 128
#endif
#ifndef VF_DEQUANT_THREADS
#define VF_DEQUANT_THREADS 256
#endif

constexpr int kQuantThreads = VF_QUANT_THREADS;      // threads per block, quantising
constexpr int kDequantThreads = VF_DEQUANT_THREADS;  // threads per block, dequantising
constexpr int kQuantRows = VF_QUANT_ROWS;        // head rows per group in flight, quantising
constexpr int kQuantRowsShort = VF_QUANT_ROWS_SHORT;   // the same, 8-element path, <= 2 vectors
                                                       // per lane (short head rows)
constexpr int kDequantRows = VF_DEQUANT_ROWS;    // the same, dequantising
static_assert(kQuantThreads % 32 == 0 && kDequantThreads % 32 == 0,
              "blocks are whole warps");
#ifndef VF_QUANT_F32X2
#define VF_QUANT_F32X2 1
#endif
constexpr int kMantissas = 128;            // bfloat16 stored-mantissa patterns

// Head rows in flight per group on the 8-element quantising path with NV
// vectors per lane.
__host__ __device__ constexpr int quant_rows8(int NV) {
    return NV >= 4 ? kQuantRows : kQuantRowsShort;
}
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
    uint32_t div_mul;      // n / heads == (umulhi(n, div_mul) + n) >> div_shift, n < 2^31
    uint32_t div_shift;
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

constexpr uint32_t kLostScaleBits = 0x7FC00000u;   // scale of a lost row (float32 quiet NaN)
constexpr uint32_t kLostValue2 = 0x7FC07FC0u;      // two bfloat16 quiet NaNs

// A 15-bit bfloat16 magnitude of a NaN or an infinity.
__device__ __forceinline__ bool non_finite_magnitude(uint32_t m) { return m >= 0x7F80u; }

// A scale that is NaN or an infinity: its row is written as NaN.
__device__ __forceinline__ bool lost_scale(float s) {
    return (__float_as_uint(s) & 0x7FFFFFFFu) >= 0x7F800000u;
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
    const uint32_t t = (__umulhi(hr, a.div_mul) + hr) >> a.div_shift;   // hr / heads
    const uint32_t hh = hr - t * uint32_t(a.heads);
    return int64_t(t) * a.row_stride + int64_t(hh) * a.head_stride + e * a.d_stride;
}

// Per 16-bit lane maximum of two words (sm_90+).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Both 15-bit magnitudes of a word of two bfloat16 patterns, lane-wise.
__device__ __forceinline__ uint32_t mag2(uint32_t w) { return w & 0x7FFF7FFFu; }

// Low byte of the integer nearest to q (ties to even), for |q| < 2^22.
__device__ __forceinline__ uint32_t rint_bits(float q) {
    return __float_as_uint(__fadd_rn(q, 12582912.0f));
}

// Two float32 products, each rounded once to nearest even: the packed f32x2
// form of sm_100 and later issues both in one instruction.  Used only where a
// conversion, never an addition, consumes the products: measured on GB300,
// ptxas fuses a packed multiply and a packed add that follows it into one
// fused multiply-add even when both carry an explicit .rn, which rounds once
// where the format rounds twice (q = x * inv exactly 63.5 after its own
// rounding came out 63).  The INT8 encoder therefore keeps the scalar
// __fmul_rn / __fadd_rn, which are never contracted.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
#if VF_QUANT_F32X2
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
#else
    return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
#endif
}

// Eight bfloat16 patterns -> eight codes.
template <int FMT>
__device__ __forceinline__ uint2 encode8(const uint4 &w, float inv) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    const float2 inv2 = make_float2(inv, inv);
    uint32_t out[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float f[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t x = in[2 * k + j];
            // elements 2j (low half) and 2j + 1 (high half) of the pair
            const float lo = __uint_as_float(x << 16), hi = __uint_as_float(x & 0xFFFF0000u);
            if constexpr (FMT == kFmtInt8) {
                f[2 * j] = __fmul_rn(lo, inv);
                f[2 * j + 1] = __fmul_rn(hi, inv);
            } else {
                const float2 q = mul2_rn(make_float2(lo, hi), inv2);
                f[2 * j] = q.x;
                f[2 * j + 1] = q.y;
            }
        }
        if constexpr (FMT == kFmtInt8) {
            const uint32_t b01 = __byte_perm(rint_bits(f[0]), rint_bits(f[1]), 0x0040);
            const uint32_t b23 = __byte_perm(rint_bits(f[2]), rint_bits(f[3]), 0x0040);
            out[k] = __byte_perm(b01, b23, 0x5410);
        } else {
            const uint32_t p01 = __nv_cvt_float2_to_fp8x2(make_float2(f[0], f[1]),
                                                          __NV_SATFINITE, __NV_E4M3);
            const uint32_t p23 = __nv_cvt_float2_to_fp8x2(make_float2(f[2], f[3]),
                                                          __NV_SATFINITE, __NV_E4M3);
            out[k] = __byte_perm(p01, p23, 0x5410);
        }
    }
    return make_uint2(out[0], out[1]);
}

// Four codes (one word) times the scale -> four bfloat16 patterns (two words).
template <int FMT>
__device__ __forceinline__ uint2 decode4(uint32_t c, float s) {
    float f[4];
    if constexpr (FMT == kFmtInt8) {
        const uint32_t u = c ^ 0x80808080u;                  // c + 128, per byte
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u | i)),
                             8388736.0f);                    // 2^23 + 128
    } else {
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(c & 0xFFFFu),
                                                          __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(c >> 16),
                                                          __NV_E4M3);
        const float2 a = __half22float2(__half2(lo));       // exact: E4M3 fits in half
        const float2 b = __half22float2(__half2(hi));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
    const float2 s2 = make_float2(s, s);
    const float2 p01 = mul2_rn(make_float2(f[0], f[1]), s2);
    const float2 p23 = mul2_rn(make_float2(f[2], f[3]), s2);
    const __nv_bfloat162 y01 = __floats2bfloat162_rn(p01.x, p01.y);
    const __nv_bfloat162 y23 = __floats2bfloat162_rn(p23.x, p23.y);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&y01),
                      *reinterpret_cast<const uint32_t *>(&y23));
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
            const bool lost = non_finite_magnitude(m[r]);
            const bool live = !lost && amax >= 0x1p-96f;
            const float inv = live ? __fdiv_rn(top, amax) : 0.0f;
            const int64_t prow = pc.first_row + hr;               // packed head row
            uint8_t *crow = a.codes + prow * a.D;
            if (lane == 0)
                a.scales[prow] = lost ? __uint_as_float(kLostScaleBits)
                                      : live ? __fdiv_rn(amax, top) : 0.0f;
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
__global__ void __launch_bounds__(kDequantThreads)
dequantise_rows(const __grid_constant__ QArgs a) {
    using B = typename QVec<VW>::B;
    using CV = typename QVec<VW>::C;
    wait_for_previous_grid();
    const QPiece &pc = a.pieces[blockIdx.y];
    const uint32_t G = 1u << a.lanes_log2;
    const uint32_t lane = threadIdx.x & (G - 1);
    const uint32_t groups = kDequantThreads >> a.lanes_log2;
    const uint32_t group = threadIdx.x >> a.lanes_log2;
    const uint32_t nrows = uint32_t(pc.rows) * uint32_t(a.heads);

    for (uint32_t base = blockIdx.x * groups * kDequantRows; base < nrows;
         base += gridDim.x * groups * kDequantRows) {
        CV cv[kDequantRows];
        float sc[kDequantRows];
        // one vector per lane per row on the fast path; loads first
        if (int(G) * 1 >= a.nvec) {
#pragma unroll
            for (int r = 0; r < kDequantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr < nrows && int(lane) < a.nvec) {
                    const int64_t prow = pc.first_row + hr;
                    cv[r] = *reinterpret_cast<const CV *>(a.codes + prow * a.D +
                                                          int64_t(lane) * VW);
                    sc[r] = a.scales[prow];
                }
            }
#pragma unroll
            for (int r = 0; r < kDequantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr >= nrows || int(lane) >= a.nvec) continue;
                uint8_t c[VW];
                memcpy(c, &cv[r], sizeof(c));
                const bool lost = lost_scale(sc[r]);
                uint16_t y[VW];
#pragma unroll
                for (int i = 0; i < VW; ++i)
                    y[i] = lost ? uint16_t(kLostValue2 & 0xFFFFu)
                                : __bfloat16_as_ushort(__float2bfloat16_rn(
                                      __fmul_rn(code_value<FMT>(c[i]), sc[r])));
                B out;
                memcpy(&out, y, sizeof(out));
                *reinterpret_cast<B *>(pc.strided + strided_offset(a, hr, int64_t(lane) * VW)) =
                    out;
            }
        } else {
            for (int r = 0; r < kDequantRows; ++r) {
                const uint32_t hr = base + group + uint32_t(r) * groups;
                if (hr >= nrows) continue;
                const int64_t prow = pc.first_row + hr;
                const float s = a.scales[prow];
                const bool lost = lost_scale(s);
                uint16_t *row = pc.strided + strided_offset(a, hr, 0);
                for (int v = int(lane); v < a.nvec; v += int(G)) {
                    const CV x = *reinterpret_cast<const CV *>(a.codes + prow * a.D +
                                                               int64_t(v) * VW);
                    uint8_t c[VW];
                    memcpy(c, &x, sizeof(c));
                    uint16_t y[VW];
#pragma unroll
                    for (int i = 0; i < VW; ++i)
                        y[i] = lost ? uint16_t(kLostValue2 & 0xFFFFu)
                                    : __bfloat16_as_ushort(__float2bfloat16_rn(
                                          __fmul_rn(code_value<FMT>(c[i]), s)));
                    B out;
                    memcpy(&out, y, sizeof(out));
                    *reinterpret_cast<B *>(row + int64_t(v) * VW * a.d_stride) = out;
                }
            }
        }
    }
}

// 8-element vectors (D % 8 == 0, d contiguous, aligned): NV vectors per
// lane, vector j of lane l at index l + j * G of the head row, so that each
// of a warp's loads covers consecutive 16-byte pieces.
template <int FMT, int NV>
__global__ void __launch_bounds__(kQuantThreads)
quantise_rows8(const __grid_constant__ QArgs a) {
    constexpr int kRows = quant_rows8(NV);
    // fl(top / M) and fl(M / top) for the 128 mantissas M = 1 + i/128, built
    // before the grid-dependency wait (it overlaps the previous grid's tail)
    const float top = top_code<FMT>();
    __shared__ float inv_of[kMantissas], scale_of[kMantissas];
    for (int i = int(threadIdx.x); i < kMantissas; i += kQuantThreads) {
        const float M = 1.0f + float(i) * (1.0f / 128.0f);      // exact
        inv_of[i] = __fdiv_rn(top, M);
        scale_of[i] = __fdiv_rn(M, top);
    }
    __syncthreads();
    wait_for_previous_grid();
    const QPiece &pc = a.pieces[blockIdx.y];
    const uint32_t G = 1u << a.lanes_log2;
    const uint32_t lane = threadIdx.x & (G - 1);
    const uint32_t groups = kQuantThreads >> a.lanes_log2;
    const uint32_t group = threadIdx.x >> a.lanes_log2;
    const uint32_t nrows = uint32_t(pc.rows) * uint32_t(a.heads);   // < 2^31, host-checked
    const uint32_t nvec = uint32_t(a.nvec);

    for (uint32_t base = blockIdx.x * groups * kRows; base < nrows;
         base += gridDim.x * groups * kRows) {
        uint4 w[kRows][NV];
        uint32_t m[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            const uint16_t *row = pc.strided + strided_offset(a, hr, 0);
            m[r] = 0;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint32_t v = lane + uint32_t(j) * G;
                w[r][j] = make_uint4(0, 0, 0, 0);
                if (hr < nrows && v < nvec)
                    w[r][j] = *reinterpret_cast<const uint4 *>(row + int64_t(v) * 8);
                m[r] = max_u16x2(m[r], max_u16x2(max_u16x2(mag2(w[r][j].x), mag2(w[r][j].y)),
                                                 max_u16x2(mag2(w[r][j].z), mag2(w[r][j].w))));
            }
        }
        // group-wide amax: all 32 lanes of every warp are here
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            for (uint32_t o = G >> 1; o > 0; o >>= 1)
                m[r] = max_u16x2(m[r], __shfl_xor_sync(0xFFFFFFFFu, m[r], int(o)));
            m[r] = max(m[r] & 0xFFFFu, m[r] >> 16);
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            if (hr >= nrows) continue;
            // m[r]: the row's largest magnitude as a bfloat16 pattern
            const bool lost = non_finite_magnitude(m[r]);
            const bool live = !lost && m[r] >= 0x0F80u;           // amax >= 2^-96 (31 << 7)
            // amax = M * 2^k: mantissa index mi, exponent k = e - 127 (both
            // used only for a live row, whose results stay normal)
            const uint32_t mi = m[r] & 0x7Fu;
            const uint32_t k23 = uint32_t((int32_t(m[r] >> 7) - 127) * (1 << 23));  // k << 23
            const float inv = live ? __uint_as_float(__float_as_uint(inv_of[mi]) - k23) : 0.0f;
            const float scale = __uint_as_float(__float_as_uint(scale_of[mi]) + k23);
            const int64_t prow = pc.first_row + hr;               // packed head row
            uint8_t *crow = a.codes + prow * a.D;
            if (lane == 0)
                a.scales[prow] = lost ? __uint_as_float(kLostScaleBits)
                                      : live ? scale : 0.0f;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint32_t v = lane + uint32_t(j) * G;
                if (v >= nvec) continue;
                uint2 c = encode8<FMT>(w[r][j], inv);
                if (!live) c = make_uint2(0, 0);
                *reinterpret_cast<uint2 *>(crow + int64_t(v) * 8) = c;
            }
        }
    }
}

template <int FMT, int NV>
__global__ void __launch_bounds__(kDequantThreads)
dequantise_rows8(const __grid_constant__ QArgs a) {
    wait_for_previous_grid();
    const QPiece &pc = a.pieces[blockIdx.y];
    const uint32_t G = 1u << a.lanes_log2;
    const uint32_t lane = threadIdx.x & (G - 1);
    const uint32_t groups = kDequantThreads >> a.lanes_log2;
    const uint32_t group = threadIdx.x >> a.lanes_log2;
    const uint32_t nrows = uint32_t(pc.rows) * uint32_t(a.heads);
    const uint32_t nvec = uint32_t(a.nvec);

    for (uint32_t base = blockIdx.x * groups * kDequantRows; base < nrows;
         base += gridDim.x * groups * kDequantRows) {
        uint2 c[kDequantRows][NV];
        float sc[kDequantRows];
#pragma unroll
        for (int r = 0; r < kDequantRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            const int64_t prow = pc.first_row + hr;
            sc[r] = hr < nrows ? a.scales[prow] : 0.0f;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint32_t v = lane + uint32_t(j) * G;
                c[r][j] = make_uint2(0, 0);
                if (hr < nrows && v < nvec)
                    c[r][j] = *reinterpret_cast<const uint2 *>(a.codes + prow * a.D +
                                                               int64_t(v) * 8);
            }
        }
#pragma unroll
        for (int r = 0; r < kDequantRows; ++r) {
            const uint32_t hr = base + group + uint32_t(r) * groups;
            if (hr >= nrows) continue;
            uint16_t *row = pc.strided + strided_offset(a, hr, 0);
            if (lost_scale(sc[r])) {                          // rare: a lost row
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const uint32_t v = lane + uint32_t(j) * G;
                    if (v < nvec)
                        *reinterpret_cast<uint4 *>(row + int64_t(v) * 8) =
                            make_uint4(kLostValue2, kLostValue2, kLostValue2, kLostValue2);
                }
                continue;
            }
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint32_t v = lane + uint32_t(j) * G;
                if (v >= nvec) continue;
                const uint2 lo = decode4<FMT>(c[r][j].x, sc[r]);
                const uint2 hi = decode4<FMT>(c[r][j].y, sc[r]);
                *reinterpret_cast<uint4 *>(row + int64_t(v) * 8) =
                    make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
        }
    }
}

}  // namespace vf
