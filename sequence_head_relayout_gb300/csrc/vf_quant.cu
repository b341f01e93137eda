// Launch policy of the lossy-transport kernels (quant_kernel.cuh): vector
// width, head-row group size, grid and the launches.  The host checks and the
// piece tables live in vf_relayout.cu; this file decides what the GPU
// executes for the quantising and dequantising relayouts.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>

#include "quant.h"
#include "vf_relayout.h"

namespace vfq {
namespace {

static_assert(vf::kFmtInt8 == VF_FORMAT_INT8 && vf::kFmtE4M3 == VF_FORMAT_E4M3,
              "kernel format tags follow vf_format");

constexpr int64_t kMaxGridX = int64_t(1) << 20;   // the kernels stride over head rows

// 16-byte vectors per lane on the 8-element path (tuning constants).
// Quantising, a head row is shared by a group of about kQuantLanes lanes,
// each holding 1, 2 or 4 vectors of it (the fewest that let kQuantLanes lanes
// cover the row); dequantising, every lane holds kDequantNV vectors.
// Measured on GB300 (pages', ragged and large workloads): groups of 4 lanes
// beat 2 and 8 at both D = 64 and D = 128.
#ifndef VF_QUANT_LANES
#define VF_QUANT_LANES 4
#endif
#ifndef VF_DEQUANT_NV
#define VF_DEQUANT_NV 2
#endif
constexpr int64_t kQuantLanes = VF_QUANT_LANES;
constexpr int kQuantMaxNV = 4;
constexpr int kDequantNV = VF_DEQUANT_NV;

// Vectors per lane when quantising a head row of nvec 16-byte vectors.
int quant_nv(int64_t nvec) {
    if (nvec <= kQuantLanes) return 1;
    if (nvec <= 2 * kQuantLanes) return 2;
    return kQuantMaxNV;
}

// Multiplier and shift with n / d == (umulhi(n, mul) + n) >> shift for all
// n < 2^31 and 1 <= d < 2^31 (Granlund and Montgomery's round-up method):
// shift = ceil(log2 d), mul = floor(2^32 (2^shift - d) / d) + 1 < 2^32.
void fast_divisor(int64_t d, uint32_t *mul, uint32_t *shift) {
    uint32_t l = 0;
    while ((int64_t(1) << l) < d) ++l;
    // 2^l - d < d < 2^31, so the numerator is below 2^63
    const uint64_t num = uint64_t((int64_t(1) << l) - d) << 32;
    *mul = uint32_t(num / uint64_t(d) + 1);
    *shift = l;
}

// Widest vector (elements) that keeps every access of both sides aligned:
// codes need VW-byte alignment (row starts are multiples of D), the
// strided side 2*VW bytes.
int pick_vector_width(const Plan &pl) {
    int64_t max_rows = 0;
    for (const auto &p : pl.pieces) max_rows = std::max(max_rows, p.rows);
    for (int vw : {8, 4, 2}) {
        if (pl.D % vw != 0 || pl.d_stride != 1) continue;
        if (reinterpret_cast<uintptr_t>(pl.codes) % uintptr_t(vw)) continue;
        if (max_rows > 1 && pl.row_stride % vw) continue;
        if (pl.heads > 1 && pl.head_stride % vw) continue;
        bool ok = true;
        for (const auto &p : pl.pieces)
            ok = ok && reinterpret_cast<uintptr_t>(p.strided) % uintptr_t(2 * vw) == 0;
        if (ok) return vw;
    }
    return 1;
}

// kPath: 0 = generic, one vector per lane; 1 = generic, per-lane loop;
// 2 = the 8-element path with NV vectors per lane.
template <int VW, int FMT, int kPath, int NV = 1>
int launch_family(const Plan &pl, int lanes_log2, cudaStream_t stream) {
    vf::QArgs a;
    std::memset(&a, 0, sizeof(a));
    a.codes = pl.codes;
    a.scales = pl.scales;
    a.row_stride = pl.row_stride;
    a.head_stride = pl.head_stride;
    a.d_stride = pl.d_stride;
    a.heads = int32_t(pl.heads);
    a.D = int32_t(pl.D);
    a.lanes_log2 = lanes_log2;
    a.nvec = int32_t(pl.D / VW);
    fast_divisor(std::max<int64_t>(pl.heads, 1), &a.div_mul, &a.div_shift);
    const int threads = pl.quantise ? vf::kQuantThreads : vf::kDequantThreads;
    const int rows = !pl.quantise ? vf::kDequantRows
                     : kPath == 2 ? vf::quant_rows8(NV) : vf::kQuantRows;
    const int64_t rows_per_block = int64_t(threads >> lanes_log2) * rows;

    const size_t n = pl.pieces.size();
    for (size_t first = 0; first < n; first += vf::kMaxQPieces) {
        const size_t cnt = std::min<size_t>(vf::kMaxQPieces, n - first);
        int64_t max_hr = 0;
        for (size_t i = 0; i < cnt; ++i) {
            a.pieces[i] = pl.pieces[first + i];
            max_hr = std::max(max_hr, a.pieces[i].rows * pl.heads);
        }
        if (max_hr == 0) continue;
        cudaLaunchConfig_t cfg = {};
        const int64_t gx = std::min(kMaxGridX, (max_hr + rows_per_block - 1) / rows_per_block);
        cfg.gridDim = dim3(unsigned(gx), unsigned(cnt), 1);
        cfg.blockDim = dim3(unsigned(threads), 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e;
        if constexpr (kPath == 2) {
            if (pl.quantise)
                e = cudaLaunchKernelEx(&cfg, vf::quantise_rows8<FMT, NV>, a);
            else
                e = cudaLaunchKernelEx(&cfg, vf::dequantise_rows8<FMT, kDequantNV>, a);
        } else {
            if (pl.quantise)
                e = cudaLaunchKernelEx(&cfg, vf::quantise_rows<VW, FMT, kPath == 0>, a);
            else
                e = cudaLaunchKernelEx(&cfg, vf::dequantise_rows<VW, FMT>, a);
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            return VF_ERR_CUDA;
        }
    }
    return VF_OK;
}

// Group size: the smallest power of two of lanes, at most 32, that covers the
// row's vectors at `per_lane` vectors each.
int lanes_log2_for(int64_t nvec, int64_t per_lane) {
    int lg = 0;
    while (lg < 5 && (int64_t(1) << lg) * per_lane < nvec) ++lg;
    return lg;
}

template <int VW, int FMT>
int launch_vw(const Plan &pl, cudaStream_t stream) {
    const int64_t nvec = pl.D / VW;
    if (VW == 8 && pl.quantise && nvec <= 32 * kQuantMaxNV) {
        switch (quant_nv(nvec)) {
            case 1: return launch_family<VW, FMT, 2, 1>(pl, lanes_log2_for(nvec, 1), stream);
            case 2: return launch_family<VW, FMT, 2, 2>(pl, lanes_log2_for(nvec, 2), stream);
            default:
                return launch_family<VW, FMT, 2, kQuantMaxNV>(
                    pl, lanes_log2_for(nvec, kQuantMaxNV), stream);
        }
    }
    if (VW == 8 && !pl.quantise && nvec <= 32 * kDequantNV)
        return launch_family<VW, FMT, 2, kDequantNV>(pl, lanes_log2_for(nvec, kDequantNV),
                                                     stream);
    const int lg = lanes_log2_for(nvec, 1);
    const bool one = nvec <= (int64_t(1) << lg);
    if (one || !pl.quantise) return launch_family<VW, FMT, 0>(pl, lg, stream);
    return launch_family<VW, FMT, 1>(pl, lg, stream);
}

template <int FMT>
int launch_fmt(const Plan &pl, int vw, cudaStream_t stream) {
    switch (vw) {
        case 8: return launch_vw<8, FMT>(pl, stream);
        case 4: return launch_vw<4, FMT>(pl, stream);
        case 2: return launch_vw<2, FMT>(pl, stream);
        default: return launch_vw<1, FMT>(pl, stream);
    }
}

}  // namespace

int launch(const Plan &pl, cudaStream_t stream) {
    if (pl.pieces.empty()) return VF_OK;
    if (pl.heads > INT32_MAX || pl.D > INT32_MAX || pl.D < 1) return VF_ERR_ARG;
    for (const auto &p : pl.pieces)
        if (p.rows > INT32_MAX / std::max<int64_t>(pl.heads, 1)) return VF_ERR_ARG;
    const int vw = pick_vector_width(pl);
    if (pl.fmt == vf::kFmtInt8) return launch_fmt<vf::kFmtInt8>(pl, vw, stream);
    if (pl.fmt == vf::kFmtE4M3) return launch_fmt<vf::kFmtE4M3>(pl, vw, stream);
    return VF_ERR_ARG;
}

}  // namespace vfq
