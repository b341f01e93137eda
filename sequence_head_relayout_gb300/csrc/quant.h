// Internal interface between the host checks (vf_relayout.cu) and the
// launches of the lossy-transport kernels (vf_quant.cu).  Not part of the
// C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "quant_kernel.cuh"

namespace vfq {

struct Plan {
    uint8_t *codes;                     // packed storage, one byte per element
    float *scales;                      // one float per packed head row
    int64_t row_stride, head_stride, d_stride;
    int64_t heads, D;                   // heads per packed token row, elements per head row
    int fmt;                            // vf::kFmtInt8 or vf::kFmtE4M3
    bool quantise;                      // true: strided -> packed (pack, split)
    std::vector<vf::QPiece> pieces;     // each with rows * heads < 2^31
};

// Enqueues the launches of one call; returns a vf_status.
int launch(const Plan &pl, cudaStream_t stream);

}  // namespace vfq
