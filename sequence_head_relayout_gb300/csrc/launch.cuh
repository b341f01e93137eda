// Launch policy of the relayout kernel: block shape, vector width, grid
// order and the launches themselves.  Included inside the anonymous
// namespace of vf_relayout.cu (it uses ceil_div and the vf_status codes);
// together with relayout_kernel.cuh it decides everything the GPU executes.
// The constants were chosen by measurement on GB300 and can be overridden at
// compile time for tuning sweeps.
#pragma once

#ifndef VF_TARGET_THREADS
#define VF_TARGET_THREADS 512
#endif
constexpr int kTargetThreads = VF_TARGET_THREADS;   // block size aimed at when rows are short
constexpr int64_t kMaxGridZ = 65535;
constexpr int64_t kMaxGridY = 65535;                // grid y limit (the pack swaps x and y)

// The pack cuts every source token row into 3*P runs (one per slab and
// destination); scheduling the pieces of a row group back to back reads each
// source row in one burst, measured 1-3% faster on GB300.  The other ops were
// 2% slower that way, so they walk rows first.
#ifndef VF_PACK_PIECE_FASTEST
#define VF_PACK_PIECE_FASTEST 1
#endif
inline bool schedule_pieces_first(int op) {
    return VF_PACK_PIECE_FASTEST && op == VF_OP_QKV_PACK;
}

// Everything one launch family needs besides the pieces.
struct Plan {
    uint16_t *packed;
    int64_t row_stride, head_stride, d_stride;
    int64_t heads, D;
    bool piece_fastest;            // schedule the pieces of a row group together
    std::vector<vf::Piece> pieces;
};

template <int VW, bool kPackedIsDst>
int launch_family(const Plan &pl, cudaStream_t stream) {
    const int dvec = int(pl.D / VW);
    const int bx = std::min(dvec, vf::kMaxThreads);
    const int by = int(std::min<int64_t>(pl.heads, std::max(1, vf::kMaxThreads / bx)));
    const int bz = std::max(1, std::min(64, kTargetThreads / (bx * by)));
    const int64_t dchunks = ceil_div(dvec, bx);
    const int64_t hchunks = ceil_div(pl.heads, by);
    const int64_t zcount = hchunks * dchunks;              // <= heads * D
    if (zcount > INT32_MAX) return VF_ERR_ARG;

    vf::Args a;
    std::memset(&a, 0, sizeof(a));
    a.packed = pl.packed;
    a.row_stride = pl.row_stride;
    a.head_stride = pl.head_stride;
    a.d_stride = pl.d_stride;
    a.heads = int32_t(pl.heads);
    a.D = int32_t(pl.D);
    a.dchunks = int32_t(dchunks);

    const int64_t rows_per_block = int64_t(vf::kRowsPerThread) * bz;
    const size_t n = pl.pieces.size();
    for (size_t first = 0; first < n; first += vf::kMaxPieces) {
        const size_t cnt = std::min<size_t>(vf::kMaxPieces, n - first);
        int64_t max_rows = 0;
        for (size_t i = 0; i < cnt; ++i) {
            a.pieces[i] = pl.pieces[first + i];
            max_rows = std::max(max_rows, a.pieces[i].rows);
        }
        if (max_rows == 0) continue;
        for (int64_t z0 = 0; z0 < zcount; z0 += kMaxGridZ) {
            a.z_base = int32_t(z0);
            cudaLaunchConfig_t cfg = {};
            const int64_t groups = ceil_div(max_rows, rows_per_block);
            const unsigned zdim = unsigned(std::min<int64_t>(kMaxGridZ, zcount - z0));
            a.piece_fastest = pl.piece_fastest && groups <= kMaxGridY;
            cfg.gridDim = a.piece_fastest ? dim3(unsigned(cnt), unsigned(groups), zdim)
                                          : dim3(unsigned(groups), unsigned(cnt), zdim);
            cfg.blockDim = dim3(unsigned(bx), unsigned(by), unsigned(bz));
            cfg.dynamicSmemBytes = 0;
            cfg.stream = stream;
#if VF_PDL
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
#endif
            if (cudaLaunchKernelEx(&cfg, vf::relayout_rows<VW, kPackedIsDst>, a) != cudaSuccess) {
                cudaGetLastError();
                return VF_ERR_CUDA;
            }
        }
    }
    return VF_OK;
}

template <bool kPackedIsDst>
int launch_dir(const Plan &pl, int vw, cudaStream_t stream) {
    switch (vw) {
        case 8: return launch_family<8, kPackedIsDst>(pl, stream);
        case 4: return launch_family<4, kPackedIsDst>(pl, stream);
        case 2: return launch_family<2, kPackedIsDst>(pl, stream);
        default: return launch_family<1, kPackedIsDst>(pl, stream);
    }
}

// Widest vector (in elements) that keeps every access of both sides aligned.
int pick_vector_width(const Plan &pl) {
    int64_t max_rows = 0;
    for (const auto &p : pl.pieces) max_rows = std::max(max_rows, p.rows);
    for (int vw : {8, 4, 2}) {
        const uintptr_t bytes = uintptr_t(2 * vw);
        if (pl.D % vw != 0) continue;
        if (pl.d_stride != 1) continue;
        if (reinterpret_cast<uintptr_t>(pl.packed) % bytes) continue;
        if (max_rows > 1 && pl.row_stride % vw) continue;
        if (pl.heads > 1 && pl.head_stride % vw) continue;
        bool ok = true;
        for (const auto &p : pl.pieces)
            ok = ok && reinterpret_cast<uintptr_t>(p.strided) % bytes == 0;
        if (ok) return vw;
    }
    return 1;
}

