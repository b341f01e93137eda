// Host side of libvf_relayout.so: argument checks, the piece tables, the
// choice of vector width and the launches.  The C ABI is declared in
// include/vf_relayout.h.
//
// Layout reading ("Sol-Engine alignment on SM86 and SM89", section "What is
// enabled": destination-major storage, Vflash's four-chunk overlap layout):
// chunk quota Q(n) = ceil(n/C) with a short tail; packed storage is blocks
// (c, p), c outer; the pack's block carries head group p as q, k, v slabs;
// the split cuts tokens into P shards of ceil(T/P) and each shard into C
// chunks of ceil(n_p/C); the merge is the inverse of a head-group split.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <vector>

#include "relayout_kernel.cuh"
#include "vf_relayout.h"

namespace {

#ifndef VF_TARGET_THREADS
#define VF_TARGET_THREADS 256
#endif
constexpr int kTargetThreads = VF_TARGET_THREADS;   // block size aimed at when rows are short
constexpr int64_t kMaxTablePieces = int64_t(1) << 20;   // P * C limit
constexpr int64_t kMaxGridZ = 65535;
constexpr int64_t kMaxTokens = int64_t(1) << 30;

// ---------------------------------------------------------------- checked math
bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_add_overflow(a, b, out); }

int64_t ceil_div(int64_t a, int64_t b) { return a == 0 ? 0 : (a - 1) / b + 1; }

// First item of part i when n items are cut with quota ceil(n / parts).
int64_t part_begin(int64_t n, int64_t parts, int64_t i) {
    const int64_t q = ceil_div(n, parts);
    // i <= parts and q * parts < n + parts, so the product cannot overflow
    return std::min(n, i * q);
}

struct Shape {
    int op;
    int64_t T, H, D, P, C;
};

int check_shape(const Shape &s) {
    if (s.op < VF_OP_QKV_PACK || s.op > VF_OP_HEAD_MERGE) return VF_ERR_ARG;
    if (s.T < 0 || s.H < 0 || s.D < 0 || s.P < 1 || s.C < 1) return VF_ERR_ARG;
    if (s.T > kMaxTokens) return VF_ERR_ARG;          // row indices stay in int32
    if (s.op != VF_OP_ATTN_SPLIT && s.H % s.P != 0) return VF_ERR_ARG;
    int64_t n, pc;
    if (!mul_ok(s.T, s.H, &n) || !mul_ok(n, s.D, &n)) return VF_ERR_OVERFLOW;
    if (s.op == VF_OP_QKV_PACK && !mul_ok(n, 3, &n)) return VF_ERR_OVERFLOW;
    if (!mul_ok(n, 2, &n)) return VF_ERR_OVERFLOW;            // bytes
    if (!mul_ok(s.P, s.C, &pc) || pc > kMaxTablePieces) return VF_ERR_ARG;
    return VF_OK;
}

int64_t packed_elems(const Shape &s) {
    return s.T * s.H * s.D * (s.op == VF_OP_QKV_PACK ? 3 : 1);
}

// One (c, p) entry of the piece table.
struct Entry {
    int64_t tok_start, tok_len, packed_off;
};

// Piece table in storage order (c outer, p inner).  Requires check_shape OK.
std::vector<Entry> piece_table(const Shape &s) {
    std::vector<Entry> out;
    out.reserve(size_t(s.P * s.C));
    int64_t cursor = 0;                                     // packed elements
    if (s.op == VF_OP_ATTN_SPLIT) {
        const int64_t per_token = s.H * s.D;
        for (int64_t c = 0; c < s.C; ++c)
            for (int64_t p = 0; p < s.P; ++p) {
                const int64_t a = part_begin(s.T, s.P, p);
                const int64_t n = part_begin(s.T, s.P, p + 1) - a;
                const int64_t u0 = part_begin(n, s.C, c);
                const int64_t len = part_begin(n, s.C, c + 1) - u0;
                out.push_back({a + u0, len, cursor});
                cursor += len * per_token;
            }
    } else {
        const int64_t per_token = (s.op == VF_OP_QKV_PACK ? 3 : 1) * (s.H / s.P) * s.D;
        for (int64_t c = 0; c < s.C; ++c) {
            const int64_t t0 = part_begin(s.T, s.C, c);
            const int64_t len = part_begin(s.T, s.C, c + 1) - t0;
            for (int64_t p = 0; p < s.P; ++p) {
                out.push_back({t0, len, cursor});
                cursor += len * per_token;
            }
        }
    }
    return out;
}

// Largest element offset a strided view addresses (all strides >= 0).
int max_offset(const int64_t *ext, const int64_t *str, int nd, int64_t *out) {
    int64_t m = 0;
    for (int i = 0; i < nd; ++i) {
        if (str[i] < 0) return VF_ERR_ARG;
        if (ext[i] <= 1) continue;
        int64_t term;
        if (!mul_ok(ext[i] - 1, str[i], &term) || !add_ok(m, term, &m)) return VF_ERR_OVERFLOW;
    }
    *out = m;
    return VF_OK;
}

// True when a write view never maps two logical elements to one address:
// sorted by stride, each stride must exceed the span of the smaller ones.
bool non_overlapping(const int64_t *ext, const int64_t *str, int nd) {
    int idx[4] = {0, 0, 0, 0};
    int k = 0;
    for (int i = 0; i < nd; ++i)
        if (ext[i] > 1) idx[k++] = i;
    for (int j = 1; j < k; ++j)                 // insertion sort by stride, k <= 4
        for (int m = j; m > 0 && str[idx[m]] < str[idx[m - 1]]; --m) std::swap(idx[m], idx[m - 1]);
    int64_t span = 0;
    for (int j = 0; j < k; ++j) {
        const int i = idx[j];
        if (str[i] <= span) return false;
        span += str[i] * (ext[i] - 1);      // bounded by max_offset, no overflow
    }
    return true;
}

// Byte ranges [a, a + na) and [b, b + nb) intersect.
bool ranges_overlap(uintptr_t a, uint64_t na, uintptr_t b, uint64_t nb) {
    if (na == 0 || nb == 0) return false;
    return a < b + nb && b < a + na;
}

int check_pointer(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return VF_ERR_CUDA;
    }
    if (at.type == cudaMemoryTypeUnregistered) return VF_ERR_ARG;
    if (at.type == cudaMemoryTypeDevice) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return VF_ERR_CUDA;
        }
        if (at.device != dev) return VF_ERR_ARG;       // another GPU's memory
    }
    return VF_OK;
}

// Everything one launch family needs besides the pieces.
struct Plan {
    const uint16_t *src;
    uint16_t *dst;
    bool packed_is_dst;
    int64_t row_stride, head_stride, d_stride, slab_stride;
    int64_t heads, D, slabs;
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
    const int64_t zcount = pl.slabs * hchunks * dchunks;   // <= 3 * heads * D
    if (zcount > INT32_MAX) return VF_ERR_ARG;

    vf::Args a;
    std::memset(&a, 0, sizeof(a));
    a.src = pl.src;
    a.dst = pl.dst;
    a.row_stride = pl.row_stride;
    a.head_stride = pl.head_stride;
    a.d_stride = pl.d_stride;
    a.slab_stride = pl.slab_stride;
    a.heads = int32_t(pl.heads);
    a.D = int32_t(pl.D);
    a.hchunks = int32_t(hchunks);
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
        a.npieces = int32_t(cnt);
        if (max_rows == 0) continue;
        for (int64_t z0 = 0; z0 < zcount; z0 += kMaxGridZ) {
            a.z_base = int32_t(z0);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(unsigned(ceil_div(max_rows, rows_per_block)), unsigned(cnt),
                               unsigned(std::min<int64_t>(kMaxGridZ, zcount - z0)));
            cfg.blockDim = dim3(unsigned(bx), unsigned(by), unsigned(bz));
            cfg.dynamicSmemBytes = 0;
            cfg.stream = stream;
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
int pick_vector_width(const Plan &pl, const void *packed, const void *strided) {
    int64_t max_rows = 0;
    for (const auto &p : pl.pieces) max_rows = std::max(max_rows, p.rows);
    for (int vw : {8, 4, 2}) {
        const int64_t bytes = 2 * vw;
        if (pl.D % vw != 0) continue;
        if (pl.d_stride != 1) continue;
        if (reinterpret_cast<uintptr_t>(packed) % bytes) continue;
        if (reinterpret_cast<uintptr_t>(strided) % bytes) continue;
        if (max_rows > 1 && pl.row_stride % vw) continue;
        if (pl.heads > 1 && pl.head_stride % vw) continue;
        if (pl.slabs > 1 && pl.slab_stride % vw) continue;
        bool ok = true;
        for (const auto &p : pl.pieces) ok = ok && (p.strided_off % vw == 0);
        if (ok) return vw;
    }
    return 1;
}

int run(const Shape &s, const void *src, const int64_t *strides, void *dst, cudaStream_t stream) {
    int rc = check_shape(s);
    if (rc != VF_OK) return rc;

    // The strided side's logical extents and strides.
    int64_t ext[4], str[4];
    int nd;
    if (s.op == VF_OP_QKV_PACK) {
        nd = 4;
        ext[0] = s.T; ext[1] = 3; ext[2] = s.H; ext[3] = s.D;
    } else {
        nd = 3;
        ext[0] = s.T; ext[1] = s.H; ext[2] = s.D;
    }
    if (strides) {
        for (int i = 0; i < nd; ++i) str[i] = strides[i];
    } else if (s.op == VF_OP_HEAD_MERGE) {
        str[0] = s.H * s.D; str[1] = s.D; str[2] = 1;
    } else {
        return VF_ERR_ARG;
    }
    for (int i = 0; i < nd; ++i) {
        if (str[i] < 0) return VF_ERR_ARG;
        if (ext[i] <= 1) str[i] = 0;             // unused: the index is always 0
    }
    int64_t span;
    if ((rc = max_offset(ext, str, nd, &span)) != VF_OK) return rc;
    int64_t strided_bytes;
    if (!add_ok(span, 1, &strided_bytes) || !mul_ok(strided_bytes, 2, &strided_bytes))
        return VF_ERR_OVERFLOW;

    const int64_t n = packed_elems(s);
    if (n == 0) return VF_OK;
    if (src == nullptr || dst == nullptr) return VF_ERR_ARG;
    // 16-bit elements: both pointers must be 2-byte aligned
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 1u)
        return VF_ERR_ARG;
    if (s.op == VF_OP_HEAD_MERGE && !non_overlapping(ext, str, nd)) return VF_ERR_ARG;

    const bool packed_is_dst = s.op != VF_OP_HEAD_MERGE;
    const void *packed = packed_is_dst ? static_cast<const void *>(dst) : src;
    const void *strided = packed_is_dst ? src : static_cast<const void *>(dst);
    const uintptr_t pa = reinterpret_cast<uintptr_t>(packed);
    const uintptr_t sa = reinterpret_cast<uintptr_t>(strided);
    if (pa > UINTPTR_MAX - uint64_t(2 * n) || sa > UINTPTR_MAX - uint64_t(strided_bytes))
        return VF_ERR_OVERFLOW;
    if (ranges_overlap(pa, uint64_t(2 * n), sa, uint64_t(strided_bytes))) return VF_ERR_ALIAS;

    if ((rc = check_pointer(src)) != VF_OK) return rc;
    if ((rc = check_pointer(dst)) != VF_OK) return rc;

    Plan pl;
    pl.src = static_cast<const uint16_t *>(src);
    pl.dst = static_cast<uint16_t *>(dst);
    pl.packed_is_dst = packed_is_dst;
    pl.D = s.D;
    const std::vector<Entry> table = piece_table(s);
    pl.pieces.reserve(table.size());
    if (s.op == VF_OP_QKV_PACK) {
        const int64_t Hp = s.H / s.P;
        pl.row_stride = str[0];
        pl.slab_stride = str[1];
        pl.head_stride = str[2];
        pl.d_stride = str[3];
        pl.heads = Hp;
        pl.slabs = 3;
        for (size_t e = 0; e < table.size(); ++e) {
            const int64_t p = int64_t(e) % s.P;
            pl.pieces.push_back({table[e].packed_off,
                                 table[e].tok_start * str[0] + p * Hp * str[2],
                                 table[e].tok_len});
        }
    } else if (s.op == VF_OP_ATTN_SPLIT) {
        pl.row_stride = str[0];
        pl.head_stride = str[1];
        pl.d_stride = str[2];
        pl.slab_stride = 0;
        pl.heads = s.H;
        pl.slabs = 1;
        for (const Entry &e : table)
            pl.pieces.push_back({e.packed_off, e.tok_start * str[0], e.tok_len});
    } else {
        const int64_t Hp = s.H / s.P;
        pl.row_stride = str[0];
        pl.head_stride = str[1];
        pl.d_stride = str[2];
        pl.slab_stride = 0;
        pl.heads = Hp;
        pl.slabs = 1;
        for (size_t e = 0; e < table.size(); ++e) {
            const int64_t p = int64_t(e) % s.P;
            pl.pieces.push_back({table[e].packed_off,
                                 table[e].tok_start * str[0] + p * Hp * str[1],
                                 table[e].tok_len});
        }
    }
    if (pl.heads > INT32_MAX || pl.D > INT32_MAX) return VF_ERR_ARG;

    const int vw = pick_vector_width(pl, packed, strided);
    return packed_is_dst ? launch_dir<true>(pl, vw, stream) : launch_dir<false>(pl, vw, stream);
}

}  // namespace

extern "C" {

int vf_qkv_pack(const void *src, const int64_t src_strides[4], int64_t T, int64_t H,
                int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return run({VF_OP_QKV_PACK, T, H, D, P, C}, src, src_strides, dst,
               reinterpret_cast<cudaStream_t>(stream));
}

int vf_attn_split(const void *src, const int64_t src_strides[3], int64_t T, int64_t H,
                  int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return run({VF_OP_ATTN_SPLIT, T, H, D, P, C}, src, src_strides, dst,
               reinterpret_cast<cudaStream_t>(stream));
}

int vf_head_merge(const void *src, const int64_t dst_strides[3], int64_t T, int64_t H,
                  int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return run({VF_OP_HEAD_MERGE, T, H, D, P, C}, src, dst_strides, dst,
               reinterpret_cast<cudaStream_t>(stream));
}

int64_t vf_packed_elems(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C) {
    const Shape s{op, T, H, D, P, C};
    const int rc = check_shape(s);
    return rc != VF_OK ? rc : packed_elems(s);
}

int64_t vf_piece_table(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                       int64_t *tok_start, int64_t *tok_len, int64_t *packed_off,
                       int64_t cap) {
    const Shape s{op, T, H, D, P, C};
    const int rc = check_shape(s);
    if (rc != VF_OK) return rc;
    if (cap < P * C) return VF_ERR_CAPACITY;
    if (!tok_start || !tok_len || !packed_off) return VF_ERR_ARG;
    const std::vector<Entry> t = piece_table(s);
    for (size_t i = 0; i < t.size(); ++i) {
        tok_start[i] = t[i].tok_start;
        tok_len[i] = t[i].tok_len;
        packed_off[i] = t[i].packed_off;
    }
    return int64_t(t.size());
}

const char *vf_status_string(int status) {
    switch (status) {
        case VF_OK: return "ok";
        case VF_ERR_ARG: return "invalid argument";
        case VF_ERR_OVERFLOW: return "size or offset overflows int64";
        case VF_ERR_ALIAS: return "destination overlaps the source";
        case VF_ERR_CUDA: return "CUDA runtime error";
        case VF_ERR_CAPACITY: return "output capacity too small";
        default: return "unknown status";
    }
}

}  // extern "C"
