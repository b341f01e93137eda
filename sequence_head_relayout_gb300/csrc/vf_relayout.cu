// Host side of libvf_relayout.so: argument checks, the piece tables, the
// choice of vector width and the launches.  The C ABI is declared in
// include/vf_relayout.h.
//
// Layout reading ("Sol-Engine alignment on SM86 and SM89", section "What is
// enabled": destination-major storage, Vflash's four-chunk overlap layout):
// chunk quota Q(n) = ceil(n/C) with a short tail; packed storage is blocks
// (c, p), c outer; the pack's block carries head group p as q, k, v slabs;
// the split cuts tokens into P shards of ceil(T/P) and each shard into C
// chunks of ceil(n_p/C); the merge is the inverse of a head-group split; the
// receive-side unpack ("速度、显存与质量", section "剖析单次去噪请求": QKV
// unpack) reads, per chunk, the pack blocks of the P source ranks' shards.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

#include "quant.h"
#include "relayout_kernel.cuh"
#include "tiled_kernel.cuh"
#include "vf_relayout.h"

namespace {

constexpr int64_t kMaxTablePieces = int64_t(1) << 20;   // P * C limit
constexpr int64_t kMaxExtent = int64_t(1) << 30;        // T, H and D limit

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

bool is_op(int op) { return op >= VF_OP_QKV_PACK && op <= VF_OP_QKV_UNPACK; }

// Pack and unpack move q, k and v slabs.
int64_t slabs_of(int op) { return (op == VF_OP_QKV_PACK || op == VF_OP_QKV_UNPACK) ? 3 : 1; }

int check_shape(const Shape &s) {
    if (!is_op(s.op)) return VF_ERR_ARG;
    if (s.T < 0 || s.H < 0 || s.D < 0 || s.P < 1 || s.C < 1) return VF_ERR_ARG;
    // row, head and d indices stay well inside int32 in the kernel
    if (s.T > kMaxExtent || s.H > kMaxExtent || s.D > kMaxExtent) return VF_ERR_ARG;
    if (s.op != VF_OP_ATTN_SPLIT && s.H % s.P != 0) return VF_ERR_ARG;
    int64_t n, pc;
    if (!mul_ok(s.T, s.H, &n) || !mul_ok(n, s.D, &n)) return VF_ERR_OVERFLOW;
    if (!mul_ok(n, 3, &n) || !mul_ok(n, 2, &n)) return VF_ERR_OVERFLOW;   // bytes, with slabs
    if (!mul_ok(s.P, s.C, &pc) || pc > kMaxTablePieces) return VF_ERR_ARG;
    return VF_OK;
}

// Elements of the packed side.
int64_t packed_elems(const Shape &s) {
    const int64_t thd = s.T * s.H * s.D;
    switch (s.op) {
        case VF_OP_QKV_PACK: return 3 * thd;
        case VF_OP_QKV_UNPACK: return 3 * thd / s.P;
        default: return thd;
    }
}

// Heads in one packed row.
int64_t heads_per_row(const Shape &s) {
    return s.op == VF_OP_ATTN_SPLIT ? s.H : s.H / s.P;
}

// One (c, p) entry of the piece table.
struct Entry {
    int64_t tok_start, tok_len, packed_off;
};

// Piece table, one entry per (c, p) at index c * P + p.  Pack and merge cut
// the T tokens of this rank into chunks; the split and the unpack cut T into
// P token shards first and each shard into chunks.  packed_off places the
// blocks back to back in the requested storage order: c outer (chunk-major,
// the overlap layout) or p outer (slot-major).  Requires check_shape OK.
std::vector<Entry> piece_table(const Shape &s, int order) {
    std::vector<Entry> out(size_t(s.P * s.C));
    const int64_t per_token = slabs_of(s.op) * heads_per_row(s) * s.D;
    const bool sharded = s.op == VF_OP_ATTN_SPLIT || s.op == VF_OP_QKV_UNPACK;
    for (int64_t c = 0; c < s.C; ++c)
        for (int64_t p = 0; p < s.P; ++p) {
            Entry &e = out[size_t(c * s.P + p)];
            if (sharded) {
                const int64_t a = part_begin(s.T, s.P, p);
                const int64_t n = part_begin(s.T, s.P, p + 1) - a;
                const int64_t u0 = part_begin(n, s.C, c);
                e.tok_start = a + u0;
                e.tok_len = part_begin(n, s.C, c + 1) - u0;
            } else {
                e.tok_start = part_begin(s.T, s.C, c);
                e.tok_len = part_begin(s.T, s.C, c + 1) - e.tok_start;
            }
        }
    int64_t cursor = 0;                                     // packed elements
    const int64_t outer = order == VF_ORDER_SLOT_MAJOR ? s.P : s.C;
    const int64_t inner = order == VF_ORDER_SLOT_MAJOR ? s.C : s.P;
    for (int64_t i = 0; i < outer; ++i)
        for (int64_t j = 0; j < inner; ++j) {
            const int64_t c = order == VF_ORDER_SLOT_MAJOR ? j : i;
            const int64_t p = order == VF_ORDER_SLOT_MAJOR ? i : j;
            Entry &e = out[size_t(c * s.P + p)];
            e.packed_off = cursor;
            cursor += e.tok_len * per_token;
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

// A byte range [lo, lo + len).
struct Range {
    uintptr_t lo;
    uint64_t len;
};

bool overlap(const Range &a, const Range &b) {
    if (a.len == 0 || b.len == 0) return false;
    return a.lo < b.lo + b.len && b.lo < a.lo + a.len;
}

int check_pointer(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return VF_ERR_CUDA;
    }
    if (at.type == cudaMemoryTypeUnregistered) return VF_ERR_ARG;
    // page-locked host memory must be mapped at the same address on the device
    if (at.type == cudaMemoryTypeHost && at.devicePointer != p) return VF_ERR_ARG;
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

// One call, after the entry point has mapped its arguments.
struct Request {
    Shape s;
    int order;                     // vf_order of the packed storage
    int64_t c_begin, c_end;        // chunk range [c_begin, c_end)
    void *packed;                  // packed storage (read for merge/unpack)
    const void *strided[3];        // strided-side base per slab
    int64_t str[3];                // strided view strides (token, head, d), elements
    int64_t heads_view;            // head extent of the strided view
    bool strided_written;          // merge, unpack
    int fmt;                       // 0: exact 16-bit; else vf_format of the codes
    float *scales;                 // lossy transport: one float per packed head row
};

// Block shape, vector width, grid order and launches.
#include "launch.cuh"

// The shared-memory staged path (tiled_kernel.cuh): 16- or 32-byte head rows
// (D = 8 or 16), unit d-stride, a head-major strided side (consecutive tokens
// of one head closer together than consecutive heads of one token), every
// head row 16-byte aligned.
#ifndef VF_TILED_MAX_D
#define VF_TILED_MAX_D 16
#endif
bool use_tiled(const Plan &pl) {
    if (pl.d_stride != 1 || pl.heads < 2) return false;
    if (pl.D > VF_TILED_MAX_D || (pl.D != 8 && pl.D != 16 && pl.D != 32 && pl.D != 64 &&
                                  pl.D != 128)) return false;
    if (pl.row_stride >= pl.head_stride) return false;
    if (pl.row_stride % 8 || pl.head_stride % 8) return false;
    if (ceil_div(pl.heads, vf::kTileHeads) > kMaxGridZ) return false;
    if (reinterpret_cast<uintptr_t>(pl.packed) % 16) return false;
    for (const auto &p : pl.pieces)
        if (reinterpret_cast<uintptr_t>(p.strided) % 16) return false;
    return true;
}

template <int DV, bool kPackedIsDst>
int launch_tiled(const Plan &pl, cudaStream_t stream) {
    vf::TiledArgs a;
    std::memset(&a, 0, sizeof(a));
    a.packed = pl.packed;
    a.row_stride = pl.row_stride;
    a.head_stride = pl.head_stride;
    a.heads = int32_t(pl.heads);
    a.head_tiles = int32_t(ceil_div(pl.heads, vf::kTileHeads));
    const size_t n = pl.pieces.size();
    for (size_t first = 0; first < n; first += vf::kMaxPieces) {
        const size_t cnt = std::min<size_t>(vf::kMaxPieces, n - first);
        int64_t max_rows = 0;
        for (size_t i = 0; i < cnt; ++i) {
            a.pieces[i] = pl.pieces[first + i];
            max_rows = std::max(max_rows, a.pieces[i].rows);
        }
        if (max_rows == 0) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(ceil_div(max_rows, vf::TileShape<DV>::kTok)), unsigned(cnt),
                           unsigned(a.head_tiles));
        cfg.blockDim = dim3(unsigned(vf::kTileThreads), 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
#if VF_PDL
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
#endif
        if (cudaLaunchKernelEx(&cfg, vf::relayout_tiled<DV, kPackedIsDst>, a) != cudaSuccess) {
            cudaGetLastError();
            return VF_ERR_CUDA;
        }
    }
    return VF_OK;
}

template <bool kPackedIsDst>
int launch_tiled_dir(const Plan &pl, cudaStream_t stream) {
    switch (pl.D) {
        case 8: return launch_tiled<1, kPackedIsDst>(pl, stream);
        case 16: return launch_tiled<2, kPackedIsDst>(pl, stream);
#if VF_TILED_MAX_D >= 32
        case 32: return launch_tiled<4, kPackedIsDst>(pl, stream);
#endif
#if VF_TILED_MAX_D >= 64
        case 64: return launch_tiled<8, kPackedIsDst>(pl, stream);
#endif
#if VF_TILED_MAX_D >= 128
        case 128: return launch_tiled<16, kPackedIsDst>(pl, stream);
#endif
        default: return VF_ERR_ARG;
    }
}

int run(Request rq, cudaStream_t stream) {
    const Shape &s = rq.s;
    int rc = check_shape(s);
    if (rc != VF_OK) return rc;
    if (rq.c_begin < 0 || rq.c_end < rq.c_begin || rq.c_end > s.C) return VF_ERR_ARG;
    if (rq.order != VF_ORDER_CHUNK_MAJOR && rq.order != VF_ORDER_SLOT_MAJOR) return VF_ERR_ARG;
    if (rq.fmt != 0 && rq.fmt != VF_FORMAT_INT8 && rq.fmt != VF_FORMAT_E4M3) return VF_ERR_ARG;
    const bool lossy = rq.fmt != 0;
    const int64_t slabs = slabs_of(s.op);

    // Geometry of one strided slab view [T][heads_view][D].
    const int64_t ext[3] = {s.T, rq.heads_view, s.D};
    for (int i = 0; i < 3; ++i) {
        if (rq.str[i] < 0) return VF_ERR_ARG;
        if (ext[i] <= 1) rq.str[i] = 0;          // unused: the index is always 0
    }
    int64_t span, view_bytes;
    if ((rc = max_offset(ext, rq.str, 3, &span)) != VF_OK) return rc;
    if (!add_ok(span, 1, &view_bytes) || !mul_ok(view_bytes, 2, &view_bytes))
        return VF_ERR_OVERFLOW;

    const int64_t n = packed_elems(s);
    if (n == 0 || rq.c_begin == rq.c_end) return VF_OK;

    // Pointers: present, aligned (16-bit elements; codes are bytes, scales
    // floats), ranges inside the address space.
    if (rq.packed == nullptr) return VF_ERR_ARG;
    if (lossy && (rq.scales == nullptr || reinterpret_cast<uintptr_t>(rq.scales) % 4u))
        return VF_ERR_ARG;
    uintptr_t bits = lossy ? 0 : reinterpret_cast<uintptr_t>(rq.packed);
    for (int64_t i = 0; i < slabs; ++i) {
        if (rq.strided[i] == nullptr) return VF_ERR_ARG;
        bits |= reinterpret_cast<uintptr_t>(rq.strided[i]);
    }
    if (bits & 1u) return VF_ERR_ARG;
    if (rq.strided_written && !non_overlapping(ext, rq.str, 3)) return VF_ERR_ARG;

    const Range packed{reinterpret_cast<uintptr_t>(rq.packed), uint64_t(lossy ? n : 2 * n)};
    if (packed.lo > UINTPTR_MAX - packed.len) return VF_ERR_OVERFLOW;
    // n > 0 here, so D > 0; n / D head rows, 4 bytes each (n * 2 fits int64)
    const Range scales{reinterpret_cast<uintptr_t>(rq.scales), lossy ? uint64_t(n / s.D) * 4 : 0};
    if (scales.lo > UINTPTR_MAX - scales.len) return VF_ERR_OVERFLOW;
    if (overlap(packed, scales)) return VF_ERR_ALIAS;
    Range views[3];
    for (int64_t i = 0; i < slabs; ++i) {
        views[i] = {reinterpret_cast<uintptr_t>(rq.strided[i]), uint64_t(view_bytes)};
        if (views[i].lo > UINTPTR_MAX - views[i].len) return VF_ERR_OVERFLOW;
        if (overlap(packed, views[i]) || overlap(scales, views[i])) return VF_ERR_ALIAS;
    }
    if (rq.strided_written)
        for (int64_t i = 0; i < slabs; ++i)
            for (int64_t j = i + 1; j < slabs; ++j)
                if (overlap(views[i], views[j])) return VF_ERR_ALIAS;

    if ((rc = check_pointer(rq.packed)) != VF_OK) return rc;
    if (lossy && (rc = check_pointer(rq.scales)) != VF_OK) return rc;
    for (int64_t i = 0; i < slabs; ++i) {
        bool seen = false;
        for (int64_t j = 0; j < i; ++j) seen = seen || rq.strided[j] == rq.strided[i];
        if (!seen && (rc = check_pointer(rq.strided[i])) != VF_OK) return rc;
    }

    // Pieces of the requested chunks, one per (c, p, slab).  Pack and merge
    // address head group p of a full-head view; the split and the unpack
    // address all heads of their view.  A pack or unpack block holds its
    // q, k, v slabs back to back, each rows x heads x D.
    const int64_t heads = heads_per_row(s);
    if (heads > INT32_MAX || s.D > INT32_MAX) return VF_ERR_ARG;
    const std::vector<Entry> table = piece_table(s, rq.order);
    const int64_t group_heads = (s.op == VF_OP_QKV_PACK || s.op == VF_OP_HEAD_MERGE)
                                    ? s.H / s.P : 0;
    const int64_t R = heads * s.D;
    struct Raw {
        int64_t packed_off;
        uint16_t *base;
        int64_t rows;
    };
    std::vector<Raw> raw;
    raw.reserve(size_t((rq.c_end - rq.c_begin) * s.P * slabs));
    for (int64_t c = rq.c_begin; c < rq.c_end; ++c)
        for (int64_t p = 0; p < s.P; ++p) {
            const Entry &e = table[size_t(c * s.P + p)];
            if (e.tok_len == 0) continue;             // empty chunk or shard
            // element offset of the block's first row in each slab view; it
            // lies inside the view (checked extent), so it cannot overflow
            const int64_t off = e.tok_start * rq.str[0] + p * group_heads * rq.str[1];
            for (int64_t sl = 0; sl < slabs; ++sl) {
                uint16_t *base = const_cast<uint16_t *>(
                    static_cast<const uint16_t *>(rq.strided[sl]));
                raw.push_back({e.packed_off + sl * e.tok_len * R, base + off, e.tok_len});
            }
        }
    if (raw.empty()) return VF_OK;
    const bool packed_is_dst = s.op == VF_OP_QKV_PACK || s.op == VF_OP_ATTN_SPLIT;

    if (lossy) {
        vfq::Plan q;
        q.codes = static_cast<uint8_t *>(rq.packed);
        q.scales = rq.scales;
        q.row_stride = rq.str[0];
        q.head_stride = rq.str[1];
        q.d_stride = rq.str[2];
        q.heads = heads;
        q.D = s.D;
        q.fmt = rq.fmt;
        q.quantise = packed_is_dst;
        // block offsets are whole head rows: multiples of D
        for (const Raw &r : raw) q.pieces.push_back({r.packed_off / s.D, r.base, r.rows});
        return vfq::launch(q, stream);
    }

    Plan pl;
    pl.packed = static_cast<uint16_t *>(rq.packed);
    pl.row_stride = rq.str[0];
    pl.head_stride = rq.str[1];
    pl.d_stride = rq.str[2];
    pl.heads = heads;
    pl.D = s.D;
    pl.piece_fastest = schedule_pieces_first(s.op);
    for (const Raw &r : raw) pl.pieces.push_back({r.packed_off, r.base, r.rows});
    if (use_tiled(pl))
        return packed_is_dst ? launch_tiled_dir<true>(pl, stream)
                             : launch_tiled_dir<false>(pl, stream);
    const int vw = pick_vector_width(pl);
    return packed_is_dst ? launch_dir<true>(pl, vw, stream) : launch_dir<false>(pl, vw, stream);
}

cudaStream_t as_stream(vf_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Chunk range [c_begin, c_begin + c_count) without overflow; run() checks it.
int64_t range_end(int64_t c_begin, int64_t c_count) {
    int64_t e;
    if (c_count < 0 || !add_ok(c_begin, c_count, &e)) return -1;
    return e;
}

int pack_common(const void *q, const void *k, const void *v, const int64_t *str,
                int64_t T, int64_t H, int64_t D, int64_t P, int64_t C, int64_t c_begin,
                int64_t c_count, void *dst, vf_stream_t stream, int fmt = 0,
                float *scales = nullptr) {
    Request rq{};
    rq.fmt = fmt;
    rq.scales = scales;
    rq.s = {VF_OP_QKV_PACK, T, H, D, P, C};
    rq.c_begin = c_begin;
    rq.c_end = range_end(c_begin, c_count);
    rq.packed = dst;
    rq.strided[0] = q;
    rq.strided[1] = k;
    rq.strided[2] = v;
    for (int i = 0; i < 3; ++i) rq.str[i] = str[i];
    rq.heads_view = H;
    rq.strided_written = false;
    return run(rq, as_stream(stream));
}

int pack4(const void *src, const int64_t src_strides[4], int64_t T, int64_t H, int64_t D,
          int64_t P, int64_t C, int64_t c_begin, int64_t c_count, void *dst,
          vf_stream_t stream, int fmt = 0, float *scales = nullptr) {
    if (src_strides == nullptr) return VF_ERR_ARG;
    const int64_t ss = src_strides[1];
    if (ss < 0) return VF_ERR_ARG;
    const int64_t str[3] = {src_strides[0], src_strides[2], src_strides[3]};
    if (src == nullptr)      // only legal when nothing is moved; run() decides
        return pack_common(nullptr, nullptr, nullptr, str, T, H, D, P, C, c_begin, c_count,
                           dst, stream, fmt, scales);
    // slab s of the [T][3][H][D] view starts s * ss elements after src
    int64_t off2;
    if (!mul_ok(ss, 4, &off2)) return VF_ERR_OVERFLOW;                 // 2 slabs x 2 bytes
    const uintptr_t base = reinterpret_cast<uintptr_t>(src);
    if (base > UINTPTR_MAX - uint64_t(off2)) return VF_ERR_OVERFLOW;
    const char *b = static_cast<const char *>(src);
    return pack_common(src, b + 2 * ss, b + 4 * ss, str, T, H, D, P, C, c_begin, c_count, dst,
                       stream, fmt, scales);
}

int split_common(const void *src, const int64_t src_strides[3], int64_t T, int64_t H,
                 int64_t D, int64_t P, int64_t C, int64_t c_begin, int64_t c_count, void *dst,
                 vf_stream_t stream, int fmt = 0, float *scales = nullptr) {
    if (src_strides == nullptr) return VF_ERR_ARG;
    Request rq{};
    rq.fmt = fmt;
    rq.scales = scales;
    rq.s = {VF_OP_ATTN_SPLIT, T, H, D, P, C};
    rq.c_begin = c_begin;
    rq.c_end = range_end(c_begin, c_count);
    rq.packed = dst;
    rq.strided[0] = src;
    for (int i = 0; i < 3; ++i) rq.str[i] = src_strides[i];
    rq.heads_view = H;
    rq.strided_written = false;
    return run(rq, as_stream(stream));
}

int merge_common(const void *src, const int64_t dst_strides[3], int64_t T, int64_t H,
                 int64_t D, int64_t P, int64_t C, int64_t c_begin, int64_t c_count, void *dst,
                 vf_stream_t stream, int fmt = 0, const float *scales = nullptr) {
    Request rq{};
    rq.fmt = fmt;
    rq.scales = const_cast<float *>(scales);
    rq.s = {VF_OP_HEAD_MERGE, T, H, D, P, C};
    rq.c_begin = c_begin;
    rq.c_end = range_end(c_begin, c_count);
    rq.packed = const_cast<void *>(src);
    rq.strided[0] = dst;
    if (dst_strides) {
        for (int i = 0; i < 3; ++i) rq.str[i] = dst_strides[i];
    } else {
        if (H < 0 || D < 0 || !mul_ok(H, D, &rq.str[0])) return VF_ERR_ARG;
        rq.str[1] = D;
        rq.str[2] = 1;
    }
    rq.heads_view = H;
    rq.strided_written = true;
    return run(rq, as_stream(stream));
}

int unpack_common(const void *recv, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                  int64_t c_begin, int64_t c_count, void *q, void *k, void *v,
                  const int64_t out_strides[3], vf_stream_t stream, int fmt = 0,
                  const float *scales = nullptr) {
    if (P < 1 || H < 0 || D < 0 || H % P != 0) return VF_ERR_ARG;
    Request rq{};
    rq.fmt = fmt;
    rq.scales = const_cast<float *>(scales);
    rq.s = {VF_OP_QKV_UNPACK, T, H, D, P, C};
    rq.c_begin = c_begin;
    rq.c_end = range_end(c_begin, c_count);
    rq.packed = const_cast<void *>(recv);
    rq.strided[0] = q;
    rq.strided[1] = k;
    rq.strided[2] = v;
    const int64_t Hp = H / P;
    if (out_strides) {
        for (int i = 0; i < 3; ++i) rq.str[i] = out_strides[i];
    } else {
        if (!mul_ok(Hp, D, &rq.str[0])) return VF_ERR_OVERFLOW;
        rq.str[1] = D;
        rq.str[2] = 1;
    }
    rq.heads_view = Hp;
    rq.strided_written = true;
    return run(rq, as_stream(stream));
}

// vf_relayout and vf_relayout_q: map the descriptor onto a Request.
int relayout_desc(const vf_relayout_desc *d, int fmt, float *scales, vf_stream_t stream) {
    Request rq{};
    rq.fmt = fmt;
    rq.scales = scales;
    rq.s = {d->op, d->T, d->H, d->D, d->P, d->C};
    if (!is_op(d->op)) return VF_ERR_ARG;
    rq.order = d->order;
    rq.c_begin = d->c_begin;
    rq.c_end = range_end(d->c_begin, d->c_count);
    rq.packed = d->packed;
    const int64_t slabs = slabs_of(d->op);
    for (int i = 0; i < 3; ++i) rq.strided[i] = i < slabs ? d->strided[i] : nullptr;
    for (int i = 0; i < 3; ++i) rq.str[i] = d->strides[i];
    if (d->P < 1 || d->H < 0) return VF_ERR_ARG;
    rq.heads_view = d->op == VF_OP_QKV_UNPACK ? d->H / d->P : d->H;
    rq.strided_written = d->op == VF_OP_HEAD_MERGE || d->op == VF_OP_QKV_UNPACK;
    return run(rq, as_stream(stream));
}

}  // namespace

extern "C" {

int vf_qkv_pack(const void *src, const int64_t src_strides[4], int64_t T, int64_t H,
                int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return pack4(src, src_strides, T, H, D, P, C, 0, C, dst, stream);
}

int vf_qkv_pack_chunks(const void *src, const int64_t src_strides[4], int64_t T, int64_t H,
                       int64_t D, int64_t P, int64_t C, int64_t c_begin, int64_t c_count,
                       void *dst, vf_stream_t stream) {
    return pack4(src, src_strides, T, H, D, P, C, c_begin, c_count, dst, stream);
}

int vf_qkv_pack3(const void *q, const void *k, const void *v, const int64_t qkv_strides[3],
                 int64_t T, int64_t H, int64_t D, int64_t P, int64_t C, int64_t c_begin,
                 int64_t c_count, void *dst, vf_stream_t stream) {
    if (qkv_strides == nullptr) return VF_ERR_ARG;
    return pack_common(q, k, v, qkv_strides, T, H, D, P, C, c_begin, c_count, dst, stream);
}

int vf_attn_split(const void *src, const int64_t src_strides[3], int64_t T, int64_t H,
                  int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return split_common(src, src_strides, T, H, D, P, C, 0, C, dst, stream);
}

int vf_attn_split_chunks(const void *src, const int64_t src_strides[3], int64_t T,
                         int64_t H, int64_t D, int64_t P, int64_t C, int64_t c_begin,
                         int64_t c_count, void *dst, vf_stream_t stream) {
    return split_common(src, src_strides, T, H, D, P, C, c_begin, c_count, dst, stream);
}

int vf_head_merge(const void *src, const int64_t dst_strides[3], int64_t T, int64_t H,
                  int64_t D, int64_t P, int64_t C, void *dst, vf_stream_t stream) {
    return merge_common(src, dst_strides, T, H, D, P, C, 0, C, dst, stream);
}

int vf_head_merge_chunks(const void *src, const int64_t dst_strides[3], int64_t T,
                         int64_t H, int64_t D, int64_t P, int64_t C, int64_t c_begin,
                         int64_t c_count, void *dst, vf_stream_t stream) {
    return merge_common(src, dst_strides, T, H, D, P, C, c_begin, c_count, dst, stream);
}

int vf_qkv_unpack(const void *recv, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                  void *q, void *k, void *v, const int64_t out_strides[3],
                  vf_stream_t stream) {
    return unpack_common(recv, T, H, D, P, C, 0, C, q, k, v, out_strides, stream);
}

int vf_qkv_unpack_chunks(const void *recv, int64_t T, int64_t H, int64_t D, int64_t P,
                         int64_t C, int64_t c_begin, int64_t c_count, void *q, void *k,
                         void *v, const int64_t out_strides[3], vf_stream_t stream) {
    return unpack_common(recv, T, H, D, P, C, c_begin, c_count, q, k, v, out_strides, stream);
}

int64_t vf_packed_elems(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C) {
    const Shape s{op, T, H, D, P, C};
    const int rc = check_shape(s);
    return rc != VF_OK ? rc : packed_elems(s);
}

int64_t vf_piece_table_ex(int op, int order, int64_t T, int64_t H, int64_t D, int64_t P,
                          int64_t C, int64_t *tok_start, int64_t *tok_len,
                          int64_t *packed_off, int64_t cap) {
    const Shape s{op, T, H, D, P, C};
    const int rc = check_shape(s);
    if (rc != VF_OK) return rc;
    if (order != VF_ORDER_CHUNK_MAJOR && order != VF_ORDER_SLOT_MAJOR) return VF_ERR_ARG;
    if (cap < P * C) return VF_ERR_CAPACITY;
    if (!tok_start || !tok_len || !packed_off) return VF_ERR_ARG;
    const std::vector<Entry> t = piece_table(s, order);
    for (size_t i = 0; i < t.size(); ++i) {
        tok_start[i] = t[i].tok_start;
        tok_len[i] = t[i].tok_len;
        packed_off[i] = t[i].packed_off;
    }
    return int64_t(t.size());
}

int64_t vf_piece_table(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                       int64_t *tok_start, int64_t *tok_len, int64_t *packed_off,
                       int64_t cap) {
    return vf_piece_table_ex(op, VF_ORDER_CHUNK_MAJOR, T, H, D, P, C, tok_start, tok_len,
                             packed_off, cap);
}

int vf_relayout_q(const vf_relayout_desc *d, int format, float *scales, vf_stream_t stream) {
    if (d == nullptr || (format != VF_FORMAT_INT8 && format != VF_FORMAT_E4M3))
        return VF_ERR_ARG;
    return relayout_desc(d, format, scales, stream);
}

int vf_relayout(const vf_relayout_desc *d, vf_stream_t stream) {
    if (d == nullptr) return VF_ERR_ARG;
    return relayout_desc(d, 0, nullptr, stream);
}

int vf_qkv_pack_int8(const void *src, const int64_t src_strides[4], int64_t T, int64_t H,
                     int64_t D, int64_t P, int64_t C, void *codes, float *scales,
                     vf_stream_t stream) {
    return pack4(src, src_strides, T, H, D, P, C, 0, C, codes, stream, VF_FORMAT_INT8, scales);
}

int vf_qkv_unpack_int8(const void *codes, const float *scales, int64_t T, int64_t H, int64_t D,
                       int64_t P, int64_t C, void *q, void *k, void *v,
                       const int64_t out_strides[3], vf_stream_t stream) {
    return unpack_common(codes, T, H, D, P, C, 0, C, q, k, v, out_strides, stream,
                         VF_FORMAT_INT8, scales);
}

int vf_attn_split_fp8(const void *src, const int64_t src_strides[3], int64_t T, int64_t H,
                      int64_t D, int64_t P, int64_t C, void *codes, float *scales,
                      vf_stream_t stream) {
    return split_common(src, src_strides, T, H, D, P, C, 0, C, codes, stream, VF_FORMAT_E4M3,
                        scales);
}

int vf_head_merge_fp8(const void *codes, const float *scales, const int64_t dst_strides[3],
                      int64_t T, int64_t H, int64_t D, int64_t P, int64_t C, void *dst,
                      vf_stream_t stream) {
    return merge_common(codes, dst_strides, T, H, D, P, C, 0, C, dst, stream, VF_FORMAT_E4M3,
                        scales);
}

int64_t vf_scale_count(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C) {
    const Shape s{op, T, H, D, P, C};
    const int rc = check_shape(s);
    if (rc != VF_OK) return rc;
    return D == 0 ? 0 : packed_elems(s) / D;
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
