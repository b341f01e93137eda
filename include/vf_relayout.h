/*
 * vf_relayout.h -- C ABI of libvf_relayout.so: exact, direct,
 * destination-major relayouts around sequence-head (Ulysses-style)
 * attention, as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Source of the operations: "Sol-Engine alignment on SM86 and SM89", section
 * "What is enabled" (with its Chinese twin "SM86 与 SM89 上的 Sol-Engine
 * 对齐", section "当前启用的优化").  The two-device sequence-head path packs
 * QKV and merges the returned attention heads with direct relayouts: each
 * reads its source through the source strides and writes destination-major
 * storage once, in place of stack/permute/contiguous or
 * cat/permute/contiguous materialisations, keeping the BF16 values and the
 * exchange's wire format.  The same table lists the attention-result split.
 * "速度、显存与质量" (speed, memory and quality), section "剖析单次去噪请求",
 * orders them on the compute stream: QKV pack -> exchange -> QKV unpack ->
 * Flash-SDPA -> attention-result pack (the split) -> exchange -> final unpack
 * (the merge).
 *
 * The pages give no index formula; this library fixes one reading:
 *   Hp = H / P heads per destination slot (H % P == 0 for the pack, the
 *   merge and the unpack).
 *   Chunk partition of n tokens into C overlap chunks: quota Q(n) =
 *   ceil(n / C); chunk c covers tokens [min(n, c*Q), min(n, (c+1)*Q)), so the
 *   last non-empty chunk may be short and trailing chunks may be empty.
 *   Packed storage is chunk blocks in order, each destination-major: block
 *   (c, p) for c = 0..C-1 (outer), p = 0..P-1 (inner), no gaps, no padding.
 *   vf_relayout can also place the same blocks p outer (vf_order).
 *
 * Elements are 16-bit (BF16) and are moved as raw bit patterns (the opt-in
 * lossy transport at the end of this file quantises instead): NaN payloads,
 * -0 and denormals arrive unchanged.  Strides are in ELEMENTS, int64, and
 * must be non-negative.  All offsets are computed in 64-bit arithmetic.
 *
 * Ownership and concurrency: the caller owns every buffer.  The library
 * allocates no memory, keeps no global state, never synchronises, and is
 * safe to call from several host threads.  Work is enqueued on `stream`
 * (NULL = the legacy default stream) of the current device; every pointer
 * must be accessible from that device: device memory of that device, managed
 * memory, or page-locked host memory mapped at the same address (the kernels
 * then read or write it directly over the host link).  The call returns once
 * the kernels are enqueued.
 *
 * Errors: every function returns VF_OK (0) or a negative vf_status.  All
 * argument checks run on the host before anything is enqueued, so a
 * rejected call leaves dst untouched.  A call whose element count is zero
 * (T, H or D equal to 0) returns VF_OK without touching the GPU.
 */
#ifndef VF_RELAYOUT_H
#define VF_RELAYOUT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t and CUstream; declared here so that C callers
 * need no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *vf_stream_t;

typedef enum vf_status {
    VF_OK = 0,
    /* NULL pointer with a non-empty tensor, negative dimension or stride,
     * P < 1, C < 1, P * C > 2^20, H % P != 0 (pack, merge, unpack),
     * T, H or D > 2^30, NULL strides for the pack or the split, a chunk range outside
     * [0, C], a pointer that is not 2-byte aligned, a written view that
     * overlaps itself, an unknown op or order, or a pointer the current
     * device cannot access (pageable host memory unknown to CUDA, another
     * GPU's memory). */
    VF_ERR_ARG = -1,
    /* An element count, offset or byte extent does not fit in int64. */
    VF_ERR_OVERFLOW = -2,
    /* The destination's byte range overlaps the bytes the source view
     * addresses (the relayouts are not in-place), or two written views
     * overlap each other (unpack). */
    VF_ERR_ALIAS = -3,
    /* The CUDA runtime reported an error while querying a pointer or
     * enqueueing a kernel (cudaGetLastError after the launch). */
    VF_ERR_CUDA = -4,
    /* cap is smaller than the number of entries to write. */
    VF_ERR_CAPACITY = -5
} vf_status;

typedef enum vf_op {
    VF_OP_QKV_PACK = 0,
    VF_OP_ATTN_SPLIT = 1,
    VF_OP_HEAD_MERGE = 2,
    VF_OP_QKV_UNPACK = 3
} vf_op;

/* Order of the (c, p) blocks in packed storage.  Chunk-major is the
 * four-chunk overlap layout of the pages (each chunk's exchange input is one
 * contiguous P-slot slab) and the order of every entry point except
 * vf_relayout.  Slot-major keeps all chunks of one destination together
 * (one contiguous span per destination for a single, unchunked exchange). */
typedef enum vf_order {
    VF_ORDER_CHUNK_MAJOR = 0,   /* [c][p] */
    VF_ORDER_SLOT_MAJOR = 1     /* [p][c] */
} vf_order;

/*
 * QKV destination pack.  ("Sol-Engine alignment on SM86 and SM89", "What is
 * enabled": QKV destination pack.  The source is the output of the merged
 * QKV projection, a single wide GEMM whose result is viewed as q, k and v:
 * table "Upstream gap and disposition", row "Merged QKV projection".)
 *
 * src:         16-bit elements of a logical [T][3][H][D] view (token, q/k/v,
 *              head, d); src_strides[4] = its element strides in that order.
 * dst:         3*T*H*D contiguous elements, written once.  Block (c, p) is
 *              head group p of chunk c's tokens as three consecutive slabs
 *              s = q, k, v, each [L_c][Hp][D]:
 *                dst[off(c,p) + ((s*L_c + tc)*Hp + hh)*D + d]
 *                  = src[t][s][p*Hp + hh][d],  t = first token of c + tc.
 * Requires H % P == 0.
 */
int vf_qkv_pack(const void *src, const int64_t src_strides[4],
                int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                void *dst, vf_stream_t stream);

/*
 * Attention-result split.  ("Sol-Engine alignment on SM86 and SM89", "What is
 * enabled": attention result split; "速度、显存与质量", "剖析单次去噪请求":
 * the attention-result pack before the outbound exchange.)
 *
 * src:         16-bit elements of the rank-local attention output, a logical
 *              [T][H][D] view (T tokens attended, H heads held);
 *              src_strides[3] = its element strides (token, head, d), e.g.
 *              (D, T*D, 1) for a head-major [H][T][D] buffer.
 * dst:         T*H*D contiguous elements, written once.  Tokens are cut into
 *              P destination shards with quota ceil(T/P); shard p (n_p
 *              tokens) into C chunks with quota ceil(n_p/C).  Block (c, p)
 *              is chunk c of shard p as [L][H][D].
 * No constraint between H and P.
 */
int vf_attn_split(const void *src, const int64_t src_strides[3],
                  int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                  void *dst, vf_stream_t stream);

/*
 * Returned-head merge.  ("Sol-Engine alignment on SM86 and SM89", "What is
 * enabled": returned-head merge, replacing cat/permute/contiguous;
 * "速度、显存与质量", "剖析单次去噪请求": the final unpack.)
 *
 * src:         T*H*D contiguous elements of received destination-major
 *              storage: block (c, p) is chunk c's tokens for head group p,
 *              [L_c][Hp][D].  (The packed side is always this canonical
 *              layout: with a short tail chunk it is not a uniformly
 *              strided tensor.)
 * dst:         16-bit elements of a logical [T][H][D] view, written once;
 *              dst_strides[3] = its element strides (token, head, d), or
 *              NULL for contiguous (H*D, D, 1).  The view must not overlap
 *              itself (checked: sorted by stride, each stride must exceed
 *              the span of the smaller ones).
 *                dst[t][p*Hp + hh][d] = src[off(c,p) + (tc*Hp + hh)*D + d].
 * Requires H % P == 0.
 */
int vf_head_merge(const void *src, const int64_t dst_strides[3],
                  int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                  void *dst, vf_stream_t stream);

/*
 * Receive-side QKV unpack.  ("速度、显存与质量", section "剖析单次去噪请求": the
 * QKV unpack between the inbound exchange and Flash-SDPA; it inverts the
 * pack of "Sol-Engine alignment on SM86 and SM89", "What is enabled", across
 * the all-to-all.)
 *
 * Shapes are the global ones: T tokens over all ranks, H heads in total,
 * P ranks; this rank owns one head group of Hp = H/P heads.  Source rank r
 * owned token shard r (quota ceil(T/P)) and packed it with chunk quota
 * ceil(n_r/C).
 * recv:        3*T*Hp*D contiguous elements as received: for each chunk c,
 *              for each source rank r, that rank's pack block for this head
 *              group, [s][L][Hp][D] (s = q, k, v).
 * q, k, v:     three [T][Hp][D] views written once, in global token order,
 *              all with the element strides out_strides[3] (token, head, d),
 *              or NULL for contiguous (Hp*D, D, 1).  Each view must not
 *              overlap itself, the others or recv.
 * Requires H % P == 0.
 */
int vf_qkv_unpack(const void *recv, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                  void *q, void *k, void *v, const int64_t out_strides[3],
                  vf_stream_t stream);

/*
 * Chunk-range variants for the overlap pipeline ("Sol-Engine alignment on
 * SM86 and SM89", "What is enabled": Vflash's four-chunk overlap layout, in
 * which chunk c's exchange overlaps the relayout of the next chunk).  Each
 * takes the same arguments as its full form plus chunks
 * [c_begin, c_begin + c_count) (0 <= c_begin, c_count >= 0,
 * c_begin + c_count <= C) and moves only those chunks' blocks: the packed
 * buffer is always the full one and block offsets are those of
 * vf_piece_table; the strided side is only touched at the chunks' tokens.
 * c_count == 0 returns VF_OK without touching the GPU.
 */
int vf_qkv_pack_chunks(const void *src, const int64_t src_strides[4],
                       int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                       int64_t c_begin, int64_t c_count, void *dst, vf_stream_t stream);
int vf_attn_split_chunks(const void *src, const int64_t src_strides[3],
                         int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                         int64_t c_begin, int64_t c_count, void *dst, vf_stream_t stream);
int vf_head_merge_chunks(const void *src, const int64_t dst_strides[3],
                         int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                         int64_t c_begin, int64_t c_count, void *dst, vf_stream_t stream);
int vf_qkv_unpack_chunks(const void *recv, int64_t T, int64_t H, int64_t D, int64_t P,
                         int64_t C, int64_t c_begin, int64_t c_count,
                         void *q, void *k, void *v, const int64_t out_strides[3],
                         vf_stream_t stream);

/*
 * QKV destination pack from three separate Q, K, V views (projections that
 * were not fused into one GEMM; "Sol-Engine alignment on SM86 and SM89",
 * table "Upstream gap and disposition", row "Merged QKV projection", is the
 * fused case).  q, k, v: [T][H][D] views sharing the element strides
 * qkv_strides[3] (token, head, d); they may overlap each other (read only).
 * Output, chunk range and rules as vf_qkv_pack_chunks: the result equals
 * vf_qkv_pack of the [T][3][H][D] view whose slabs are q, k, v.
 */
int vf_qkv_pack3(const void *q, const void *k, const void *v, const int64_t qkv_strides[3],
                 int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                 int64_t c_begin, int64_t c_count, void *dst, vf_stream_t stream);

/*
 * General form of every operation above, with the block order as a field.
 * The named entry points are this call with order = VF_ORDER_CHUNK_MAJOR.
 *
 * op, order:   vf_op, vf_order.
 * T..C:        as for the named entry points (the unpack takes the global T
 *              and H, as vf_qkv_unpack does).
 * c_begin, c_count: chunks to move, (0, C) for all.
 * packed:      the packed storage (written by the pack and the split, read
 *              by the merge and the unpack), in `order`.
 * strided:     the strided-side views, all with the element strides
 *              `strides` (token, head, d): pack -> q, k, v [T][H][D] (read;
 *              for a fused [T][3][H][D] view pass its three slab bases);
 *              split -> [0] = [T][H][D] (read); merge -> [0] = [T][H][D]
 *              (written); unpack -> q, k, v [T][H/P][D] (written).  Entries
 *              past the op's slab count are ignored.
 * Errors as for the named entry points; an unknown order is VF_ERR_ARG.
 */
typedef struct vf_relayout_desc {
    int32_t op;
    int32_t order;
    int64_t T, H, D, P, C;
    int64_t c_begin, c_count;
    void *packed;
    void *strided[3];
    int64_t strides[3];
} vf_relayout_desc;

int vf_relayout(const vf_relayout_desc *desc, vf_stream_t stream);

/*
 * Number of elements of the packed side of `op` (3*T*H*D for the pack,
 * T*H*D for the split and the merge, 3*T*(H/P)*D for the unpack), or a
 * negative vf_status on bad arguments or overflow.  Pure host function.
 */
int64_t vf_packed_elems(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C);

/*
 * The piece table of `op`: entry c*P + p describes block (c, p): the first
 * token (tok_start; for the split and the unpack, counted in the strided
 * view's token numbering, so shard p's chunk c), the token count (tok_len)
 * and the element offset of the block in packed storage (packed_off) for
 * chunk-major storage.  For the unpack, p is the source rank.  Writes C*P
 * entries into each caller-owned array of capacity `cap` and returns C*P, or
 * a negative vf_status (VF_ERR_CAPACITY when cap < C*P).  Pure host function.
 */
int64_t vf_piece_table(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                       int64_t *tok_start, int64_t *tok_len, int64_t *packed_off,
                       int64_t cap);

/* vf_piece_table with the block order given: entries are still indexed
 * c*P + p; packed_off places the blocks in `order` (vf_order). */
int64_t vf_piece_table_ex(int op, int order, int64_t T, int64_t H, int64_t D, int64_t P,
                          int64_t C, int64_t *tok_start, int64_t *tok_len,
                          int64_t *packed_off, int64_t cap);

/*
 * Opt-in lossy transport.  ("Sol-Engine alignment on SM86 and SM89", table
 * "Upstream gap and disposition", row "INT8 QKV and FP8 output transport": a
 * profile that moves Q/K/V as INT8 and the attention output as FP8 across the
 * exchange.  The pages keep it out of the exact default and give no format;
 * nothing above changes when these calls are not used.)
 *
 * Format, per head row (the D elements of one token and one head), all in
 * float32 with one rounding per step, to nearest even:
 *   amax = max |x|.  If amax < 2^-96: scale = 0 and every code is 0.
 *   Else, top = 127 (VF_FORMAT_INT8) or 448 (VF_FORMAT_E4M3):
 *     inv = top / amax;  scale = amax / top;  q = x * inv;
 *     INT8: code = clamp(round(q), -127, 127), an int8 byte;
 *     E4M3: code = q as OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7,
 *           3 mantissa bits), saturating at +-448, never NaN.
 *   Receive side: y = bfloat16(value(code) * scale).
 * The 16-bit elements are BF16 values on both sides (the quantisers read
 * them as BF16, the dequantisers write BF16).
 * Non-finite values: a head row holding a NaN or an infinity cannot be
 * scaled, so it is sent as a lost row: scale = the float32 quiet NaN
 * 0x7FC00000 and every code 0; no other row is affected.  The receive side
 * writes the BF16 quiet NaN 0x7FC0 into every element of a row whose scale
 * is not finite (NaN or an infinity).  The E4M3 codes 0x7F and 0xFF (the
 * format's NaN) are never written; a receive side given one writes a NaN
 * there (payload unspecified).  A finite product that overflows float32
 * arrives as an infinity.
 *
 * Storage: codes: one byte per element, in exactly the element layout of
 * the exact op (vf_packed_elems bytes; block offsets are vf_piece_table's
 * packed_off in bytes).  scales: one float per head row of that layout, in
 * the same order (vf_scale_count floats; row i covers code bytes
 * [i*D, (i+1)*D)); 4-byte aligned.  Codes and scales must not overlap each
 * other or the strided views.  Codes may be at any address; the kernels use
 * 8-element vectors when D % 8 == 0, the strided side is 16-byte aligned
 * with d contiguous, and codes are 8-byte aligned.
 * Errors as for the exact calls, plus: an unknown format, NULL scales (when
 * anything is moved) or scales not 4-byte aligned -> VF_ERR_ARG; scales that
 * overlap the codes or a strided view -> VF_ERR_ALIAS; tokens x heads of any
 * one (chunk, destination) block at or above 2^31 -> VF_ERR_ARG.
 */
typedef enum vf_format {
    VF_FORMAT_INT8 = 1,
    VF_FORMAT_E4M3 = 2
} vf_format;

/* vf_relayout with quantised packed storage: desc->packed holds the codes
 * (written by the pack and the split, read by the merge and the unpack) and
 * `scales` the per-row scales (written or read likewise).  Any op, order and
 * chunk range; an unknown format is VF_ERR_ARG. */
int vf_relayout_q(const vf_relayout_desc *desc, int format, float *scales,
                  vf_stream_t stream);

/* The pairings the pages name: INT8 for the QKV pack and its receive-side
 * unpack, E4M3 for the attention-result split and the returned-head merge.
 * Arguments as for the exact entry points, with the 16-bit packed buffer
 * replaced by codes + scales. */
int vf_qkv_pack_int8(const void *src, const int64_t src_strides[4],
                     int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                     void *codes, float *scales, vf_stream_t stream);
int vf_qkv_unpack_int8(const void *codes, const float *scales,
                       int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                       void *q, void *k, void *v, const int64_t out_strides[3],
                       vf_stream_t stream);
int vf_attn_split_fp8(const void *src, const int64_t src_strides[3],
                      int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                      void *codes, float *scales, vf_stream_t stream);
int vf_head_merge_fp8(const void *codes, const float *scales, const int64_t dst_strides[3],
                      int64_t T, int64_t H, int64_t D, int64_t P, int64_t C,
                      void *dst, vf_stream_t stream);

/* Number of scales of `op`'s packed side: vf_packed_elems / D (0 when D is
 * 0), or a negative vf_status.  Pure host function. */
int64_t vf_scale_count(int op, int64_t T, int64_t H, int64_t D, int64_t P, int64_t C);

/* Static, NUL-terminated description of a vf_status value. */
const char *vf_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* VF_RELAYOUT_H */
