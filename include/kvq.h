/*
 * kvq.h -- C ABI of the GB300 (sm_103a) KV-cache write path for
 * DeepSeek-V4-style serving: block quantisation of new K rows into a paged
 * pool (optionally pooled by a ratio-r softmax compressor, RMS-normalised and
 * rotated), the once-per-step full->SWA slot translation, and the paged
 * dequant back to a bf16 workspace.
 *
 * Sources (page title, section):
 *  [P1] "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
 *       (sglang#39123): section 1 kv_layout.cuh (V41 / V41_FP4 layouts,
 *       PagedKV, store_row), section 2 c1.cuh/c2.cuh (ratio compressors,
 *       kv_page_bytes), section 4 dequant_k_cache.py, the store-latency
 *       table (store, store + RoPE, fused K norm + RoPE, c1, c2).
 *  [P2] "[sglang] Hoist DSv4 draft-extend SWA write locs" (sglang#34890):
 *       section 1 (translate once per step into a preallocated int32
 *       buffer, zero the tail, no buffer when n exceeds it), section 2.
 *  [P3] "[vLLM] DeepSeek V4 Sparse FP8 Compressor kernel" (vllm#44161):
 *       section 2 (per-element online-softmax pooling), section 3 (RoPE,
 *       bf16 cast, per-32-value absmax and fp8 scale).
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    allocates nothing, frees nothing and never synchronises.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and
 *    launched with programmatic dependent launch enabled: a kernel waits for
 *    its predecessor on the stream before its first global read.
 *  - Arguments are checked on the host before anything is launched; a
 *    failing check returns a status and enqueues no work.
 *  - Problems only the device can see (an index outside its table) set bits
 *    in `*err` (when err is not NULL; atomic OR, KVQ_DEVERR_*) and skip that
 *    row or page; the caller zeroes *err and reads it after its own sync.
 *    Kernels never trap.
 *  - Row data are 512 dims ("head dim"); RoPE rotates the last 64 dims
 *    (448..511) as interleaved pairs (448+2i, 449+2i); a quant block is 32
 *    consecutive dims, 16 blocks per token.
 *  - Slots in one call must be distinct (scatter targets do not overlap);
 *    with repeated slots the surviving row is unspecified.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* = cudaStream_t */

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or enum */
    KVQ_ERR_UNSUPPORTED = 2, /* valid request with no compiled instance    */
    KVQ_ERR_CAPACITY = 3,    /* n > out_capacity in kvq_translate_loc      */
    KVQ_ERR_LAUNCH = 4       /* the CUDA launch itself failed              */
} kvq_status;

/* [P1] section 1.  V41: 512 e4m3 codes + 16 ue8m0 scales = 528 B/token.
 * V41_FP4: 256 B of e2m1 codes (two per byte, even dim in the low nibble)
 * + 16 e4m3 scales + 16 B of zero padding = 288 B/token. */
typedef enum { KVQ_LAYOUT_V41 = 1, KVQ_LAYOUT_V41_FP4 = 2 } kvq_layout;
typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1 } kvq_dtype;
typedef enum { KVQ_I32 = 0, KVQ_I64 = 1 } kvq_index_dtype;
enum { KVQ_FLAG_ROPE = 1, KVQ_FLAG_NORM = 2 };

/* bits of the device error word */
enum {
    KVQ_DEVERR_SLOT = 1,  /* a slot outside [0, pool_slots) (row skipped)        */
    KVQ_DEVERR_POS = 2,   /* a RoPE position outside [0, cos_sin_rows) (skipped) */
    KVQ_DEVERR_PAGE = 4,  /* a page-table entry outside [0, pool_pages) (skipped)*/
    KVQ_DEVERR_LOC = 8,   /* a full slot outside the translation table (-> -1)   */
                          /* (bit 16 is unused: no kernel has a bounded wait)    */
    KVQ_DEVERR_STATE = 32    /* a request index outside [0, n_state) or a count   */
                             /* outside [0, ratio): that request is skipped       */
};

/* Bytes one token occupies: 528 (V41) or 288 (V41_FP4); 0 for a bad layout.
 * [P1] section 1 and "Why is this good" 1. */
size_t kvq_bytes_per_token(kvq_layout layout);

/* Bytes of one page of 2^page_bits tokens: all code rows, then all scale
 * rows ([P1] section 2, kv_page_bytes).  0 for a bad layout / page_bits. */
size_t kvq_page_bytes(kvq_layout layout, int page_bits);

/* 1 if page_bits has a compiled instance (the layout's page size is a
 * compile-time constant of every kernel), else 0. */
int kvq_page_bits_supported(int page_bits);

/* Full -> SWA slot translation, hoisted to once per step ([P2] sections 1-2).
 *   full_loc     [n] int32 or int64 (loc_dtype): slots of the full pool.
 *   full_to_swa  [full_slots] int32: the SWA slot of each full slot.
 *   out          [out_capacity] int32: out[i] = full_to_swa[full_loc[i]] for
 *                i < n, and out[n:out_capacity] = 0.
 * n > out_capacity returns KVQ_ERR_CAPACITY and enqueues nothing (the
 * caller then translates into a buffer of its own, as the eager fallback
 * does).  A full_loc[i] outside [0, full_slots) writes -1 there and sets
 * KVQ_DEVERR_LOC. */
kvq_status kvq_translate_loc(const void *full_loc, kvq_index_dtype loc_dtype, int64_t n,
                             const int32_t *full_to_swa, int64_t full_slots,
                             int32_t *out, int64_t out_capacity,
                             int32_t *err, struct CUstream_st *stream);

/* Quantise n new rows and scatter them into the paged pool ([P1] section 1
 * store_row, the store / store + RoPE / fused K norm + RoPE kernels).
 *   x            [n, x_row_stride] fp32 or bf16 (x_dtype); the first 512
 *                elements of each row are used; 16-byte aligned rows.
 *   loc          [n] int32 or int64: destination slot of each row.
 *   flags        KVQ_FLAG_NORM: y = x * rsqrt(mean(x^2) + eps) * norm_weight
 *                (norm_weight [512] fp32); KVQ_FLAG_ROPE: rotate dims
 *                448..511 by row pos[i] of cos_sin ([cos_sin_rows, 64] fp32,
 *                32 cosines then 32 sines).  Norm runs before RoPE, all in
 *                fp32, and the result is rounded to bf16 before quantising;
 *                without flags the input is quantised as given.
 *   pool         [pool_slots / 2^page_bits pages] of kvq_page_bytes each;
 *                pool_slots a multiple of 2^page_bits.
 * V41: per 32 dims, scale byte = (amax exponent field - 8) clamped at 0,
 * code = e4m3_satfinite(x * 2^(127 - byte)).  V41_FP4: scale =
 * e4m3(amax / 6), code = e2m1_satfinite(x * rcp(scale)) (a zero scale gives
 * zero codes). */
kvq_status kvq_store(kvq_layout layout, int page_bits, unsigned flags,
                     const void *x, kvq_dtype x_dtype, int64_t n, int64_t x_row_stride,
                     const void *loc, kvq_index_dtype loc_dtype,
                     const float *norm_weight, float eps,
                     const float *cos_sin, int64_t cos_sin_rows, const int32_t *pos,
                     uint8_t *pool, int64_t pool_slots,
                     int32_t *err, struct CUstream_st *stream);

/* Ratio-r softmax compressor + store ([P1] section 2 c1/c2; [P3] sections
 * 2-3, C4A / C128A).  Group g pools rows g*ratio .. g*ratio+ratio-1:
 *   out[d] = sum_t softmax_t(scores[t, d]) * values[t, d]   (per dim d),
 * then (KVQ_FLAG_ROPE) rotates dims 448..511 by row group_pos[g] of cos_sin,
 * rounds to bf16 and quantises into slot loc[g] as kvq_store does.
 *   values, scores  [n_groups * ratio, 512] fp32, contiguous, 16-B aligned.
 *   loc             [n_groups] int32 (already translated slots).
 *   ratio           1, 2, 4 or 128.  KVQ_FLAG_NORM is not accepted. */
kvq_status kvq_compress(kvq_layout layout, int page_bits, int ratio, unsigned flags,
                        const float *values, const float *scores, int64_t n_groups,
                        const float *cos_sin, int64_t cos_sin_rows, const int32_t *group_pos,
                        const int32_t *loc, uint8_t *pool, int64_t pool_slots,
                        int32_t *err, struct CUstream_st *stream);

/* Decode-time ratio-r compressor ([P1] section 2, flash_c1/c2_decode_kernel;
 * [P3] section 2, the online max / sum softmax): each call brings ONE new row
 * per request, and the softmax pool of the request's unfinished group is
 * carried between calls as online state.
 *   values, scores  [n, 512] fp32: request i's new row.
 *   state           [n_state, 3, 512] fp32, caller-owned, per request slot:
 *                   running max m, sum of exp(s - m) and sum of
 *                   exp(s - m) * v of the rows seen so far, per dim.
 *   count           [n_state] int32: rows of the open group (0 .. ratio-1);
 *                   start at 0 with any state contents.
 *   req             [n] int32: state slot of request i (NULL: slot i).
 * When request i's row is the group's ratio-th, the pooled row acc / sum is
 * rotated by row group_pos[i] of cos_sin (KVQ_FLAG_ROPE), rounded to bf16,
 * quantised and stored into slot loc[i] exactly as kvq_compress does, and
 * count returns to 0; otherwise only state and count change and the values
 * of loc[i] and group_pos[i] are ignored.  The kernel reads both arrays
 * before it knows the count (to overlap their latency), so they must hold n
 * readable entries on every call.  A bad request index or count sets
 * KVQ_DEVERR_STATE and skips that request.  Requests in one call must use
 * distinct state slots.  KVQ_FLAG_NORM is not accepted. */
kvq_status kvq_compress_decode(kvq_layout layout, int page_bits, int ratio, unsigned flags,
                               const float *values, const float *scores, int64_t n,
                               float *state, int32_t *count, const int32_t *req, int64_t n_state,
                               const float *cos_sin, int64_t cos_sin_rows, const int32_t *group_pos,
                               const int32_t *loc, uint8_t *pool, int64_t pool_slots,
                               int32_t *err, struct CUstream_st *stream);

/* Paged dequant to a bf16 workspace ([P1] section 4, dequant_k_cache.py).
 *   page_table  [n_tokens / 2^page_bits] int32: physical page of each
 *               logical page; n_tokens must be a multiple of 2^page_bits.
 *   out_bf16    [n_tokens, out_row_stride] bf16 (stride >= 512, rows 16-B
 *               aligned): row t = decode(page_table[t >> page_bits], row
 *               t & (2^page_bits - 1)).  V41: e4m3 * 2^(byte - 127);
 *               V41_FP4: e2m1 * e4m3 scale; both exact in bf16.
 * An entry outside [0, pool_pages) sets KVQ_DEVERR_PAGE and leaves that
 * page's rows untouched. */
kvq_status kvq_dequant(kvq_layout layout, int page_bits,
                       const uint8_t *pool, int64_t pool_pages,
                       const int32_t *page_table, int64_t n_tokens,
                       void *out_bf16, int64_t out_row_stride,
                       int32_t *err, struct CUstream_st *stream);

/* Dequant of selected tokens to bf16 rows: the consumer side of [P1] section
 * 4 (dequant_k_cache.py) restricted to the tokens a sparse attention picks
 * (the FlashMLA sparse-FP8 reader of [P3]).
 *   slots       [n] int32 or int64 (slot_dtype): pool slot of output row i.
 *   out_bf16    [n, out_row_stride] bf16 (stride >= 512, rows 16-B aligned):
 *               row i = decode(slot slots[i]), exact in bf16 as in kvq_dequant.
 * Slot -1 is padding and writes a zero row.  Any other slot outside
 * [0, pool_slots) sets KVQ_DEVERR_SLOT and leaves row i untouched. */
kvq_status kvq_dequant_slots(kvq_layout layout, int page_bits,
                             const uint8_t *pool, int64_t pool_slots,
                             const void *slots, kvq_index_dtype slot_dtype, int64_t n,
                             void *out_bf16, int64_t out_row_stride,
                             int32_t *err, struct CUstream_st *stream);

/* Human-readable name of a status. */
const char *kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
