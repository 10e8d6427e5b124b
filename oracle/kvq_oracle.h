/*
 * kvq_oracle.h -- plain, slow, single-threaded CPU oracle of the DeepSeek-V4
 * KV-cache write path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page title, section):
 *  [P1] "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
 *       (sglang#39123), sections 1 kv_layout.cuh, 2 c1/c2, 4 dequant_k_cache.py,
 *       "Why is this good" 1 (footprint) and the store-latency table.
 *  [P2] "[sglang] Hoist DSv4 draft-extend SWA write locs" (sglang#34890),
 *       sections 1 (hoisting) and 2 (eager mode).
 *  [P3] "[vLLM] DeepSeek V4 Sparse FP8 Compressor kernel" (vllm#44161),
 *       sections 2 (online softmax), 3 (RoPE, FP8 scale absmax).
 *  [OCP] OCP 8-bit Floating Point spec (E4M3) and OCP Microscaling (MX) v1.0
 *       (E8M0 shared scale, E2M1 elements) -- the format definitions.
 *
 * Parity status per function is stated in the .c file header.
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OR_D 512          /* head dim */
#define OR_ROPE_D 64      /* rope dims = last 64 */
#define OR_BLOCK 32       /* values per quant block */
#define OR_NBLK 16        /* blocks per token */

enum { OR_V41 = 1, OR_FP4 = 2 };
enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_ROPE = 1, OR_NORM = 2 };

/* status: 0 ok, 1 invalid argument, 3 capacity, 5 index out of range */
enum { OR_OK = 0, OR_EINVAL = 1, OR_ECAP = 3, OR_ERANGE = 5 };

/* ---- scalar formats ---- */
uint8_t or_e4m3_encode(float x);
double or_e4m3_decode(uint8_t c);
uint8_t or_e2m1_encode(float x);
double or_e2m1_decode(uint8_t nib);
uint16_t or_bf16_bits(float x);
float or_bf16_round(float x);
float or_bf16_to_f32(uint16_t b);
void or_e4m3_encode_n(const float *x, uint8_t *c, int64_t n);
void or_e4m3_decode_n(const uint8_t *c, double *v, int64_t n);
void or_e2m1_encode_n(const float *x, uint8_t *c, int64_t n);
void or_e2m1_decode_n(const uint8_t *c, double *v, int64_t n);
void or_bf16_bits_n(const float *x, uint16_t *b, int64_t n);

/* ---- per-token building blocks ---- */
size_t or_bytes_per_token(int layout);
size_t or_code_bytes(int layout);
size_t or_scale_bytes(int layout);
size_t or_page_bytes(int layout, int page_bits);

void or_encode_v41(const float *y, uint8_t *codes, uint8_t *scales);
void or_encode_fp4(const float *y, uint8_t *codes, uint8_t *scales);
void or_rmsnorm(float *y, const float *w, float eps);
void or_rope(float *y, const float *cs_row);
void or_pool(const float *v, const float *s, int r, float *out);

/* ---- whole calls (same meaning as the library's entry points) ---- */
int or_store(int layout, int page_bits, unsigned flags,
             const void *x, int x_dtype, int64_t n, int64_t x_row_stride,
             const int64_t *loc, const float *norm_weight, float eps,
             const float *cos_sin, int64_t cos_sin_rows, const int32_t *pos,
             uint8_t *pool, int64_t pool_slots);

int or_compress(int layout, int page_bits, int ratio, unsigned flags,
                const float *values, const float *scores, int64_t n_groups,
                const float *cos_sin, int64_t cos_sin_rows,
                const int32_t *group_pos, const int64_t *loc,
                uint8_t *pool, int64_t pool_slots);

int or_dequant(int layout, int page_bits, const uint8_t *pool, int64_t pool_pages,
               const int32_t *page_table, int64_t n_tokens,
               uint16_t *out_bf16, int64_t out_row_stride);

int or_dequant_slots(int layout, int page_bits, const uint8_t *pool, int64_t pool_slots,
                     const int64_t *slots, int64_t n, uint16_t *out_bf16, int64_t out_row_stride);

int or_translate(const int64_t *loc, int64_t n, const int32_t *full_to_swa,
                 int64_t full_slots, int32_t *out, int64_t capacity);

/* the bytes one token occupies (codes then scale row), no pool */
int or_token_bytes(int layout, unsigned flags, const void *x, int x_dtype,
                   const float *norm_weight, float eps, const float *cs_row,
                   uint8_t *codes, uint8_t *scales);
int or_group_bytes(int layout, int ratio, unsigned flags, const float *values,
                   const float *scores, const float *cs_row,
                   uint8_t *codes, uint8_t *scales);

/* the fp32 values a token is quantised from (after pool/norm/rope/bf16) */
int or_token_prequant(unsigned flags, const void *x, int x_dtype,
                      const float *norm_weight, float eps, const float *cs_row,
                      float *y);
int or_group_prequant(int ratio, unsigned flags, const float *values,
                      const float *scores, const float *cs_row, float *y);

#ifdef __cplusplus
}
#endif
#endif
