/*
 * kvq_oracle.c -- CPU oracle of the DeepSeek-V4 KV-cache write path.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library.  It shares no code with the CUDA
 * library: the number formats below are written from the OCP definitions, the
 * steps from the pages' problem statement, one plain loop per definition.
 * Build: gcc -O2 -ffp-contract=off (no fused multiply-add anywhere, so every
 * float operation is one IEEE-754 binary32 rounding, as written).
 *
 * Pins (tests/test_oracle_*.py) per function:
 *   or_e4m3_encode/decode  pinned: torch's float8_e4m3fn cast, brute-force
 *                           nearest search over all codes, hand-worked blocks
 *   or_e2m1_encode/decode  pinned: brute-force nearest over the 8 E2M1 values,
 *                           hand-worked grid and tie blocks
 *   or_bf16_bits           pinned: torch's bfloat16 cast (ties, subnormals)
 *   or_encode_v41          pinned: hand-worked blocks (golden), error bound
 *   or_encode_fp4          pinned: hand-worked blocks (golden), error bound
 *   or_rmsnorm             pinned: constant-vector closed form, scale invariance
 *   or_rope                pinned: complex multiplication, pos-0 identity,
 *                           quarter-turn, norm preservation, angle addition
 *   or_pool                pinned: r=1 identity, equal scores = mean, dominant
 *                           score, two-row sigmoid closed form, convexity,
 *                           row-permutation and score-shift invariance
 *   or_store/or_compress   pinned: brute force on tiny pools vs an independent
 *                           address model; footprint closed forms
 *   or_dequant             pinned: dequant of hand-worked blocks, error bound,
 *                           page-table permutation brute force
 *   or_dequant_slots       pinned: equals the paged dequant's rows (identity
 *                           page table), padding and range rules
 *   or_translate           pinned: brute-force gather, zero tail, capacity rule
 */
#include "kvq_oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double that is exactly representable to the nearest
 * integer, ties to even. */
static double rne_nonneg(double q)
{
    double f = floor(q);
    double frac = q - f;
    if (frac > 0.5) return f + 1.0;
    if (frac < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Magnitude code of a sign-less minifloat with `mbits` mantissa bits and
 * exponent bias `bias`: code = (biased exponent << mbits) | mantissa, the
 * biased exponent 0 holding the subnormals.  Round to nearest, ties to even;
 * anything at or above the largest finite value `maxval` gives `maxcode`
 * (saturating conversion). */
static unsigned minifloat_encode_mag(double a, int mbits, int bias,
                                     unsigned maxcode, double maxval)
{
    if (a >= maxval) return maxcode;
    if (a == 0.0) return 0;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;               /* floor(log2 a) */
    int emin = 1 - bias;          /* exponent of the smallest normal */
    if (e < emin) e = emin;       /* subnormals use the smallest normal's step */
    double step = ldexp(1.0, e - mbits);
    double r = rne_nonneg(a / step);   /* division by a power of two: exact */
    unsigned code = ((unsigned)(e - emin) << mbits) + (unsigned)r;
    if (code > maxcode) code = maxcode;
    return code;
}

static double minifloat_decode_mag(unsigned code, int mbits, int bias)
{
    unsigned E = code >> mbits, M = code & ((1u << mbits) - 1u);
    if (E == 0) return ldexp((double)M, 1 - bias - mbits);
    return ldexp((double)((1u << mbits) + M), (int)E - bias - mbits);
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities, S.1111.111 is NaN, largest finite 448 = S.1111.110. */
uint8_t or_e4m3_encode(float x)
{
    double a = fabs((double)x);
    unsigned mag = minifloat_encode_mag(a, 3, 7, 0x7Eu, 448.0);
    return (uint8_t)((signbit(x) ? 0x80u : 0u) | mag);
}

double or_e4m3_decode(uint8_t c)
{
    unsigned mag = c & 0x7Fu;
    if (mag == 0x7Fu) return NAN;
    double v = minifloat_decode_mag(mag, 3, 7);
    return (c & 0x80u) ? -v : v;
}

/* OCP MX E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; values
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6; no NaN or infinity. */
uint8_t or_e2m1_encode(float x)
{
    double a = fabs((double)x);
    unsigned mag = minifloat_encode_mag(a, 1, 1, 0x7u, 6.0);
    return (uint8_t)((signbit(x) ? 0x8u : 0u) | mag);
}

double or_e2m1_decode(uint8_t nib)
{
    double v = minifloat_decode_mag(nib & 0x7u, 1, 1);
    return (nib & 0x8u) ? -v : v;
}

/* bfloat16 = the top 16 bits of a binary32; round to nearest even by adding
 * half of the dropped range (plus the kept LSB for ties).  Finite inputs. */
uint16_t or_bf16_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

float or_bf16_round(float x) { return or_bf16_to_f32(or_bf16_bits(x)); }

/* array forms of the scalar conversions (for the tests) */
void or_e4m3_encode_n(const float *x, uint8_t *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) c[i] = or_e4m3_encode(x[i]);
}
void or_e4m3_decode_n(const uint8_t *c, double *v, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) v[i] = or_e4m3_decode(c[i]);
}
void or_e2m1_encode_n(const float *x, uint8_t *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) c[i] = or_e2m1_encode(x[i]);
}
void or_e2m1_decode_n(const uint8_t *c, double *v, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) v[i] = or_e2m1_decode(c[i]);
}
void or_bf16_bits_n(const float *x, uint16_t *b, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) b[i] = or_bf16_bits(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Layout sizes: [P1] section 1 (V41 528 B/token, V41_FP4 288 B/token),      */
/* "Why is this good" 1 (-9.6% / -50.7% against V4's 584 B/token).           */
/* ------------------------------------------------------------------------ */

size_t or_code_bytes(int layout)
{
    return layout == OR_V41 ? 512u : layout == OR_FP4 ? 256u : 0u;
}

/* V41: 16 ue8m0 bytes.  FP4: 16 e4m3 bytes + 16 bytes of zero padding that
 * make up the stated 288 B/token. */
size_t or_scale_bytes(int layout)
{
    return layout == OR_V41 ? 16u : layout == OR_FP4 ? 32u : 0u;
}

size_t or_bytes_per_token(int layout)
{
    return or_code_bytes(layout) + or_scale_bytes(layout);
}

/* A page holds P = 2^page_bits token rows: all code rows, then all scale
 * rows ([P1] section 1, PagedKV page / row / scale-row addressing). */
size_t or_page_bytes(int layout, int page_bits)
{
    return ((size_t)1 << page_bits) * or_bytes_per_token(layout);
}

/* ------------------------------------------------------------------------ */
/* Block quantisation                                                        */
/* ------------------------------------------------------------------------ */

static float block_amax(const float *y)
{
    float amax = 0.0f;
    for (int i = 0; i < OR_BLOCK; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    return amax;
}

/* V41 ([P1] section 1): one ue8m0 scale per 32 values, its exponent taken
 * from the amax bits (no division).  OCP MX rule: shared exponent =
 * floor(log2 amax) - emax(E4M3) = floor(log2 amax) - 8, i.e. the biased byte
 * is the amax's binary32 exponent field minus 8 (clamped at 0).  Each value
 * is scaled by 2^(127 - byte) and converted to E4M3, saturating at 448. */
void or_encode_v41(const float *y, uint8_t *codes, uint8_t *scales)
{
    for (int b = 0; b < OR_NBLK; ++b) {
        const float *blk = y + b * OR_BLOCK;
        float amax = block_amax(blk);
        uint32_t bits;
        memcpy(&bits, &amax, 4);
        int e_field = (int)((bits >> 23) & 0xFFu);
        int byte = e_field - 8;
        if (byte < 0) byte = 0;
        scales[b] = (uint8_t)byte;
        float mult = ldexpf(1.0f, 127 - byte);
        for (int i = 0; i < OR_BLOCK; ++i)
            codes[b * OR_BLOCK + i] = or_e4m3_encode(blk[i] * mult);
    }
}

/* V41_FP4 ([P1] section 1): 512 E2M1 codes (two per byte, the even element in
 * the low nibble) and one E4M3 scale per 32 values.  Scale = E4M3(amax / 6)
 * so the block's largest value lands on E2M1's largest (6); codes =
 * E2M1(x * (1 / scale)) with a correctly rounded reciprocal.  A zero scale
 * gives all-zero codes.  The scale row is 16 scale bytes then 16 zero bytes. */
void or_encode_fp4(const float *y, uint8_t *codes, uint8_t *scales)
{
    for (int b = 0; b < OR_NBLK; ++b) {
        const float *blk = y + b * OR_BLOCK;
        float amax = block_amax(blk);
        uint8_t s8 = or_e4m3_encode(amax / 6.0f);
        float S = (float)or_e4m3_decode(s8);
        scales[b] = s8;
        scales[OR_NBLK + b] = 0;
        for (int j = 0; j < OR_BLOCK / 2; ++j) {
            uint8_t lo = 0, hi = 0;
            if (S != 0.0f) {
                float inv = 1.0f / S;
                lo = or_e2m1_encode(blk[2 * j] * inv);
                hi = or_e2m1_encode(blk[2 * j + 1] * inv);
            }
            codes[b * (OR_BLOCK / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Pre-quantisation math                                                     */
/* ------------------------------------------------------------------------ */

/* K RMSNorm ([P1] store-latency table, "fused K norm + RoPE"): over all 512
 * dims, eps inside the square root, weight applied after normalising.  The
 * sum of squares is taken in double and rounded once. */
void or_rmsnorm(float *y, const float *w, float eps)
{
    double acc = 0.0;
    for (int d = 0; d < OR_D; ++d) acc += (double)y[d] * (double)y[d];
    float ms = (float)acc / (float)OR_D;
    float inv = 1.0f / sqrtf(ms + eps);
    for (int d = 0; d < OR_D; ++d) y[d] = (y[d] * inv) * w[d];
}

/* RoPE on the last 64 dims ([P1] table "store + RoPE"; [P3] section 3), in
 * binary32.  Pair i rotates dims (448+2i, 449+2i) by the angle whose cosine
 * and sine are cs_row[i] and cs_row[32+i]. */
void or_rope(float *y, const float *cs_row)
{
    for (int i = 0; i < OR_ROPE_D / 2; ++i) {
        float *p = y + (OR_D - OR_ROPE_D) + 2 * i;
        float a = p[0], b = p[1];
        float c = cs_row[i], s = cs_row[OR_ROPE_D / 2 + i];
        float ac = a * c, bs = b * s, as = a * s, bc = b * c;
        p[0] = ac - bs;
        p[1] = as + bc;
    }
}

/* Per-element softmax pooling of r rows ([P1] section 2 c1/c2 compressors;
 * [P3] section 2): out[d] = sum_t softmax_t(s[t,d]) * v[t,d].  Two-pass
 * textbook form: the max in binary32, exp and both sums in double, one
 * rounding of the quotient. */
void or_pool(const float *v, const float *s, int r, float *out)
{
    for (int d = 0; d < OR_D; ++d) {
        float m = s[d];
        for (int t = 1; t < r; ++t)
            if (s[(size_t)t * OR_D + d] > m) m = s[(size_t)t * OR_D + d];
        double num = 0.0, den = 0.0;
        for (int t = 0; t < r; ++t) {
            double e = exp((double)s[(size_t)t * OR_D + d] - (double)m);
            num += e * (double)v[(size_t)t * OR_D + d];
            den += e;
        }
        out[d] = (float)(num / den);
    }
}

/* ------------------------------------------------------------------------ */
/* Token / group pipelines                                                   */
/* ------------------------------------------------------------------------ */

static void widen_row(const void *x, int x_dtype, float *y)
{
    if (x_dtype == OR_F32) {
        memcpy(y, x, OR_D * sizeof(float));
    } else {
        const uint16_t *h = (const uint16_t *)x;
        for (int d = 0; d < OR_D; ++d) y[d] = or_bf16_to_f32(h[d]);
    }
}

/* Store path: widen, optional norm, optional RoPE, and a round to bf16 after
 * any of that fp32 math ([P3] section 3 casts the rotated values to bf16);
 * an untouched input is quantised as given. */
int or_token_prequant(unsigned flags, const void *x, int x_dtype,
                      const float *norm_weight, float eps, const float *cs_row,
                      float *y)
{
    if ((flags & OR_NORM) && !norm_weight) return OR_EINVAL;
    if ((flags & OR_ROPE) && !cs_row) return OR_EINVAL;
    widen_row(x, x_dtype, y);
    if (flags & OR_NORM) or_rmsnorm(y, norm_weight, eps);
    if (flags & OR_ROPE) or_rope(y, cs_row);
    if (flags & (OR_NORM | OR_ROPE))
        for (int d = 0; d < OR_D; ++d) y[d] = or_bf16_round(y[d]);
    return OR_OK;
}

/* Compress path: pool r rows, optional RoPE, round to bf16. */
int or_group_prequant(int ratio, unsigned flags, const float *values,
                      const float *scores, const float *cs_row, float *y)
{
    if (ratio < 1) return OR_EINVAL;
    if ((flags & OR_ROPE) && !cs_row) return OR_EINVAL;
    or_pool(values, scores, ratio, y);
    if (flags & OR_ROPE) or_rope(y, cs_row);
    for (int d = 0; d < OR_D; ++d) y[d] = or_bf16_round(y[d]);
    return OR_OK;
}

static int encode_layout(int layout, const float *y, uint8_t *codes, uint8_t *scales)
{
    if (layout == OR_V41) or_encode_v41(y, codes, scales);
    else if (layout == OR_FP4) or_encode_fp4(y, codes, scales);
    else return OR_EINVAL;
    return OR_OK;
}

int or_token_bytes(int layout, unsigned flags, const void *x, int x_dtype,
                   const float *norm_weight, float eps, const float *cs_row,
                   uint8_t *codes, uint8_t *scales)
{
    float y[OR_D];
    int rc = or_token_prequant(flags, x, x_dtype, norm_weight, eps, cs_row, y);
    if (rc) return rc;
    return encode_layout(layout, y, codes, scales);
}

int or_group_bytes(int layout, int ratio, unsigned flags, const float *values,
                   const float *scores, const float *cs_row,
                   uint8_t *codes, uint8_t *scales)
{
    float y[OR_D];
    int rc = or_group_prequant(ratio, flags, values, scores, cs_row, y);
    if (rc) return rc;
    return encode_layout(layout, y, codes, scales);
}

/* ------------------------------------------------------------------------ */
/* Paged scatter ([P1] section 1 PagedKV, section 2 kv_page_bytes)           */
/* ------------------------------------------------------------------------ */

static void slot_addresses(int layout, int page_bits, uint8_t *pool, int64_t slot,
                           uint8_t **code_row, uint8_t **scale_row)
{
    int64_t P = (int64_t)1 << page_bits;
    int64_t page = slot >> page_bits, row = slot & (P - 1);
    uint8_t *base = pool + page * (int64_t)or_page_bytes(layout, page_bits);
    *code_row = base + row * (int64_t)or_code_bytes(layout);
    *scale_row = base + P * (int64_t)or_code_bytes(layout) + row * (int64_t)or_scale_bytes(layout);
}

static int valid_layout(int layout) { return layout == OR_V41 || layout == OR_FP4; }

int or_store(int layout, int page_bits, unsigned flags,
             const void *x, int x_dtype, int64_t n, int64_t x_row_stride,
             const int64_t *loc, const float *norm_weight, float eps,
             const float *cos_sin, int64_t cos_sin_rows, const int32_t *pos,
             uint8_t *pool, int64_t pool_slots)
{
    if (!valid_layout(layout) || page_bits < 1 || page_bits > 16 || n < 0) return OR_EINVAL;
    if (x_dtype != OR_F32 && x_dtype != OR_BF16) return OR_EINVAL;
    if ((flags & OR_ROPE) && (!cos_sin || !pos)) return OR_EINVAL;
    if ((flags & OR_NORM) && !norm_weight) return OR_EINVAL;
    size_t esz = x_dtype == OR_F32 ? 4 : 2;
    int rc = OR_OK;
    uint8_t codes[512], scales[32];
    for (int64_t t = 0; t < n; ++t) {
        int64_t slot = loc[t];
        if (slot < 0 || slot >= pool_slots) { rc = OR_ERANGE; continue; }
        const float *cs_row = NULL;
        if (flags & OR_ROPE) {
            if (pos[t] < 0 || pos[t] >= cos_sin_rows) { rc = OR_ERANGE; continue; }
            cs_row = cos_sin + (int64_t)pos[t] * OR_ROPE_D;
        }
        const uint8_t *xrow = (const uint8_t *)x + (size_t)t * (size_t)x_row_stride * esz;
        or_token_bytes(layout, flags, xrow, x_dtype, norm_weight, eps, cs_row, codes, scales);
        uint8_t *crow, *srow;
        slot_addresses(layout, page_bits, pool, slot, &crow, &srow);
        memcpy(crow, codes, or_code_bytes(layout));
        memcpy(srow, scales, or_scale_bytes(layout));
    }
    return rc;
}

int or_compress(int layout, int page_bits, int ratio, unsigned flags,
                const float *values, const float *scores, int64_t n_groups,
                const float *cos_sin, int64_t cos_sin_rows,
                const int32_t *group_pos, const int64_t *loc,
                uint8_t *pool, int64_t pool_slots)
{
    if (!valid_layout(layout) || page_bits < 1 || page_bits > 16 || n_groups < 0) return OR_EINVAL;
    if (ratio < 1 || (flags & OR_NORM)) return OR_EINVAL;
    if ((flags & OR_ROPE) && (!cos_sin || !group_pos)) return OR_EINVAL;
    int rc = OR_OK;
    uint8_t codes[512], scales[32];
    for (int64_t g = 0; g < n_groups; ++g) {
        int64_t slot = loc[g];
        if (slot < 0 || slot >= pool_slots) { rc = OR_ERANGE; continue; }
        const float *cs_row = NULL;
        if (flags & OR_ROPE) {
            if (group_pos[g] < 0 || group_pos[g] >= cos_sin_rows) { rc = OR_ERANGE; continue; }
            cs_row = cos_sin + (int64_t)group_pos[g] * OR_ROPE_D;
        }
        size_t off = (size_t)g * (size_t)ratio * OR_D;
        or_group_bytes(layout, ratio, flags, values + off, scores + off, cs_row, codes, scales);
        uint8_t *crow, *srow;
        slot_addresses(layout, page_bits, pool, slot, &crow, &srow);
        memcpy(crow, codes, or_code_bytes(layout));
        memcpy(srow, scales, or_scale_bytes(layout));
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Dequant to a bf16 workspace ([P1] section 4 dequant_k_cache.py)           */
/* ------------------------------------------------------------------------ */

/* ue8m0 byte -> 2^(byte-127); 0xFF is NaN in OCP MX. */
static double ue8m0_value(uint8_t s)
{
    if (s == 0xFFu) return NAN;
    return ldexp(1.0, (int)s - 127);
}

static uint16_t bf16_of_double(double v)
{
    /* every product here has at most 6 significant bits and is at least
     * 2^-136 in magnitude, so the double -> binary32 step is exact (or
     * overflows to infinity); one rounding to bf16 follows. */
    return or_bf16_bits((float)v);
}

/* One token's 512 bf16 values from its code row and scale row. */
static void decode_row(int layout, const uint8_t *codes, const uint8_t *scales, uint16_t *o)
{
    for (int d = 0; d < OR_D; ++d) {
        double v;
        if (layout == OR_V41) {
            v = or_e4m3_decode(codes[d]) * ue8m0_value(scales[d / OR_BLOCK]);
        } else {
            uint8_t byte = codes[d / 2];
            uint8_t nib = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xFu);
            v = or_e2m1_decode(nib) * or_e4m3_decode(scales[d / OR_BLOCK]);
        }
        o[d] = bf16_of_double(v);
    }
}

int or_dequant(int layout, int page_bits, const uint8_t *pool, int64_t pool_pages,
               const int32_t *page_table, int64_t n_tokens,
               uint16_t *out_bf16, int64_t out_row_stride)
{
    if (!valid_layout(layout) || page_bits < 1 || page_bits > 16 || n_tokens < 0) return OR_EINVAL;
    int64_t P = (int64_t)1 << page_bits;
    if (n_tokens % P) return OR_EINVAL;
    int64_t PB = (int64_t)or_page_bytes(layout, page_bits);
    int64_t CB = (int64_t)or_code_bytes(layout), SB = (int64_t)or_scale_bytes(layout);
    int rc = OR_OK;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t phys = page_table[t >> page_bits];
        if (phys < 0 || phys >= pool_pages) { rc = OR_ERANGE; continue; }
        int64_t row = t & (P - 1);
        decode_row(layout, pool + phys * PB + row * CB, pool + phys * PB + P * CB + row * SB,
                   out_bf16 + t * out_row_stride);
    }
    return rc;
}

/* Dequant of selected tokens (the consumer side of [P1] section 4: only the
 * slots a sparse attention picks): out row i = the token in slot slots[i].
 * Slot -1 is padding and gives a zero row; any other slot outside the pool
 * leaves row i untouched and returns the out-of-range status. */
int or_dequant_slots(int layout, int page_bits, const uint8_t *pool, int64_t pool_slots,
                     const int64_t *slots, int64_t n, uint16_t *out_bf16, int64_t out_row_stride)
{
    if (!valid_layout(layout) || page_bits < 1 || page_bits > 16 || n < 0) return OR_EINVAL;
    int rc = OR_OK;
    for (int64_t i = 0; i < n; ++i) {
        uint16_t *o = out_bf16 + i * out_row_stride;
        int64_t s = slots[i];
        if (s == -1) {
            for (int d = 0; d < OR_D; ++d) o[d] = 0;
            continue;
        }
        if (s < 0 || s >= pool_slots) { rc = OR_ERANGE; continue; }
        uint8_t *crow, *srow;
        slot_addresses(layout, page_bits, (uint8_t *)pool, s, &crow, &srow);
        decode_row(layout, crow, srow, o);
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Full -> SWA slot translation, once per step ([P2] sections 1 and 2):      */
/* out[:n] = table[loc] as int32, out[n:capacity] = 0, and n > capacity is   */
/* the "no buffer" case (the caller falls back).  A loc outside the table    */
/* gives -1 there and an out-of-range status.                                */
/* ------------------------------------------------------------------------ */

int or_translate(const int64_t *loc, int64_t n, const int32_t *full_to_swa,
                 int64_t full_slots, int32_t *out, int64_t capacity)
{
    if (n < 0 || capacity < 0) return OR_EINVAL;
    if (n > capacity) return OR_ECAP;
    int rc = OR_OK;
    for (int64_t i = 0; i < n; ++i) {
        int64_t l = loc[i];
        if (l < 0 || l >= full_slots) { out[i] = -1; rc = OR_ERANGE; continue; }
        out[i] = full_to_swa[l];
    }
    for (int64_t i = n; i < capacity; ++i) out[i] = 0;
    return rc;
}
