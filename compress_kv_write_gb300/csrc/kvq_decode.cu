// kvq_decode.cu -- decode-time compressor: the c1 / c2 decode kernels of
// "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats" (section 2)
// and the C4A / C128A windows of "[vLLM] DeepSeek V4 Sparse FP8 Compressor
// kernel" fed one row per request per call, with the same online softmax
// (section 2), RoPE, bf16 cast and absmax (section 3) as kvq_compress.cu.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

// Decode-time compressor: one new row per request per call, the group's
// softmax carried between calls as per-dim online state (running max m,
// sum of exp(s - m) and sum of exp(s - m) * v), 3 x 512 fp32 per request.
// One CTA of four warps per request: warp w owns the dims 128 w .. 128 w +
// 127, lane l of it the float4 column 32 w + l, so every warp access is one
// contiguous 512-byte span and a quant block is 8 adjacent lanes.  Four
// warps per request rather than one make each request's dependent chain of
// loads, exponentials, divisions, shuffles and conversions a quarter as long
// (the whole launch at small batches) and keep four times as many rows in
// flight per resident request at large ones.  The count is read by every
// thread of the CTA and rewritten by thread 0 after a barrier.

constexpr int kDecWarps = 4;  // warps per CTA: one request
static_assert(kDecWarps * 32 * 4 == kD, "one float4 column per thread");

struct DecodeArgs {
    const float *values;
    const float *scores;
    int64_t n;
    float *state;
    int32_t *count;
    const int32_t *req;
    int64_t n_state;
    const float *cs;
    int64_t cs_rows;
    const int32_t *group_pos;
    const int32_t *loc;
    uint8_t *pool;
    int64_t pool_slots;
    int32_t *err;
    int warm;  // prefetch each request's row and state into L2 before the PDL wait
};

template <Layout L, int PageBits, int R, bool kRope>
__global__ void __launch_bounds__(kDecWarps * 32) compress_decode_kernel(const DecodeArgs a) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    const int t = threadIdx.x;   // float4 column: dims 4t .. 4t+3, quant block t / 8
    const int lane = t & 31;
    const int64_t i = blockIdx.x;  // the request (the grid is exactly n CTAs)
    // While the upstream grid drains: L2 hints for this request's new row and
    // its state (hints only; every load below comes after the wait).
    if (a.warm) {
        const int64_t rh = a.req ? -1 : i;  // the state row is known only without an index array
        if (t == 0) prefetch_l2_bulk(a.values + i * kD, kD * 4);
        if (t == 32) prefetch_l2_bulk(a.scores + i * kD, kD * 4);
        if (t == 64 && rh >= 0 && rh < a.n_state) prefetch_l2_bulk(a.state + rh * (3 * kD), 3 * kD * 4);
    }
    pdl_wait();

    // Everything that does not depend on the request's count is requested
    // first: the new row, the group's slot and position (and, for ratio 1,
    // where every row completes a group, its cos/sin values).  Only the state
    // waits for the count.
    const int64_t ri = a.req ? int64_t(__ldg(a.req + i)) : i;
    const float4 v = ld_f4(a.values + i * kD + 4 * t);
    const float4 sc = ld_f4(a.scores + i * kD + 4 * t);
    const int64_t slot = __ldg(a.loc + i);
    const int32_t pos = kRope ? __ldg(a.group_pos + i) : 0;
    const bool pos_ok = !kRope || (pos >= 0 && int64_t(pos) < a.cs_rows);
    const bool rope_col = kRope && 4 * t >= kRopeStart;  // rotated dims of this column
    float2 cs_c = make_float2(1.f, 1.f), cs_s = make_float2(0.f, 0.f);
    auto load_cs = [&]() {
        if (rope_col && pos_ok) {
            const int i0 = (4 * t - kRopeStart) / 2;
            const float *cs = a.cs + int64_t(pos) * kRopeD;
            cs_c = __ldg(reinterpret_cast<const float2 *>(cs + i0));
            cs_s = __ldg(reinterpret_cast<const float2 *>(cs + kRopeD / 2 + i0));
        }
    };
    if constexpr (R == 1) load_cs();
    pdl_trigger();  // the next launch may start its prologue; its wait still covers this grid
    const int32_t c = (ri >= 0 && ri < a.n_state) ? a.count[ri] : -1;
    __syncthreads();  // every thread has read the count before thread 0 rewrites it
    if (c < 0 || c >= R) {
        if (t == 0) raise_err(a.err, KVQ_DEVERR_STATE);
        return;
    }
    if constexpr (R > 1) {
        if (c == R - 1) load_cs();
    }
    float *st = a.state + ri * (3 * kD) + 4 * t;
    float4 m = sc, l = make_float4(1.f, 1.f, 1.f, 1.f), acc = v;
    if (c > 0) {
        const float4 m0 = *reinterpret_cast<const float4 *>(st);
        const float4 l0 = *reinterpret_cast<const float4 *>(st + kD);
        const float4 a0 = *reinterpret_cast<const float4 *>(st + 2 * kD);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float mo = (&m0.x)[e], so = (&sc.x)[e];
            const float mn = fmaxf(mo, so);
            const float al = ex2_approx((mo - mn) * kLog2e);
            const float p = ex2_approx((so - mn) * kLog2e);
            (&m.x)[e] = mn;
            (&l.x)[e] = fmaf((&l0.x)[e], al, p);
            (&acc.x)[e] = fmaf(p, (&v.x)[e], (&a0.x)[e] * al);
        }
    }
    if (c + 1 < R) {  // the group is still open: keep the state
        *reinterpret_cast<float4 *>(st) = m;
        *reinterpret_cast<float4 *>(st + kD) = l;
        *reinterpret_cast<float4 *>(st + 2 * kD) = acc;
        if (t == 0) a.count[ri] = c + 1;
        return;
    }
    // the group is complete: pool, rotate, round, quantise, store; restart
    if (R > 1 && t == 0) a.count[ri] = 0;  // ratio 1: the count is 0 already
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = R == 1 ? (&acc.x)[e] : __fdiv_rn((&acc.x)[e], (&l.x)[e]);  // ratio 1: l = 1
    if (rope_col && pos_ok) {
        const float c2[2] = {cs_c.x, cs_c.y}, s2[2] = {cs_s.x, cs_s.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float x0 = y[2 * q], x1 = y[2 * q + 1];
            y[2 * q] = __fsub_rn(__fmul_rn(x0, c2[q]), __fmul_rn(x1, s2[q]));
            y[2 * q + 1] = __fadd_rn(__fmul_rn(x0, s2[q]), __fmul_rn(x1, c2[q]));
        }
    }
    if (!pos_ok || slot < 0 || slot >= a.pool_slots) {
        if (t == 0) raise_err(a.err, pos_ok ? KVQ_DEVERR_SLOT : KVQ_DEVERR_POS);
        return;
    }
    uint8_t *crow = PK::code_row(a.pool, slot);
    uint8_t *srow = PK::scale_row(a.pool, slot);
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = round_bf16(y[e]);
    uint32_t am = max(max(abs_bits(y[0]), abs_bits(y[1])), max(abs_bits(y[2]), abs_bits(y[3])));
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, off));
    uint32_t sbyte;
    if constexpr (L == Layout::V41) {
        sbyte = v41_scale_byte(am);
        const float mult = v41_multiplier(sbyte);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(y[0], mult), __fmul_rn(y[1], mult));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(y[2], mult), __fmul_rn(y[3], mult));
        *reinterpret_cast<uint32_t *>(crow + 4 * t) = lo | (hi << 16);
    } else {
        sbyte = fp4_scale_byte(am);
        const float S = e4m3x2_to_f32x2(sbyte).x;
        const float inv = __frcp_rn(S);
        uint32_t word = 0;
        if (S != 0.0f)
            word = cvt_e2m1x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) |
                   (cvt_e2m1x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 8);
        *reinterpret_cast<uint16_t *>(crow + 2 * t) = uint16_t(word);
    }
    if ((lane & 7) == 0) srow[t >> 3] = uint8_t(sbyte);
    if constexpr (T::kScaleBytes == 32) {
        if (t == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
    }
}

template <Layout L, int PB, int R, bool RP>
kvq_status launch_compress_decode(DecodeArgs a, cudaStream_t stream) {
    constexpr auto kern = compress_decode_kernel<L, PB, R, RP>;
    if (a.n > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    int64_t wave = 0;
    const kvq_status st = resident_grid<kern, kDecWarps * 32>(0, &wave);
    if (st != KVQ_OK) return st;
    // Beyond one wave the hints would only duplicate the loads of CTAs that
    // start after the upstream grid has finished.
    a.warm = a.n <= wave;
    return launch_pdl(kern, dim3(unsigned(a.n)), dim3(kDecWarps * 32), stream, a);
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_compress_decode(kvq_layout layout, int page_bits, int ratio, unsigned flags,
                                          const float *values, const float *scores, int64_t n, float *state,
                                          int32_t *count, const int32_t *req, int64_t n_state,
                                          const float *cos_sin, int64_t cos_sin_rows, const int32_t *group_pos,
                                          const int32_t *loc, uint8_t *pool, int64_t pool_slots, int32_t *err,
                                          struct CUstream_st *stream) {
    kvq_status st = check_pool(layout, page_bits, pool, pool_slots);
    if (st != KVQ_OK) return st;
    if (flags & ~unsigned(KVQ_FLAG_ROPE | KVQ_FLAG_NORM)) return KVQ_ERR_INVALID_ARG;
    if (flags & KVQ_FLAG_NORM) return KVQ_ERR_UNSUPPORTED;
    if (ratio < 1) return KVQ_ERR_INVALID_ARG;
    if (ratio != 1 && ratio != 2 && ratio != 4 && ratio != 128) return KVQ_ERR_UNSUPPORTED;
    if (n < 0 || n_state < 0) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;  // nothing to enqueue
    if (!values || !scores || !aligned(values, 16) || !aligned(scores, 16)) return KVQ_ERR_INVALID_ARG;
    if (!state || !aligned(state, 16) || !count || !aligned(count, 4) || n_state == 0) return KVQ_ERR_INVALID_ARG;
    if (req && !aligned(req, 4)) return KVQ_ERR_INVALID_ARG;
    if (!req && n > n_state) return KVQ_ERR_INVALID_ARG;
    if (!loc || !aligned(loc, 4)) return KVQ_ERR_INVALID_ARG;
    const bool rope = flags & KVQ_FLAG_ROPE;
    if (rope && (!cos_sin || !aligned(cos_sin, 16) || cos_sin_rows <= 0 || !group_pos || !aligned(group_pos, 4)))
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;

    DecodeArgs a;
    a.values = values;
    a.scores = scores;
    a.n = n;
    a.state = state;
    a.count = count;
    a.req = req;
    a.n_state = n_state;
    a.cs = cos_sin;
    a.cs_rows = cos_sin_rows;
    a.group_pos = group_pos;
    a.loc = loc;
    a.pool = pool;
    a.pool_slots = pool_slots;
    a.err = err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return with_ratio(ratio, [&](auto Rc) {
                return with_bool(rope, [&](auto RPc) {
                    return launch_compress_decode<decltype(Lc)::value, decltype(PBc)::value,
                                                  decltype(Rc)::value, decltype(RPc)::value>(a, s);
                });
            });
        });
    });
}
