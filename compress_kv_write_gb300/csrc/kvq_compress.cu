// kvq_compress.cu -- ratio-r per-element softmax compressor over whole
// groups, fused with RoPE, bf16 rounding, block quantisation and the paged
// store: the C4A / C128A compressors of "[vLLM] DeepSeek V4 Sparse FP8
// Compressor kernel" (section 2: online max / sum softmax; section 3: RoPE,
// bf16 cast, per-32-value absmax), and ratios 1 / 2 of the c1 / c2
// compressors of "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
// (section 2).  The decode-time form is in kvq_decode.cu.
//
// Mapping: 128 threads per group; thread t owns dims 4t..4t+3 (one float4
// column), so each row is one fully coalesced 2 KB sweep by the group's
// threads.  A thread streams its column of the r value and score rows in
// chunks of U rows (all 2U 16-byte loads of a chunk in flight), keeping an
// online softmax state per dim: chunk max first, then one rescale of the
// running sum / accumulator per chunk (1 + 1/U exponentials per element-row).
// A quant block is 8 adjacent threads of one warp (3 xor shuffles).
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kGroupThreads = 128;

struct CompressArgs {
    const float *values;
    const float *scores;
    int64_t n_groups;
    const float *cs;
    int64_t cs_rows;
    const int32_t *group_pos;
    const int32_t *loc;
    uint8_t *pool;
    int64_t pool_slots;
    int32_t *err;
};

template <Layout L, int PageBits, int R, bool kRope, int GPC>
__global__ void __launch_bounds__(kGroupThreads *GPC) compress_kernel(const CompressArgs a) {
    constexpr int U = R < 8 ? R : 8;  // rows per chunk
    static_assert(R % U == 0, "ratio must be a multiple of the chunk");
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;

    __shared__ __align__(16) uint8_t s_scale[GPC][kNBlk];

    const int sub = threadIdx.x / kGroupThreads;
    const int t = threadIdx.x % kGroupThreads;
    const int lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * GPC + sub;
    const bool active = g < a.n_groups;

    pdl_wait();

    int64_t slot = -1;
    int32_t pos = 0;
    if (active) {
        slot = __ldg(a.loc + g);
        if constexpr (kRope) pos = __ldg(a.group_pos + g);
    }
    const bool rope_thread = kRope && (4 * t >= kRopeStart);

    float m[4], l[4], acc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        m[e] = -INFINITY;
        l[e] = 0.f;
        acc[e] = 0.f;
    }
    float2 cs_c = make_float2(1.f, 1.f), cs_s = make_float2(0.f, 0.f);
    bool pos_ok = true;

    if (active) {
        const float *vcol = a.values + g * (int64_t(R) * kD) + 4 * t;
        const float *scol = a.scores + g * (int64_t(R) * kD) + 4 * t;
#pragma unroll(R / U <= 4 ? R / U : 1)
        for (int r0 = 0; r0 < R; r0 += U) {
            float4 vv[U], ss[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                vv[u] = ld_f4(vcol + int64_t(r0 + u) * kD);
                ss[u] = ld_f4(scol + int64_t(r0 + u) * kD);
            }
            if (r0 == 0) {
                // the rotation angles: issued once the first rows are in flight
                if constexpr (kRope) {
                    pos_ok = pos >= 0 && int64_t(pos) < a.cs_rows;
                    if (rope_thread && pos_ok) {
                        const int i0 = (4 * t - kRopeStart) / 2;
                        const float *cs = a.cs + int64_t(pos) * kRopeD;
                        cs_c = __ldg(reinterpret_cast<const float2 *>(cs + i0));
                        cs_s = __ldg(reinterpret_cast<const float2 *>(cs + kRopeD / 2 + i0));
                    }
                }
                if (R == U) pdl_trigger();
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float cm = m[e];
#pragma unroll
                for (int u = 0; u < U; ++u) cm = fmaxf(cm, (&ss[u].x)[e]);
                const float cml = cm * kLog2e;
                const float alpha = ex2_approx(fmaf(m[e], kLog2e, -cml));
                float ls = l[e] * alpha, as = acc[e] * alpha;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float p = ex2_approx(fmaf((&ss[u].x)[e], kLog2e, -cml));
                    ls += p;
                    as = fmaf(p, (&vv[u].x)[e], as);
                }
                m[e] = cm;
                l[e] = ls;
                acc[e] = as;
            }
        }
    }
    if (R != U) pdl_trigger();

    // ---- pooled value, RoPE, bf16
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = active ? __fdiv_rn(acc[e], l[e]) : 0.f;
    if (kRope && rope_thread) {
        const float c[2] = {cs_c.x, cs_c.y}, s[2] = {cs_s.x, cs_s.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float x0 = y[2 * q], x1 = y[2 * q + 1];
            y[2 * q] = __fsub_rn(__fmul_rn(x0, c[q]), __fmul_rn(x1, s[q]));
            y[2 * q + 1] = __fadd_rn(__fmul_rn(x0, s[q]), __fmul_rn(x1, c[q]));
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = round_bf16(y[e]);

    // ---- block absmax over 8 threads (32 dims)
    uint32_t am = max(max(abs_bits(y[0]), abs_bits(y[1])), max(abs_bits(y[2]), abs_bits(y[3])));
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, off));

    const bool write = active && slot >= 0 && slot < a.pool_slots && pos_ok;
    uint32_t sbyte;
    if constexpr (L == Layout::V41) {
        sbyte = v41_scale_byte(am);
        const float mult = v41_multiplier(sbyte);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(y[0], mult), __fmul_rn(y[1], mult));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(y[2], mult), __fmul_rn(y[3], mult));
        if (write) *reinterpret_cast<uint32_t *>(PK::code_row(a.pool, slot) + 4 * t) = lo | (hi << 16);
    } else {
        sbyte = fp4_scale_byte(am);
        const float S = e4m3x2_to_f32x2(sbyte).x;
        const float inv = __frcp_rn(S);
        uint32_t word = 0;
        if (S != 0.0f) {
            word = cvt_e2m1x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) |
                   (cvt_e2m1x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 8);
        }
        if (write) *reinterpret_cast<uint16_t *>(PK::code_row(a.pool, slot) + 2 * t) = uint16_t(word);
    }
    if ((t & 7) == 0) s_scale[sub][t >> 3] = uint8_t(sbyte);
    __syncthreads();
    if (write) {
        uint8_t *srow = PK::scale_row(a.pool, slot);
        if (t == 0) st_u4(srow, *reinterpret_cast<const uint4 *>(s_scale[sub]));
        if constexpr (T::kScaleBytes == 32) {
            if (t == 1) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
        }
    } else if (active && t == 0) {
        raise_err(a.err, pos_ok ? KVQ_DEVERR_SLOT : KVQ_DEVERR_POS);
    }
    (void)lane;
}

template <Layout L, int PB, int R, bool RP>
kvq_status launch_compress(const CompressArgs &a, cudaStream_t stream) {
    constexpr int GPC = R <= 4 ? 2 : 1;
    const int64_t blocks = (a.n_groups + GPC - 1) / GPC;
    if (blocks > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    return launch_pdl(compress_kernel<L, PB, R, RP, GPC>, dim3(unsigned(blocks)),
                      dim3(kGroupThreads * GPC), stream, a);
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_compress(kvq_layout layout, int page_bits, int ratio, unsigned flags,
                                   const float *values, const float *scores, int64_t n_groups,
                                   const float *cos_sin, int64_t cos_sin_rows,
                                   const int32_t *group_pos, const int32_t *loc, uint8_t *pool,
                                   int64_t pool_slots, int32_t *err, struct CUstream_st *stream) {
    kvq_status st = check_pool(layout, page_bits, pool, pool_slots);
    if (st != KVQ_OK) return st;
    if (flags & ~unsigned(KVQ_FLAG_ROPE | KVQ_FLAG_NORM)) return KVQ_ERR_INVALID_ARG;
    if (flags & KVQ_FLAG_NORM) return KVQ_ERR_UNSUPPORTED;
    if (ratio < 1) return KVQ_ERR_INVALID_ARG;
    if (ratio != 1 && ratio != 2 && ratio != 4 && ratio != 128) return KVQ_ERR_UNSUPPORTED;
    if (n_groups < 0) return KVQ_ERR_INVALID_ARG;
    if (n_groups == 0) return KVQ_OK;  // nothing to enqueue; inputs may be empty (null)
    if (!values || !scores || !aligned(values, 16) || !aligned(scores, 16)) return KVQ_ERR_INVALID_ARG;
    if (!loc || !aligned(loc, 4)) return KVQ_ERR_INVALID_ARG;
    const bool rope = flags & KVQ_FLAG_ROPE;
    if (rope && (!cos_sin || !aligned(cos_sin, 16) || cos_sin_rows <= 0 || !group_pos ||
                 !aligned(group_pos, 4)))
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;

    CompressArgs a;
    a.values = values;
    a.scores = scores;
    a.n_groups = n_groups;
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
                    return launch_compress<decltype(Lc)::value, decltype(PBc)::value,
                                           decltype(Rc)::value, decltype(RPc)::value>(a, s);
                });
            });
        });
    });
}
