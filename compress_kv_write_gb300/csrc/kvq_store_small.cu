// kvq_store_small.cu -- the store / store + RoPE / fused K norm + RoPE of
// "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats" (section 1
// store_row, and the store-latency table at bs 1 .. 512) for small batches,
// both layouts.
//
// A small batch is one dependent chain per token: the row, slot and position
// loads, the position -> cos/sin load, the norm's reduction, the rounding,
// the block absmax and the conversions.  The persistent kernels give a token
// to one warp (16 values per lane), so at a few hundred tokens the launch
// lasts as long as one warp's instruction stream.  Here a token is one CTA
// of four warps and thread t owns the dims 4t .. 4t+3: a quarter of the
// per-thread chain, with the norm's sum reduced over the four warps through
// shared memory.  Semantics, roundings and error bits are those of the
// persistent kernels (kvq_store.cu).
#include "kvq_store.cuh"

namespace kvq {
namespace {

constexpr int kTokThreads = kD / 4;  // one CTA per token, four dims per thread
static_assert(kTokThreads % 32 == 0 && kBlock % 4 == 0, "whole warps; a quant block is whole threads");

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope>
__global__ void __launch_bounds__(kTokThreads) store_token_kernel(const StoreArgs a) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int kTPB = kBlock / 4;  // threads per quant block
    __shared__ float s_ss[kTokThreads / 32];
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int64_t i = blockIdx.x;  // the token (the grid is exactly n CTAs)
    const uint8_t *xr = a.x + i * a.row_stride_bytes;

    // While the upstream grid drains: L2 hints for the row and the token's
    // slot / position lines (the loads come after the wait).
    if (t == 0) prefetch_l2_bulk(xr, kD * (kBf16 ? 2 : 4));
    if (t == 32)
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + i)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + i));
    if (kRope && t == 64) prefetch_l2(a.pos + i);
    pdl_wait();

    float v[4];
    if constexpr (kBf16) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(xr) + t);
        v[0] = bf16_lo(r.x), v[1] = bf16_hi(r.x), v[2] = bf16_lo(r.y), v[3] = bf16_hi(r.y);
    } else {
        const float4 f = ld_f4(reinterpret_cast<const float *>(xr) + 4 * t);
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    }
    const int64_t s = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + i)
                             : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + i));
    const bool rot = kRope && 4 * t >= kRopeStart;  // this thread's dims are rotated
    int32_t p = 0;
    bool pos_ok = true;
    float2 cs_c = make_float2(1.f, 1.f), cs_s = make_float2(0.f, 0.f);
    if constexpr (kRope) {
        p = __ldg(a.pos + i);
        pos_ok = p >= 0 && int64_t(p) < a.cs_rows;
        if (rot && pos_ok) {
            const int i0 = (4 * t - kRopeStart) / 2;  // first of this thread's two pairs
            const float *cs = a.cs + int64_t(p) * kRopeD;
            cs_c = __ldg(reinterpret_cast<const float2 *>(cs + i0));
            cs_s = __ldg(reinterpret_cast<const float2 *>(cs + kRopeD / 2 + i0));
        }
    }
    float4 w = make_float4(1.f, 1.f, 1.f, 1.f);
    if constexpr (kNorm) w = __ldg(reinterpret_cast<const float4 *>(a.w) + t);
    pdl_trigger();

    // Same checks, same order and same error bits as the persistent kernels;
    // both conditions are the token's, so the whole CTA leaves together.
    if (!pos_ok) {
        if (t == 0) raise_err(a.err, KVQ_DEVERR_POS);
        return;
    }
    if (s < 0 || s >= a.pool_slots) {
        if (t == 0) raise_err(a.err, KVQ_DEVERR_SLOT);
        return;
    }

    if constexpr (kNorm) {
        float ss = __fmul_rn(v[0], v[0]);
#pragma unroll
        for (int e = 1; e < 4; ++e) ss = fmaf(v[e], v[e], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) s_ss[t >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int k = 0; k < kTokThreads / 32; ++k) ss += s_ss[k];
        const float inv = rsqrt_approx(__fadd_rn(ss * (1.0f / kD), a.eps));
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], inv), wv[e]);
    }
    if (rot) {
        const float c2[2] = {cs_c.x, cs_c.y}, s2[2] = {cs_s.x, cs_s.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float x0 = v[2 * q], x1 = v[2 * q + 1];
            v[2 * q] = __fsub_rn(__fmul_rn(x0, c2[q]), __fmul_rn(x1, s2[q]));
            v[2 * q + 1] = __fadd_rn(__fmul_rn(x0, s2[q]), __fmul_rn(x1, c2[q]));
        }
    }
    // bf16 rounding: the rotated dims once after the rotation; the others
    // after the norm, and with RoPE also fp32 input (as the persistent kernels).
    if (rot || kNorm || (kRope && !kBf16)) {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = round_bf16(v[e]);
    }

    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 1; off < kTPB; off <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    uint8_t *crow = PK::code_row(a.pool, s);
    uint8_t *srow = PK::scale_row(a.pool, s);
    uint32_t sbyte;
    if constexpr (L == Layout::V41) {
        sbyte = v41_scale_byte(__float_as_uint(am));
        const float mult = v41_multiplier(sbyte);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[0], mult), __fmul_rn(v[1], mult));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[2], mult), __fmul_rn(v[3], mult));
        *reinterpret_cast<uint32_t *>(crow + 4 * t) = lo | (hi << 16);
    } else {
        sbyte = fp4_scale_byte(__float_as_uint(am));
        const float S = e4m3x2_to_f32x2(sbyte).x;
        uint32_t word = 0;
        if (S != 0.0f) {
            const float inv = __frcp_rn(S);
            word = cvt_e2m1x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
                   (cvt_e2m1x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 8);
        }
        *reinterpret_cast<uint16_t *>(crow + 2 * t) = uint16_t(word);
    }
    if ((t & (kTPB - 1)) == 0) srow[t / kTPB] = uint8_t(sbyte);
    if constexpr (T::kScaleBytes == 32) {
        if (t == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
    }
}

}  // namespace

kvq_status launch_store_small(int layout, int page_bits, bool bf16, bool loc64, bool norm, bool rope,
                              const StoreArgs &a, cudaStream_t stream) {
    if (a.n > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;  // one CTA per token
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return with_bool(bf16, [&](auto B16) {
                return with_bool(loc64, [&](auto L64) {
                    return with_bool(norm, [&](auto Nc) {
                        return with_bool(rope, [&](auto Rc) {
                            constexpr auto kern =
                                store_token_kernel<decltype(Lc)::value, decltype(PBc)::value, decltype(B16)::value,
                                                   decltype(L64)::value, decltype(Nc)::value, decltype(Rc)::value>;
                            return launch_pdl(kern, dim3(unsigned(a.n)), dim3(kTokThreads), stream, a);
                        });
                    });
                });
            });
        });
    });
}

}  // namespace kvq
