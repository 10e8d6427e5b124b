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
// of four warps, thread t owning dims 4t .. 4t+3 (a quarter of the
// per-thread chain), or half a CTA, eight dims per thread, where one CTA per
// token would cost more to schedule than the shorter chain saves.  The
// norm's sum is reduced over the token's warps through shared memory.
// Semantics, roundings and error bits are those of the persistent kernels
// (kvq_store.cu).
#include "kvq_store.cuh"

namespace kvq {
namespace {

constexpr int kTokThreads = 128;  // threads per CTA

// kTPC tokens per CTA: thread t serves token t / (128 / kTPC) and owns
// kV = 4 kTPC consecutive dims of it.  With two tokens per CTA each token's
// two warps meet at a named barrier of their own (1 + token), so a token that
// leaves early (a bad slot or position, or past the batch) holds up nobody.
template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope, int kTPC>
__global__ void __launch_bounds__(kTokThreads) store_token_kernel(const StoreArgs a) {
    static_assert(kTPC == 1 || kTPC == 2, "one or two tokens per CTA (named barriers 1 and 2)");
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int kTT = kTokThreads / kTPC;  // threads per token
    constexpr int kV = kD / kTT;             // values per thread
    constexpr int kTPB = kBlock / kV;        // threads per quant block
    static_assert(kTT % 32 == 0 && kV % 4 == 0 && kBlock % kV == 0, "whole warps, whole float4s, whole blocks");
    __shared__ float s_ss[kTokThreads / 32];
    const int lane = threadIdx.x & 31;
    const int tok = threadIdx.x / kTT;           // token of the CTA
    const int t = threadIdx.x % kTT;             // thread within the token
    const int64_t i = int64_t(blockIdx.x) * kTPC + tok;  // the token
    if (i >= a.n) return;  // a whole token's threads; no barrier waits on them
    const uint8_t *xr = a.x + i * a.row_stride_bytes;

    // While the upstream grid drains: L2 hints for the row and the token's
    // slot / position lines (the loads come after the wait).
    if (t == 0) prefetch_l2_bulk(xr, kD * (kBf16 ? 2 : 4));
    if (t == 32)
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + i)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + i));
    if (kRope && t == kTT - 1) prefetch_l2(a.pos + i);
    pdl_wait();

    float v[kV];
#pragma unroll
    for (int q = 0; q < kV / 4; ++q) {
        if constexpr (kBf16) {
            const uint2 r = __ldg(reinterpret_cast<const uint2 *>(xr) + t * (kV / 4) + q);
            v[4 * q] = bf16_lo(r.x), v[4 * q + 1] = bf16_hi(r.x);
            v[4 * q + 2] = bf16_lo(r.y), v[4 * q + 3] = bf16_hi(r.y);
        } else {
            const float4 f = ld_f4(reinterpret_cast<const float *>(xr) + kV * t + 4 * q);
            v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
        }
    }
    const int64_t s = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + i)
                             : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + i));
    const bool rot = kRope && kV * t >= kRopeStart;  // this thread's dims are rotated
    int32_t p = 0;
    bool pos_ok = true;
    float cs_c[kV / 2], cs_s[kV / 2];
#pragma unroll
    for (int q = 0; q < kV / 2; ++q) cs_c[q] = 1.f, cs_s[q] = 0.f;
    if constexpr (kRope) {
        p = __ldg(a.pos + i);
        pos_ok = p >= 0 && int64_t(p) < a.cs_rows;
        if (rot && pos_ok) {
            const int i0 = (kV * t - kRopeStart) / 2;  // first of this thread's kV / 2 pairs
            const float *cs = a.cs + int64_t(p) * kRopeD;
#pragma unroll
            for (int q = 0; q < kV / 4; ++q) {
                const float2 c = __ldg(reinterpret_cast<const float2 *>(cs + i0) + q);
                const float2 sn = __ldg(reinterpret_cast<const float2 *>(cs + kRopeD / 2 + i0) + q);
                cs_c[2 * q] = c.x, cs_c[2 * q + 1] = c.y, cs_s[2 * q] = sn.x, cs_s[2 * q + 1] = sn.y;
            }
        }
    }
    float w[kV];
#pragma unroll
    for (int q = 0; q < kV / 4; ++q) {
        float4 f = make_float4(1.f, 1.f, 1.f, 1.f);
        if constexpr (kNorm) f = __ldg(reinterpret_cast<const float4 *>(a.w) + t * (kV / 4) + q);
        w[4 * q] = f.x, w[4 * q + 1] = f.y, w[4 * q + 2] = f.z, w[4 * q + 3] = f.w;
    }
    pdl_trigger();

    // Same checks, same order and same error bits as the persistent kernels;
    // both conditions are the token's, so all its threads leave together.
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
        for (int e = 1; e < kV; ++e) ss = fmaf(v[e], v[e], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) s_ss[threadIdx.x >> 5] = ss;
        if constexpr (kTPC == 1) {
            __syncthreads();
        } else {
            // immediate barrier ids (a register id would reserve all sixteen)
            if (tok == 0) {
                asm volatile("bar.sync 1, %0;" ::"n"(kTT) : "memory");
            } else {
                asm volatile("bar.sync 2, %0;" ::"n"(kTT) : "memory");
            }
        }
        ss = 0.f;
#pragma unroll
        for (int k = 0; k < kTT / 32; ++k) ss += s_ss[tok * (kTT / 32) + k];
        const float inv = rsqrt_approx(__fadd_rn(ss * (1.0f / kD), a.eps));
#pragma unroll
        for (int e = 0; e < kV; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], inv), w[e]);
    }
    if (rot) {
#pragma unroll
        for (int q = 0; q < kV / 2; ++q) {
            const float x0 = v[2 * q], x1 = v[2 * q + 1];
            v[2 * q] = __fsub_rn(__fmul_rn(x0, cs_c[q]), __fmul_rn(x1, cs_s[q]));
            v[2 * q + 1] = __fadd_rn(__fmul_rn(x0, cs_s[q]), __fmul_rn(x1, cs_c[q]));
        }
    }
    // bf16 rounding: the rotated dims once after the rotation; the others
    // after the norm, and with RoPE also fp32 input (as the persistent kernels).
    if (rot || kNorm || (kRope && !kBf16)) {
#pragma unroll
        for (int e = 0; e < kV; ++e) v[e] = round_bf16(v[e]);
    }

    float am = fabsf(v[0]);
#pragma unroll
    for (int e = 1; e < kV; ++e) am = fmaxf(am, fabsf(v[e]));
#pragma unroll
    for (int off = 1; off < kTPB; off <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    uint8_t *crow = PK::code_row(a.pool, s);
    uint8_t *srow = PK::scale_row(a.pool, s);
    uint32_t sbyte;
    if constexpr (L == Layout::V41) {
        sbyte = v41_scale_byte(__float_as_uint(am));
        const float mult = v41_multiplier(sbyte);
        uint32_t wd[kV / 4];
#pragma unroll
        for (int q = 0; q < kV / 4; ++q)
            wd[q] = cvt_e4m3x2(__fmul_rn(v[4 * q], mult), __fmul_rn(v[4 * q + 1], mult)) |
                    (cvt_e4m3x2(__fmul_rn(v[4 * q + 2], mult), __fmul_rn(v[4 * q + 3], mult)) << 16);
        if constexpr (kV == 4) {
            *reinterpret_cast<uint32_t *>(crow + 4 * t) = wd[0];
        } else {
            *reinterpret_cast<uint2 *>(crow + 8 * t) = make_uint2(wd[0], wd[1]);
        }
    } else {
        sbyte = fp4_scale_byte(__float_as_uint(am));
        const float S = e4m3x2_to_f32x2(sbyte).x;
        uint32_t word = 0;
        if (S != 0.0f) {
            const float inv = __frcp_rn(S);
#pragma unroll
            for (int q = 0; q < kV / 2; ++q)
                word |= cvt_e2m1x2(__fmul_rn(v[2 * q], inv), __fmul_rn(v[2 * q + 1], inv)) << (8 * q);
        }
        if constexpr (kV == 4) {
            *reinterpret_cast<uint16_t *>(crow + 2 * t) = uint16_t(word);
        } else {
            *reinterpret_cast<uint32_t *>(crow + 4 * t) = word;
        }
    }
    if ((t & (kTPB - 1)) == 0) srow[t / kTPB] = uint8_t(sbyte);
    if constexpr (T::kScaleBytes == 32) {
        if (t == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
    }
}

}  // namespace

kvq_status launch_store_small(int layout, int page_bits, bool bf16, bool loc64, bool norm, bool rope,
                              int tokens_per_cta, const StoreArgs &a, cudaStream_t stream) {
    if (a.n > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;  // one CTA per token
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return with_bool(bf16, [&](auto B16) {
                return with_bool(loc64, [&](auto L64) {
                    return with_bool(norm, [&](auto Nc) {
                        return with_bool(rope, [&](auto Rc) {
                            constexpr auto kern1 =
                                store_token_kernel<decltype(Lc)::value, decltype(PBc)::value, decltype(B16)::value,
                                                   decltype(L64)::value, decltype(Nc)::value, decltype(Rc)::value, 1>;
                            constexpr auto kern2 =
                                store_token_kernel<decltype(Lc)::value, decltype(PBc)::value, decltype(B16)::value,
                                                   decltype(L64)::value, decltype(Nc)::value, decltype(Rc)::value, 2>;
                            if (tokens_per_cta == 2)
                                return launch_pdl(kern2, dim3(unsigned((a.n + 1) / 2)), dim3(kTokThreads), stream, a);
                            return launch_pdl(kern1, dim3(unsigned(a.n)), dim3(kTokThreads), stream, a);
                        });
                    });
                });
            });
        });
    });
}

}  // namespace kvq
