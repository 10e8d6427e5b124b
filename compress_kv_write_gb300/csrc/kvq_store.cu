// kvq_store.cu -- fused (K RMSNorm) + (RoPE) + block quantisation + paged
// scatter of new K rows: the store / store + RoPE / fused K norm + RoPE
// kernels of "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
// (section 1 store_row, and the store-latency table).
//
// Mapping: one warp per token row, TPW rows per warp loaded up front.  Lane l
// owns the 16-byte chunks l, l+32, ... of the row, so every warp-wide load
// and store instruction touches one contiguous span.  A 32-value quant block
// is LPB = 32 / (values per chunk) adjacent lanes (4 for bf16, 8 for fp32);
// its absmax is an unsigned max of |x| bits over those lanes with xor
// shuffles.  The block's scale bytes are gathered in shared memory and the
// scale row is written with one 16-byte store.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kStoreThreads = 128;
constexpr int kStoreWarps = kStoreThreads / 32;

struct StoreArgs {
    const uint8_t *x;
    int64_t n;
    int64_t row_stride_bytes;
    const void *loc;
    const float *w;
    float eps;
    const float *cs;
    int64_t cs_rows;
    const int32_t *pos;
    uint8_t *pool;
    int64_t pool_slots;
    int32_t *err;
};

template <bool kBf16>
__device__ __forceinline__ void unpack_chunk(const uint4 &r, float *v) {
    if constexpr (kBf16) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16_lo(w[i]);
            v[2 * i + 1] = bf16_hi(w[i]);
        }
    } else {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z);
        v[3] = __uint_as_float(r.w);
    }
}

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope, int TPW>
__global__ void __launch_bounds__(kStoreThreads) store_kernel(const StoreArgs a) {
    constexpr int E = kBf16 ? 8 : 4;          // values per 16-byte chunk
    constexpr int K = kD / E / 32;            // chunks per lane
    constexpr int LPB = kBlock / E;           // lanes per quant block
    constexpr int kRopeLane0 = kRopeStart / E - (K - 1) * 32;  // first rope lane of chunk K-1
    static_assert(kRopeLane0 >= 0 && kRopeLane0 < 32, "rope dims sit in the last chunk");
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;

    __shared__ __align__(16) uint8_t s_scale[kStoreWarps][kNBlk];

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int64_t t0 = (int64_t(blockIdx.x) * kStoreWarps + wid) * TPW;

    pdl_wait();

    // ---- issue every global load of this warp's rows first
    uint4 raw[TPW][K];
    int64_t slot[TPW];
    int32_t pos[TPW];
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        const int64_t t = t0 + j;
        slot[j] = -1;
        pos[j] = 0;
        if (t < a.n) {
            const uint8_t *row = a.x + t * a.row_stride_bytes;
#pragma unroll
            for (int k = 0; k < K; ++k) raw[j][k] = ld_stream_u4(row + (k * 32 + lane) * 16);
            slot[j] = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + t)
                             : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + t));
            if constexpr (kRope) pos[j] = __ldg(a.pos + t);
        }
    }
    float wreg[K][E];
    if constexpr (kNorm) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float4 *wp = reinterpret_cast<const float4 *>(a.w + (k * 32 + lane) * E);
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                float4 f = __ldg(wp + q);
                wreg[k][4 * q] = f.x;
                wreg[k][4 * q + 1] = f.y;
                wreg[k][4 * q + 2] = f.z;
                wreg[k][4 * q + 3] = f.w;
            }
        }
    }
    // cos / sin of this lane's rope pairs (pair index i0 .. i0 + E/2 - 1)
    float cosv[TPW][E / 2], sinv[TPW][E / 2];
    bool pos_ok[TPW];
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        pos_ok[j] = true;
        if constexpr (kRope) {
            pos_ok[j] = pos[j] >= 0 && int64_t(pos[j]) < a.cs_rows;
            if (slot[j] >= 0 && pos_ok[j] && lane >= kRopeLane0) {
                const int i0 = ((K - 1) * 32 + lane) * E / 2 - kRopeStart / 2;
                const float *cs = a.cs + int64_t(pos[j]) * kRopeD;
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    cosv[j][q] = __ldg(cs + i0 + q);
                    sinv[j][q] = __ldg(cs + kRopeD / 2 + i0 + q);
                }
            }
        }
    }
    pdl_trigger();

#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        const int64_t t = t0 + j;
        if (t >= a.n) break;
        if (slot[j] < 0 || slot[j] >= a.pool_slots) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_SLOT);
            continue;
        }
        if (!pos_ok[j]) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_POS);
            continue;
        }
        float v[K][E];
#pragma unroll
        for (int k = 0; k < K; ++k) unpack_chunk<kBf16>(raw[j][k], v[k]);

        if constexpr (kNorm) {
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) ss = fmaf(v[k][e], v[k][e], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float ms = ss * (1.0f / kD);
            const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) v[k][e] = __fmul_rn(__fmul_rn(v[k][e], inv), wreg[k][e]);
        }
        if constexpr (kRope) {
            if (lane >= kRopeLane0) {
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    const float x0 = v[K - 1][2 * q], x1 = v[K - 1][2 * q + 1];
                    const float c = cosv[j][q], s = sinv[j][q];
                    v[K - 1][2 * q] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
                    v[K - 1][2 * q + 1] = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
                }
            }
        }
        if constexpr (kNorm || kRope) {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) v[k][e] = round_bf16(v[k][e]);
        }

        // ---- block absmax over LPB lanes
        uint32_t am[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            uint32_t m = 0;
#pragma unroll
            for (int e = 0; e < E; ++e) m = max(m, abs_bits(v[k][e]));
#pragma unroll
            for (int off = 1; off < LPB; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
            am[k] = m;
        }

        uint8_t *crow = PK::code_row(a.pool, slot[j]);
        uint8_t *srow = PK::scale_row(a.pool, slot[j]);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int c = k * 32 + lane;  // chunk index in the row
            uint32_t sbyte;
            if constexpr (L == Layout::V41) {
                sbyte = v41_scale_byte(am[k]);
                const float mult = v41_multiplier(sbyte);
                uint32_t wds[E / 4];
#pragma unroll
                for (int q = 0; q < E / 4; ++q) {
                    const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[k][4 * q], mult), __fmul_rn(v[k][4 * q + 1], mult));
                    const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[k][4 * q + 2], mult), __fmul_rn(v[k][4 * q + 3], mult));
                    wds[q] = lo | (hi << 16);
                }
                if constexpr (E == 8) {
                    *reinterpret_cast<uint2 *>(crow + c * 8) = make_uint2(wds[0], wds[1]);
                } else {
                    *reinterpret_cast<uint32_t *>(crow + c * 4) = wds[0];
                }
            } else {
                sbyte = fp4_scale_byte(am[k]);
                const float S = e4m3x2_to_f32x2(sbyte).x;
                const float inv = __frcp_rn(S);
                uint32_t word = 0;
                if (S != 0.0f) {
#pragma unroll
                    for (int q = 0; q < E / 2; ++q)
                        word |= cvt_e2m1x2(__fmul_rn(v[k][2 * q], inv), __fmul_rn(v[k][2 * q + 1], inv)) << (8 * q);
                }
                if constexpr (E == 8) {
                    *reinterpret_cast<uint32_t *>(crow + c * 4) = word;
                } else {
                    *reinterpret_cast<uint16_t *>(crow + c * 2) = uint16_t(word);
                }
            }
            if (lane % LPB == 0) s_scale[wid][c / LPB] = uint8_t(sbyte);
        }
        __syncwarp();
        if (lane == 0) st_u4(srow, *reinterpret_cast<const uint4 *>(s_scale[wid]));
        if constexpr (T::kScaleBytes == 32) {
            if (lane == 1) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
        }
        __syncwarp();
    }
}

template <Layout L, int PB, bool B16, bool L64, bool N, bool R>
kvq_status launch_store(const StoreArgs &a, cudaStream_t stream) {
    constexpr int TPW = 2;
    const int64_t warps = (a.n + TPW - 1) / TPW;
    const int64_t blocks = (warps + kStoreWarps - 1) / kStoreWarps;
    if (blocks > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    return launch_pdl(store_kernel<L, PB, B16, L64, N, R, TPW>, dim3(unsigned(blocks)),
                      dim3(kStoreThreads), stream, a);
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_store(kvq_layout layout, int page_bits, unsigned flags, const void *x,
                                kvq_dtype x_dtype, int64_t n, int64_t x_row_stride, const void *loc,
                                kvq_index_dtype loc_dtype, const float *norm_weight, float eps,
                                const float *cos_sin, int64_t cos_sin_rows, const int32_t *pos,
                                uint8_t *pool, int64_t pool_slots, int32_t *err,
                                struct CUstream_st *stream) {
    kvq_status st = check_pool(layout, page_bits, pool, pool_slots);
    if (st != KVQ_OK) return st;
    if (flags & ~unsigned(KVQ_FLAG_ROPE | KVQ_FLAG_NORM)) return KVQ_ERR_INVALID_ARG;
    if (x_dtype != KVQ_F32 && x_dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
    if (loc_dtype != KVQ_I32 && loc_dtype != KVQ_I64) return KVQ_ERR_INVALID_ARG;
    if (n < 0) return KVQ_ERR_INVALID_ARG;
    const int64_t esz = x_dtype == KVQ_F32 ? 4 : 2;
    if (!x || !aligned(x, 16) || x_row_stride < kD || (x_row_stride * esz) % 16 != 0)
        return KVQ_ERR_INVALID_ARG;
    if (!loc || !aligned(loc, loc_dtype == KVQ_I64 ? 8 : 4)) return KVQ_ERR_INVALID_ARG;
    const bool norm = flags & KVQ_FLAG_NORM, rope = flags & KVQ_FLAG_ROPE;
    if (norm && (!norm_weight || !aligned(norm_weight, 16))) return KVQ_ERR_INVALID_ARG;
    if (rope && (!cos_sin || !aligned(cos_sin, 16) || cos_sin_rows <= 0 || !pos || !aligned(pos, 4)))
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;

    StoreArgs a;
    a.x = static_cast<const uint8_t *>(x);
    a.n = n;
    a.row_stride_bytes = x_row_stride * esz;
    a.loc = loc;
    a.w = norm_weight;
    a.eps = eps;
    a.cs = cos_sin;
    a.cs_rows = cos_sin_rows;
    a.pos = pos;
    a.pool = pool;
    a.pool_slots = pool_slots;
    a.err = err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return with_bool(x_dtype == KVQ_BF16, [&](auto B16) {
                return with_bool(loc_dtype == KVQ_I64, [&](auto L64) {
                    return with_bool(norm, [&](auto Nc) {
                        return with_bool(rope, [&](auto Rc) {
                            return launch_store<decltype(Lc)::value, decltype(PBc)::value,
                                                decltype(B16)::value, decltype(L64)::value,
                                                decltype(Nc)::value, decltype(Rc)::value>(a, s);
                        });
                    });
                });
            });
        });
    });
}
