// kvq_store.cu -- fused (K RMSNorm) + (RoPE) + block quantisation + paged
// scatter of new K rows: the store / store + RoPE / fused K norm + RoPE
// kernels of "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
// (section 1 store_row, and the store-latency table).
//
// Design (HBM-bound streaming, one pass):
//  * Persistent CTAs, as many as are resident at once; CTA b owns the
//    contiguous token range [n*b/G, n*(b+1)/G).
//  * A producer warp streams each token's 512-value row (and, with RoPE,
//    its 256-byte cos/sin row) into a ring of S shared-memory slots with 1-D
//    bulk async copies that complete on the slot's "full" mbarrier.  Lane l
//    owns slots l, l+32, ...; it prefetches the next token's slot index and
//    position while the current copies are in flight.
//  * Eight consumer warps take tokens round-robin.  A consumer reads its row
//    out of the slot (lane l: 16-byte chunks l, l+32, ... -- conflict-free),
//    frees the slot on its "empty" mbarrier, then computes in registers and
//    writes the codes with coalesced stores (every warp store instruction
//    covers one contiguous span of the code row) and the scale row with one
//    16-byte store.
//  * A 32-value quant block is LPB = 32 / (values per chunk) adjacent lanes
//    (4 for bf16 rows, 8 for fp32); its absmax is a max of |x| over the
//    lane's values and an xor-shuffle over those lanes.
//  * Every mbarrier wait is bounded (2 s); a wait that runs out sets
//    KVQ_DEVERR_TIMEOUT and the warp stops.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kConsumers = 8;
constexpr int kStoreThreads = (kConsumers + 1) * 32;

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

template <bool kBf16, bool kRope>
struct StoreSmem {
    static constexpr int XB = kD * (kBf16 ? 2 : 4);   // input row bytes
    static constexpr int CSB = kRope ? kRopeD * 4 : 0;  // cos/sin row bytes
    static constexpr int S = kBf16 ? 64 : 32;          // ring slots
    static_assert(S % 32 == 0, "each producer lane owns whole slots");
    static constexpr int kX = 0;
    static constexpr int kCs = kX + S * XB;
    static constexpr int kLoc = kCs + S * CSB;
    static constexpr int kFlag = kLoc + S * 8;
    static constexpr int kFull = kFlag + S * 4;
    static constexpr int kEmpty = kFull + S * 8;
    static constexpr int kScale = kEmpty + S * 8;
    static constexpr int kBytes = kScale + kConsumers * kNBlk;
    static_assert(kCs % 16 == 0 && kLoc % 16 == 0 && kFull % 8 == 0, "aligned smem regions");
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

// Quantise one token held as v[K][E] (lane's chunks k*32 + lane) and write it.
template <Layout L, int PageBits, int E, int K>
__device__ __forceinline__ void encode_store(float (&v)[K][E], int64_t slot, uint8_t *pool,
                                             uint8_t *scale_scratch, int lane) {
    constexpr int LPB = kBlock / E;
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    float am[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) m = fmaxf(m, fabsf(v[k][e]));
#pragma unroll
        for (int off = 1; off < LPB; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        am[k] = m;
    }
    uint8_t *crow = PK::code_row(pool, slot);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * 32 + lane;  // chunk index in the row
        uint32_t sbyte;
        if constexpr (L == Layout::V41) {
            sbyte = v41_scale_byte(__float_as_uint(am[k]));
            const float mult = v41_multiplier(sbyte);
            uint32_t wds[E / 4];
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                const float2 a = fmul2(make_float2(v[k][4 * q], v[k][4 * q + 1]), make_float2(mult, mult));
                const float2 b = fmul2(make_float2(v[k][4 * q + 2], v[k][4 * q + 3]), make_float2(mult, mult));
                wds[q] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
            }
            if constexpr (E == 8) {
                *reinterpret_cast<uint2 *>(crow + c * 8) = make_uint2(wds[0], wds[1]);
            } else {
                *reinterpret_cast<uint32_t *>(crow + c * 4) = wds[0];
            }
        } else {
            sbyte = fp4_scale_byte(__float_as_uint(am[k]));
            const float S = e4m3x2_to_f32x2(sbyte).x;
            const float inv = __frcp_rn(S);
            uint32_t word = 0;
            if (S != 0.0f) {
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    const float2 a = fmul2(make_float2(v[k][2 * q], v[k][2 * q + 1]), make_float2(inv, inv));
                    word |= cvt_e2m1x2(a.x, a.y) << (8 * q);
                }
            }
            if constexpr (E == 8) {
                *reinterpret_cast<uint32_t *>(crow + c * 4) = word;
            } else {
                *reinterpret_cast<uint16_t *>(crow + c * 2) = uint16_t(word);
            }
        }
        if (lane % LPB == 0) scale_scratch[c / LPB] = uint8_t(sbyte);
    }
    __syncwarp();
    uint8_t *srow = PK::scale_row(pool, slot);
    if (lane == 0) st_u4(srow, *reinterpret_cast<const uint4 *>(scale_scratch));
    if constexpr (T::kScaleBytes == 32) {
        if (lane == 1) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
    }
    __syncwarp();
}

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope>
__global__ void __launch_bounds__(kStoreThreads, 2) store_kernel(const StoreArgs a) {
    using SM = StoreSmem<kBf16, kRope>;
    constexpr int S = SM::S;
    constexpr int E = kBf16 ? 8 : 4;          // values per 16-byte chunk
    constexpr int K = kD / E / 32;            // chunks per lane
    constexpr int kRopeLane0 = kRopeStart / E - (K - 1) * 32;  // first rope lane of chunk K-1
    static_assert(kRopeLane0 >= 0 && kRopeLane0 < 32, "rope dims sit in the last chunk");

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *s_x = smem + SM::kX;
    float *s_cs = reinterpret_cast<float *>(smem + SM::kCs);
    int64_t *s_loc = reinterpret_cast<int64_t *>(smem + SM::kLoc);
    int32_t *s_flag = reinterpret_cast<int32_t *>(smem + SM::kFlag);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::kFull);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + SM::kEmpty);
    uint8_t *s_scale = smem + SM::kScale;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t start = a.n * int64_t(blockIdx.x) / G;
    const int cnt = int(a.n * (int64_t(blockIdx.x) + 1) / G - start);

    if (threadIdx.x < S) {
        mbar_init(&full[threadIdx.x], 1);
        mbar_init(&empty[threadIdx.x], 1);
    }
    fence_mbar_init();
    __syncthreads();
    pdl_wait();

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        int64_t lc = 0;
        int32_t p = 0;
        if (lane < cnt) {
            lc = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + start + lane)
                        : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + start + lane));
            if constexpr (kRope) p = __ldg(a.pos + start + lane);
        }
        bool ok = true;
        int i = lane;
        for (; i < cnt; i += 32) {
            const int64_t lc_cur = lc;
            const int32_t p_cur = p;
            if (i + 32 < cnt) {  // prefetch the next token's slot index and position
                lc = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + start + i + 32)
                            : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + start + i + 32));
                if constexpr (kRope) p = __ldg(a.pos + start + i + 32);
            }
            const int s = i % S;
            const uint32_t r = uint32_t(i / S);
            if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1u)) {
                raise_err(a.err, KVQ_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            mbar_expect_tx(&full[s], SM::XB);
            bulk_g2s(s_x + s * SM::XB, a.x + (start + i) * a.row_stride_bytes, SM::XB, &full[s]);
            int32_t flag = 0;
            if constexpr (kRope) {
                if (p_cur >= 0 && int64_t(p_cur) < a.cs_rows) {
                    mbar_expect_tx(&full[s], SM::CSB);
                    bulk_g2s(s_cs + s * kRopeD, a.cs + int64_t(p_cur) * kRopeD, SM::CSB, &full[s]);
                } else {
                    flag = 1;
                }
            }
            s_loc[s] = lc_cur;
            s_flag[s] = flag;
            mbar_arrive(&full[s]);
        }
        pdl_trigger();
        // drain: the last copies issued into this lane's slots have landed
        // before the CTA (and its shared memory) can go away
        for (int j = i - 32; j >= 0 && j >= i - S; j -= 32) {
            if (!mbar_wait(&full[j % S], uint32_t(j / S) & 1u)) {
                if (ok) raise_err(a.err, KVQ_DEVERR_TIMEOUT);
                break;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    float wreg[K][E];
    if constexpr (kNorm) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float4 *wp = reinterpret_cast<const float4 *>(a.w + (k * 32 + lane) * E);
#pragma unroll
            for (int q = 0; q < E / 4; ++q) {
                const float4 f = __ldg(wp + q);
                wreg[k][4 * q] = f.x;
                wreg[k][4 * q + 1] = f.y;
                wreg[k][4 * q + 2] = f.z;
                wreg[k][4 * q + 3] = f.w;
            }
        }
    }
    uint8_t *scratch = s_scale + warp * kNBlk;

    for (int i = warp; i < cnt; i += kConsumers) {
        const int s = i % S;
        const bool got = mbar_wait(&full[s], uint32_t(i / S) & 1u);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_TIMEOUT);
            break;
        }
        uint4 raw[K];
        const uint8_t *xs = s_x + s * SM::XB;
#pragma unroll
        for (int k = 0; k < K; ++k) raw[k] = lds_u4(xs + (k * 32 + lane) * 16);
        float cosv[E / 2], sinv[E / 2];
        if constexpr (kRope) {
            if (lane >= kRopeLane0) {
                const int i0 = ((K - 1) * 32 + lane) * E / 2 - kRopeStart / 2;
                const float *cs = s_cs + s * kRopeD;
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    cosv[q] = cs[i0 + q];
                    sinv[q] = cs[kRopeD / 2 + i0 + q];
                }
            }
        }
        const int64_t slot = s_loc[s];
        const int32_t flag = s_flag[s];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the slot is free again

        if (flag) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_POS);
            continue;
        }
        if (slot < 0 || slot >= a.pool_slots) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_SLOT);
            continue;
        }

        float v[K][E];
#pragma unroll
        for (int k = 0; k < K; ++k) unpack_chunk<kBf16>(raw[k], v[k]);

        if constexpr (kNorm) {
            float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float2 t = make_float2(v[k][e], v[k][e + 1]);
                    ss2 = ffma2(t, t, ss2);
                }
            float ss = ss2.x + ss2.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float ms = ss * (1.0f / kD);
            const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    float2 t = fmul2(make_float2(v[k][e], v[k][e + 1]), make_float2(inv, inv));
                    t = fmul2(t, make_float2(wreg[k][e], wreg[k][e + 1]));
                    v[k][e] = t.x;
                    v[k][e + 1] = t.y;
                }
        }
        if constexpr (kRope) {
            if (lane >= kRopeLane0) {
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    const float x0 = v[K - 1][2 * q], x1 = v[K - 1][2 * q + 1];
                    const float c = cosv[q], sn = sinv[q];
                    v[K - 1][2 * q] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
                    v[K - 1][2 * q + 1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
                }
            }
        }
        if constexpr (kNorm || kRope) {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const uint32_t b = pack_bf16x2(v[k][e], v[k][e + 1]);
                    v[k][e] = bf16_lo(b);
                    v[k][e + 1] = bf16_hi(b);
                }
        }
        encode_store<L, PageBits, E, K>(v, slot, a.pool, scratch, lane);
    }
}

template <Layout L, int PB, bool B16, bool L64, bool N, bool R>
kvq_status launch_store(const StoreArgs &a, cudaStream_t stream) {
    constexpr auto kern = store_kernel<L, PB, B16, L64, N, R>;
    constexpr size_t smem = StoreSmem<B16, R>::kBytes;
    int64_t cap = 0;
    kvq_status st = resident_grid<kern>(kStoreThreads, smem, &cap);
    if (st != KVQ_OK) return st;
    const int64_t grid = a.n < cap ? a.n : cap;
    return launch_pdl_smem(kern, dim3(unsigned(grid)), dim3(kStoreThreads), smem, stream, a);
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
    if (n < 0 || n > (int64_t(1) << 40)) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;  // nothing to enqueue; x / loc may be empty (null)
    const int64_t esz = x_dtype == KVQ_F32 ? 4 : 2;
    if (!x || !aligned(x, 16) || x_row_stride < kD || (x_row_stride * esz) % 16 != 0)
        return KVQ_ERR_INVALID_ARG;
    if (!loc || !aligned(loc, loc_dtype == KVQ_I64 ? 8 : 4)) return KVQ_ERR_INVALID_ARG;
    const bool norm = flags & KVQ_FLAG_NORM, rope = flags & KVQ_FLAG_ROPE;
    if (norm && (!norm_weight || !aligned(norm_weight, 16))) return KVQ_ERR_INVALID_ARG;
    if (rope && (!cos_sin || !aligned(cos_sin, 16) || cos_sin_rows <= 0 || !pos || !aligned(pos, 4)))
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;

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
