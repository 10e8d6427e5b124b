// kvq_store.cu -- fused (K RMSNorm) + (RoPE) + block quantisation + paged
// scatter of new K rows: the store / store + RoPE / fused K norm + RoPE
// kernels of "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
// (section 1 store_row, and the store-latency table), for both layouts.
//
// Small batches (up to 1024-3072 tokens by instance) take one four-warp CTA
// per token or per two tokens (kvq_store_small.cu).  Larger ones take one of
// two persistent kernels that share the structure below and differ in how a
// token maps onto lanes (launch_store says which instance and batch size
// uses which, and why):
//
//  * store_warp_kernel: one warp per token.  Lane l owns the 16-byte chunks
//    l, l+32, ... of the row, so every warp load / store instruction covers
//    one contiguous span; a 32-value quant block is 32/(values per chunk)
//    adjacent lanes, reduced with xor shuffles.  Each lane copies and reads
//    back only its own chunks: no cross-lane waits.  With RoPE a token's
//    cos/sin values are a second commit group, so that everything but the
//    rotated chunk is finished while they land.
//  * store_half_kernel: two tokens per warp; half-warp h holds token 2k+h
//    and lane i of the half owns quant block i, so a block's absmax needs no
//    shuffle and its scale (V41 exponent byte, or FP4 e4m3 scale with its
//    correctly rounded division and reciprocal) is computed once.  With
//    RoPE the 64 rotated dims (the last two blocks) are spread over all 16
//    lanes instead: lane i rotates the quad of dims 448+4i .. 448+4i+3, the
//    two rotated blocks' absmax is an 8-lane shuffle reduction, and lanes 14
//    and 15 own no whole block.  Rows land block-swizzled in shared memory
//    so that the block-per-lane reads are bank-conflict-free; a V41 block's
//    32 code bytes leave in one 32-byte store per lane.
//
// Shared structure: persistent CTAs (as many as are resident at once); warp
// w owns a contiguous token range computed on the host (partition) and keeps
// its next rows in flight in a per-warp shared-memory ring filled with
// cp.async.  Before the PDL wait each warp prefetches into L2 the rows it
// requests first.  Slot indices and positions of 32 tokens sit one per lane, validated
// once, and are fetched with a shuffle.  Math is fp32; the products of the
// RMSNorm and of the rotation are rounded one by one, as in the definition.
#include "kvq_store.cuh"

namespace kvq {
namespace {

// Token range [start, start + cnt) of warp gw (see StoreArgs).
__device__ __forceinline__ void token_range(const StoreArgs &a, int64_t gw, int64_t &start, int &cnt) {
    const int64_t e1 = a.extra + a.skew, w2 = a.warps - a.skew;
    start = gw * a.per_warp + (gw < e1 ? gw : e1) - (gw > w2 ? gw - w2 : 0);
    cnt = int(a.per_warp) + (gw < e1 ? 1 : 0) - (gw >= w2 ? 1 : 0);
}

// 16-byte chunk position of (block, sub-chunk) inside a row: the sub-chunks
// of a block are rotated so that eight lanes reading sub-chunk j of eight
// consecutive blocks hit eight different bank groups.
template <int SUBS>
__device__ __forceinline__ int swz(int blk, int sub) {
    const int rot = SUBS == 4 ? (blk >> 1) : blk;
    return blk * SUBS + ((sub + rot) & (SUBS - 1));
}

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

template <bool kBf16, bool kRope, int kDepth = 3>
struct WarpStoreSmem {
    static constexpr int XB = kD * (kBf16 ? 2 : 4);    // input row bytes
    static constexpr int CSB = kRope ? kRopeD * 4 : 0;  // this token's cos/sin values
    static constexpr int D = kDepth;                    // tokens in flight per warp
    static constexpr int NS = 4;                        // ring slots per warp (a power of two)
    static_assert((NS & (NS - 1)) == 0 && NS > D, "ring index by mask; a free slot to refill");
    static constexpr int SLOT = XB + CSB;
    static constexpr int kWarpBytes = NS * SLOT;
    static_assert(SLOT % 16 == 0 && kWarpBytes % 16 == 0, "16-byte aligned slots");
};

// Code row and scale row of slot `slot` (validated, < 2^31).
template <Layout L, int PageBits>
__device__ __forceinline__ void row_ptrs(int32_t slot, uint8_t *pool, uint8_t *&crow, uint8_t *&srow) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    uint8_t *page = pool + int64_t(slot >> PageBits) * PK::kPageBytes;
    const int row = slot & int(PK::kPage - 1);
    crow = page + row * T::kCodeBytes;
    srow = page + PK::kPage * T::kCodeBytes + row * T::kScaleBytes;
}

// Block absmax of chunks K0 .. K1-1 of one token held as v[K][E] (lane's
// chunks k*32 + lane): a quant block spans kBlock / E adjacent lanes.
template <int E, int K, int K0, int K1>
__device__ __forceinline__ void block_amax(float (&v)[K][E], float (&am)[K]) {
    constexpr int LPB = kBlock / E;
#pragma unroll
    for (int k = K0; k < K1; ++k) {
        float mm;
        if constexpr (E == 8) {
            const float t0 = fmax3(fabsf(v[k][0]), fabsf(v[k][1]), fabsf(v[k][2]));
            const float t1 = fmax3(fabsf(v[k][3]), fabsf(v[k][4]), fabsf(v[k][5]));
            mm = fmax3(t0, t1, fmaxf(fabsf(v[k][6]), fabsf(v[k][7])));
        } else {
            mm = fmaxf(fmax3(fabsf(v[k][0]), fabsf(v[k][1]), fabsf(v[k][2])), fabsf(v[k][3]));
        }
#pragma unroll
        for (int off = 1; off < LPB; off <<= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
        am[k] = mm;
    }
}

// Quantise chunks K0 .. K1-1 with their block absmax into the token's V41
// code row and scale row.  The lane that leads a quant block writes its
// scale byte.
template <Layout L, int E, int K, int K0, int K1>
__device__ __forceinline__ void quant_store(float (&v)[K][E], const float (&am)[K], uint8_t *crow, uint8_t *srow,
                                            int lane) {
    static_assert(L == Layout::V41, "the one-warp-per-token mapping serves V41 only");
    constexpr int LPB = kBlock / E;
#pragma unroll
    for (int k = K0; k < K1; ++k) {
        const int c = k * 32 + lane;  // chunk index in the row
        const uint32_t sbyte = v41_scale_byte(__float_as_uint(am[k]));
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
        if (lane % LPB == 0) srow[c / LPB] = uint8_t(sbyte);
    }
}

// Round v[k] to bf16 (ties to even), in place, for chunks K0 .. K1-1.
template <int E, int K, int K0, int K1>
__device__ __forceinline__ void round_chunks(float (&v)[K][E]) {
#pragma unroll
    for (int kk = K0; kk < K1; ++kk)
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const uint32_t b = pack_bf16x2(v[kk][e], v[kk][e + 1]);
            v[kk][e] = bf16_lo(b);
            v[kk][e + 1] = bf16_hi(b);
        }
}

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope, int kWarps, int kDepth = 3>
__global__ void __launch_bounds__(32 * kWarps, 32 / kWarps) store_warp_kernel(const StoreArgs a) {
    using SM = WarpStoreSmem<kBf16, kRope, kDepth>;
    constexpr int D = SM::D, NS = SM::NS;
    constexpr int E = kBf16 ? 8 : 4;          // values per 16-byte chunk
    constexpr int K = kD / E / 32;            // chunks per lane
    constexpr int kRopeLane0 = kRopeStart / E - (K - 1) * 32;  // first rope lane of chunk K-1
    static_assert(kRopeLane0 >= 0 && kRopeLane0 < 32, "rope dims sit in the last chunk");
    static_assert((32 - kRopeLane0) * E * 4 == SM::CSB || !kRope, "rope lanes fill the cos/sin area");
    static_assert(D < 32, "a token's slot index is in the current or the next batch of 32");

    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t wsm = smem_addr(smem) + warp * SM::kWarpBytes;  // this warp's ring (shared window)
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    int64_t start;
    int cnt;
    token_range(a, gw, start, cnt);

    // While the upstream grid drains: pull this warp's first rows and its
    // slot / position lines into L2 (hints only; the loads come after the
    // wait).  Only the rows requested first: more compete with the upstream
    // grid's tail (measured at 16384 tokens: norm + RoPE 6.46 us with four
    // rows, 6.06 with its two in flight; the plain store 4.82 with four,
    // 4.77 with one).
    constexpr int kPrefetchRows = kRope ? D : 1;
    if (lane < cnt && lane < kPrefetchRows) prefetch_l2_bulk(a.x + (start + lane) * a.row_stride_bytes, SM::XB);
    if (lane == 0 && cnt > 0) {
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + start)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + start));
        if constexpr (kRope) prefetch_l2(a.pos + start);
    }
    pdl_wait();

    // Without RoPE the rows of the first D tokens are requested before the
    // slot loads (which are waited for only when first used); with RoPE the
    // first copies wait for the positions (measured at 16384 tokens: each
    // order is the faster one for its instance).
    const uint8_t *src_next = a.x + start * a.row_stride_bytes + lane * 16;
    int ring_in = 0;
    if constexpr (!kRope) {
#pragma unroll
        for (int j = 0; j < D; ++j) {
            if (j < cnt) {
                const uint32_t slot = wsm + ring_in * SM::SLOT + lane * 16;
#pragma unroll
                for (int k = 0; k < K; ++k) cp_async16(slot + k * 512, src_next + k * 512);
                src_next += a.row_stride_bytes;
                ring_in = (ring_in + 1) & (NS - 1);
            }
            cp_async_commit();
        }
    }

    // Slot / position of tokens 32b .. 32b+31 of this warp, one per lane,
    // validated once: an out-of-range slot or position becomes -1.
    auto ld_slot = [&](int j) -> int32_t {
        const int64_t s = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + start + j)
                                 : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + start + j));
        return (s >= 0 && s < a.pool_slots) ? int32_t(s) : -1;
    };
    auto ld_pos = [&](int j) -> int32_t {
        const int32_t p = __ldg(a.pos + start + j);
        return (p >= 0 && int64_t(p) < a.cs_rows) ? p : -1;
    };
    int32_t sl_cur = -1, sl_nxt = -1, p_cur = -1, p_nxt = -1;
    if (lane < cnt) {
        sl_cur = ld_slot(lane);
        if constexpr (kRope) p_cur = ld_pos(lane);
    }
    if (32 + lane < cnt) {
        sl_nxt = ld_slot(32 + lane);
        if constexpr (kRope) p_nxt = ld_pos(32 + lane);
    }
    int cur_b = 0;

    // Copies of token j into the next ring slot: one commit group for the
    // row and, with RoPE, a second one for its cos/sin values (which wait on
    // the position), so the rest of the row can be finished while they land.
    auto issue = [&](int j) {
        if (j < cnt) {
            const uint32_t slot = wsm + ring_in * SM::SLOT + lane * 16;
#pragma unroll
            for (int k = 0; k < K; ++k) cp_async16(slot + k * 512, src_next + k * 512);
            if constexpr (kRope) {
                cp_async_commit();
                const int32_t pj = __shfl_sync(0xffffffffu, (j >> 5) == cur_b ? p_cur : p_nxt, j & 31);
                if (lane >= kRopeLane0 && pj >= 0) {
                    const int i0 = ((K - 1) * 32 + lane) * E / 2 - kRopeStart / 2;
                    const float *cs = a.cs + int64_t(pj) * kRopeD;
                    const uint32_t dst = wsm + ring_in * SM::SLOT + SM::XB + (lane - kRopeLane0) * E * 4;
                    if constexpr (E == 8) {
                        cp_async16(dst, cs + i0);
                        cp_async16(dst + 16, cs + kRopeD / 2 + i0);
                    } else {
                        cp_async8(dst, cs + i0);
                        cp_async8(dst + 8, cs + kRopeD / 2 + i0);
                    }
                }
            }
            src_next += a.row_stride_bytes;
            ring_in = (ring_in + 1) & (NS - 1);
        } else if constexpr (kRope) {
            cp_async_commit();  // keep two groups per token
        }
        cp_async_commit();
    };
    // groups committed per token, and the waits for token k's row and cos/sin
    constexpr int kGroups = kRope ? 2 : 1;

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

    if (kRope && cnt > 1) {
        // Let the first row land before asking for the next ones: every warp
        // starts at once, and behind the position -> cos/sin chain the first
        // row is what holds the warp up.  Warps with a single token are
        // faster without the wait.
        issue(0);
        pdl_trigger();
        cp_async_wait<kGroups - 1>();
#pragma unroll
        for (int j = 1; j < D; ++j) issue(j);
    } else if constexpr (kRope) {
#pragma unroll
        for (int j = 0; j < D; ++j) issue(j);
        pdl_trigger();
    } else {
        pdl_trigger();  // the first rows went out above
    }

    int ring_out = 0;
    for (int k = 0; k < cnt; ++k) {
        if ((k & 31) == 0 && k > 0) {  // next batch of slots / positions
            sl_cur = sl_nxt;
            p_cur = p_nxt;
            cur_b = k >> 5;
            if (k + 32 + lane < cnt) {
                sl_nxt = ld_slot(k + 32 + lane);
                if constexpr (kRope) p_nxt = ld_pos(k + 32 + lane);
            }
        }
        // Token k's row has landed once at most kGroups * D - 1 groups are pending.
        cp_async_wait<kGroups * D - 1>();
        const uint32_t slot_sm = wsm + ring_out * SM::SLOT;
        ring_out = (ring_out + 1) & (NS - 1);
        uint4 raw[K];
#pragma unroll
        for (int kk = 0; kk < K; ++kk) raw[kk] = lds_u4(slot_sm + (kk * 32 + lane) * 16);
        const int32_t slot = __shfl_sync(0xffffffffu, sl_cur, k & 31);
        int32_t pk = 0;
        if constexpr (kRope) pk = __shfl_sync(0xffffffffu, p_cur, k & 31);
        issue(k + D);  // refill the ring while this token is computed

        if (kRope && pk < 0) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_POS);
            continue;
        }
        if (slot < 0) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_SLOT);
            continue;
        }

        float v[K][E];
#pragma unroll
        for (int kk = 0; kk < K; ++kk) unpack_chunk<kBf16>(raw[kk], v[kk]);

        if constexpr (kNorm) {
            // four independent partial sums (short dependency chains)
            float2 ss2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int kk = 0; kk < K; ++kk)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float2 t = make_float2(v[kk][e], v[kk][e + 1]);
                    const int j = (kk * E / 2 + e / 2) & 3;
                    ss2[j] = ffma2(t, t, ss2[j]);
                }
            const float2 s4 = fadd2(fadd2(ss2[0], ss2[1]), fadd2(ss2[2], ss2[3]));
            float ss = s4.x + s4.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float ms = ss * (1.0f / kD);
            const float inv = rsqrt_approx(__fadd_rn(ms, a.eps));
#pragma unroll
            for (int kk = 0; kk < K; ++kk)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    float2 t = fmul2(make_float2(v[kk][e], v[kk][e + 1]), make_float2(inv, inv));
                    t = fmul2(t, make_float2(wreg[kk][e], wreg[kk][e + 1]));
                    v[kk][e] = t.x;
                    v[kk][e + 1] = t.y;
                }
        }
        uint8_t *crow, *srow;
        float am[K];
        if constexpr (kRope) {
            // Chunks before the rotated one are final: round and store them
            // while this token's cos/sin copies land.
            if constexpr (kNorm || !kBf16) round_chunks<E, K, 0, K - 1>(v);
            block_amax<E, K, 0, K - 1>(v, am);
            row_ptrs<L, PageBits>(slot, a.pool, crow, srow);
            quant_store<L, E, K, 0, K - 1>(v, am, crow, srow, lane);
            cp_async_wait<2 * D>();  // ... and its cos/sin values (two groups were added since)
            if (lane >= kRopeLane0) {
                float cosv[E / 2], sinv[E / 2];
                const uint32_t cs = slot_sm + SM::XB + (lane - kRopeLane0) * E * 4;
                if constexpr (E == 8) {
                    const uint4 c4 = lds_u4(cs), s4 = lds_u4(cs + 16);
                    cosv[0] = __uint_as_float(c4.x), cosv[1] = __uint_as_float(c4.y);
                    cosv[2] = __uint_as_float(c4.z), cosv[3] = __uint_as_float(c4.w);
                    sinv[0] = __uint_as_float(s4.x), sinv[1] = __uint_as_float(s4.y);
                    sinv[2] = __uint_as_float(s4.z), sinv[3] = __uint_as_float(s4.w);
                } else {
                    const uint2 c2 = lds_u2(cs), s2 = lds_u2(cs + 8);
                    cosv[0] = __uint_as_float(c2.x), cosv[1] = __uint_as_float(c2.y);
                    sinv[0] = __uint_as_float(s2.x), sinv[1] = __uint_as_float(s2.y);
                }
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    const float x0 = v[K - 1][2 * q], x1 = v[K - 1][2 * q + 1];
                    const float c = cosv[q], sn = sinv[q];
                    v[K - 1][2 * q] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
                    v[K - 1][2 * q + 1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
                }
                // bf16 input without norm: only the rotated values left the bf16 grid
                if constexpr (!kNorm && kBf16) round_chunks<E, K, K - 1, K>(v);
            }
            if constexpr (kNorm || !kBf16) round_chunks<E, K, K - 1, K>(v);
            block_amax<E, K, K - 1, K>(v, am);
            quant_store<L, E, K, K - 1, K>(v, am, crow, srow, lane);
        } else {
            if constexpr (kNorm) round_chunks<E, K, 0, K>(v);
            block_amax<E, K, 0, K>(v, am);
            row_ptrs<L, PageBits>(slot, a.pool, crow, srow);
            quant_store<L, E, K, 0, K>(v, am, crow, srow, lane);
        }
    }
    cp_async_wait<0>();
}

// Round v[0..N) to bf16 (ties to even), in place.
template <int N>
__device__ __forceinline__ void round_bf16_n(float *v) {
#pragma unroll
    for (int e = 0; e < N; e += 2) {
        const uint32_t b = pack_bf16x2(v[e], v[e + 1]);
        v[e] = bf16_lo(b);
        v[e + 1] = bf16_hi(b);
    }
}

// max |v[i]| over 32 values (three-operand max: 16 instructions).
__device__ __forceinline__ float amax32(const float *v) {
    float m[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float t = fmax3(fabsf(v[8 * q]), fabsf(v[8 * q + 1]), fabsf(v[8 * q + 2]));
        t = fmax3(t, fabsf(v[8 * q + 3]), fabsf(v[8 * q + 4]));
        t = fmax3(t, fabsf(v[8 * q + 5]), fabsf(v[8 * q + 6]));
        m[q] = fmaxf(t, fabsf(v[8 * q + 7]));
    }
    return fmaxf(fmax3(m[0], m[1], m[2]), m[3]);
}

// Four V41 codes of x * mult (mult = 2^(127 - byte)), low byte first.
__device__ __forceinline__ uint32_t v41_word(const float *x, float mult) {
    const float2 a = fmul2(make_float2(x[0], x[1]), make_float2(mult, mult));
    const float2 b = fmul2(make_float2(x[2], x[3]), make_float2(mult, mult));
    return cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
}

// Eight e2m1 codes of x * inv, low nibble first: four converted bytes
// packed into one word by a single mov.
__device__ __forceinline__ uint32_t fp4_word(const float *x, float inv) {
    float2 y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) y[q] = fmul2(make_float2(x[2 * q], x[2 * q + 1]), make_float2(inv, inv));
    uint32_t w;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(w)
        : "f"(y[0].x), "f"(y[0].y), "f"(y[1].x), "f"(y[1].y), "f"(y[2].x), "f"(y[2].y), "f"(y[3].x),
          "f"(y[3].y));
    return w;
}

// V41_FP4 block scale byte e4m3(fl(amax / 6)) with a two-FMA quotient in
// place of a correctly rounded division: the quotient can differ from the
// correctly rounded one in its last bit, but an exhaustive run over every
// positive finite fp32 amax on the GB300 found the e4m3 byte identical in all
// cases, so the stored scale is the one the definition gives.
__device__ __forceinline__ uint32_t fp4_scale_byte_fast(float amax) {
    const float c = __uint_as_float(0x3E2AAAABu);  // 1/6 rounded to nearest
    const float q0 = __fmul_rn(amax, c);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, 6.0f, amax), c, q0);
    return cvt_e4m3x2(q1, 0.0f) & 0xFFu;
}

template <Layout L, bool kBf16, bool kRope, bool kNorm>
struct StoreSmem {
    static constexpr int E = kBf16 ? 8 : 4;             // values per 16-byte chunk
    static constexpr int SUBS = kBlock / E;             // chunks per quant block
    static constexpr int CPR = kD / E;                  // chunks per row
    static constexpr int XB = kD * (kBf16 ? 2 : 4);     // row bytes
    static constexpr int CSB = kRope ? kRopeD * 4 : 0;  // cos/sin row bytes
    static constexpr int D = kBf16 ? 3 : 1;             // token pairs in flight per warp
    static constexpr int NS = D + 1;                    // ring slots per warp (a power of two)
    static_assert((NS & (NS - 1)) == 0, "ring index by mask");
    static constexpr int SLOT = 2 * XB + 2 * CSB;
    static constexpr int kWarpBytes = NS * SLOT;
    static constexpr int kWBytes = kNorm ? kD * 4 : 0;  // the norm weights, once per CTA
    static constexpr int kRcpBytes = L == Layout::FP4 ? 128 * 4 : 0;  // 1/scale per e4m3 scale byte
    static constexpr int bytes(int warps) { return kWBytes + kRcpBytes + warps * kWarpBytes; }
    static_assert(SLOT % 16 == 0, "16-byte aligned slots");
    static_assert((2 * CPR) % 32 == 0, "a pair is whole chunks per lane");
};

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope, int kWarps>
__global__ void __launch_bounds__(32 * kWarps, 16 / kWarps) store_half_kernel(const StoreArgs a) {
    using SM = StoreSmem<L, kBf16, kRope, kNorm>;
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int D = SM::D, NS = SM::NS, E = SM::E, SUBS = SM::SUBS, CPR = SM::CPR;
    constexpr int NC = 2 * CPR / 32;                 // chunks each lane copies per pair
    constexpr int kRopeBlk0 = kRopeStart / kBlock;   // first rotated block (14)
    constexpr int kOwn = kRope ? kRopeBlk0 : kNBlk;  // lanes that own a whole block
    static_assert(kRopeD == 2 * kBlock && kRopeD / 4 == 16, "the rotated dims are 16 quads, two blocks");
    static_assert(D < 16, "a pair's slot index is in the current or the next batch of 32");
    // values after the fp32 math are rounded to bf16; a bf16 row without the
    // norm keeps its (already bf16) non-rotated values as they are
    constexpr bool kRoundBlk = kNorm || (kRope && !kBf16);
    constexpr bool kRoundQuad = kNorm || kRope;

    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h = lane >> 4;   // token of the pair
    const int bi = lane & 15;  // quant block owned (and, with RoPE, rotated quad)
    const float *s_w = reinterpret_cast<const float *>(smem);
    float *s_rcp = reinterpret_cast<float *>(smem + SM::kWBytes);
    const uint32_t wsm = smem_addr(smem) + SM::kWBytes + SM::kRcpBytes + warp * SM::kWarpBytes;  // this warp's ring
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    int64_t start;
    int cnt;
    token_range(a, gw, start, cnt);
    const int npairs = (cnt + 1) >> 1;
    // 32-byte code stores need a 32-byte aligned pool (the ABI asks for 16)
    const bool pool32 = (reinterpret_cast<uintptr_t>(a.pool) & 31) == 0;

    // While the upstream grid drains: L2 hints for this warp's first rows and
    // its slot / position lines (the loads come after the wait).  Two pairs;
    // one for FP4 with few tokens per warp, the whole ring with many.  More
    // compete with the upstream grid's tail (measured at 16384 tokens: store
    // + RoPE 5.55 us with four pairs, 5.09 with two; FP4 4.42 with four, 4.26
    // with two, 4.07 with one; FP4 at 32768 tokens: 8.2, 6.7 and 7.5 us); in
    // long launches (262144 tokens, 54-108 tokens per warp) four pairs gain
    // 1-2% over two.
    const int pf_rows = (L == Layout::FP4 && a.per_warp <= 5) ? 2 : a.per_warp >= 48 ? 2 * NS : 4;
    if (lane < cnt && lane < pf_rows) prefetch_l2_bulk(a.x + (start + lane) * a.row_stride_bytes, SM::XB);
    if (lane == 0 && cnt > 0) {
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + start)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + start));
        if constexpr (kRope) prefetch_l2(a.pos + start);
    }
    if constexpr (L == Layout::FP4) {
        // The correctly rounded reciprocal of every positive e4m3 scale (byte 0,
        // a zero scale, gives zero codes and is never read).
        for (int b = threadIdx.x; b < 128; b += 32 * kWarps) s_rcp[b] = __frcp_rn(e4m3x2_to_f32x2(b).x);
        if constexpr (kWarps > 1) {
            __syncthreads();
        } else {
            __syncwarp();
        }
    }
    pdl_wait();

    // With RoPE the first pair's rows go out before anything that could
    // stall the warp, and the pairs' cos/sin rows are commit groups of their
    // own (they wait on the positions), so that the non-rotated blocks are
    // finished while they land: kG groups per pair, rows then cos/sin.
    // Without RoPE the first pair is requested after the slot loads (both
    // orders measured at 16384 tokens: each is the faster one for its
    // instance).
    constexpr int kG = kRope ? 2 : 1;  // commit groups per pair
    int ring_in = 0;
    const uint8_t *xw = a.x + start * a.row_stride_bytes;  // this warp's first row
    auto issue_rows = [&](int p) {
        if (p < npairs) {
            const uint32_t slot = wsm + ring_in * SM::SLOT;
            const uint8_t *r0 = xw + int64_t(2 * p) * a.row_stride_bytes;
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                constexpr int kPerRow = CPR / 32;          // copy instructions per row
                const int r = m / kPerRow;                 // token of the pair (compile-time)
                const int cc = 32 * (m % kPerRow) + lane;  // chunk in the row
                if (2 * p + r < cnt)
                    cp_async16(slot + (r * CPR + swz<SUBS>(cc / SUBS, cc % SUBS)) * 16,
                               r0 + r * a.row_stride_bytes + cc * 16);
            }
            ring_in = (ring_in + 1) & (NS - 1);
        }
        cp_async_commit();
    };
    if constexpr (kRope) issue_rows(0);

    if constexpr (kNorm) {  // the weight row, block-swizzled like fp32 rows
        float *w = reinterpret_cast<float *>(smem);
        for (int c = threadIdx.x; c < kD / 4; c += 32 * kWarps)
            *reinterpret_cast<float4 *>(w + 4 * swz<8>(c >> 3, c & 7)) =
                __ldg(reinterpret_cast<const float4 *>(a.w) + c);
        if constexpr (kWarps > 1) {
            __syncthreads();
        } else {
            __syncwarp();
        }
    }

    // Slot / position of tokens 32b .. 32b+31 of this warp, one per lane,
    // validated once: an out-of-range slot or position becomes -1.
    auto ld_slot = [&](int j) -> int32_t {
        const int64_t s = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + start + j)
                                 : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + start + j));
        return (s >= 0 && s < a.pool_slots) ? int32_t(s) : -1;
    };
    auto ld_pos = [&](int j) -> int32_t {
        const int32_t p = __ldg(a.pos + start + j);
        return (p >= 0 && int64_t(p) < a.cs_rows) ? p : -1;
    };
    int32_t sl_cur = -1, sl_nxt = -1, p_cur = -1, p_nxt = -1;
    if (lane < cnt) {
        sl_cur = ld_slot(lane);
        if constexpr (kRope) p_cur = ld_pos(lane);
    }
    if (32 + lane < cnt) {
        sl_nxt = ld_slot(32 + lane);
        if constexpr (kRope) p_nxt = ld_pos(32 + lane);
    }
    int cur_b = 0;

    auto issue_cs = [&](int p) {
        if constexpr (kRope) {
            const int t = 2 * p + h;
            const int32_t pt = __shfl_sync(0xffffffffu, (t >> 5) == cur_b ? p_cur : p_nxt, t & 31);
            if (t < cnt && pt >= 0)
                cp_async16(wsm + (p & (NS - 1)) * SM::SLOT + 2 * SM::XB + h * SM::CSB + bi * 16,
                           a.cs + int64_t(pt) * kRopeD + bi * 4);
            cp_async_commit();
        }
    };
    auto issue = [&](int p) {
        issue_rows(p);
        issue_cs(p);
    };
    if constexpr (kRope) {
        issue_cs(0);
    } else {
        issue_rows(0);
    }
    if (npairs > 1) {
        // The first pair lands before the next ones are requested: every warp
        // starts at once, and the first pair is what holds it up.
        pdl_trigger();
        cp_async_wait<kG - 1>();
#pragma unroll
        for (int p = 1; p < D; ++p) issue(p);
    } else {
#pragma unroll
        for (int p = 1; p < D; ++p) issue(p);
        pdl_trigger();
    }

    int ring_out = 0;
    for (int k = 0; k < npairs; ++k) {
        if ((k & 15) == 0 && k > 0) {  // next batch of slots / positions
            sl_cur = sl_nxt;
            p_cur = p_nxt;
            cur_b = k >> 4;
            if (2 * k + 32 + lane < cnt) {
                sl_nxt = ld_slot(2 * k + 32 + lane);
                if constexpr (kRope) p_nxt = ld_pos(2 * k + 32 + lane);
            }
        }
        cp_async_wait<kG * D - 1>();  // this lane's row copies of pair k have landed ...
        __syncwarp();                 // ... and so have the other lanes'
        const uint32_t slot_sm = wsm + ring_out * SM::SLOT;
        ring_out = (ring_out + 1) & (NS - 1);
        const uint32_t row = slot_sm + h * SM::XB;

        // this lane's block (lanes 14 and 15 read the rotated blocks, unused with RoPE)
        float v[kBlock];
#pragma unroll
        for (int j = 0; j < SUBS; ++j) unpack_chunk<kBf16>(lds_u4(row + swz<SUBS>(bi, j) * 16), v + j * E);
        // with RoPE: this lane's quad of rotated dims
        float qv[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kRope) {
            const int blk = kRopeBlk0 + (bi >> 3);
            const int off = (4 * bi) & (kBlock - 1);  // first value of the quad inside its block
            const uint32_t qp = row + swz<SUBS>(blk, off / E) * 16 + (off % E) * (kBf16 ? 2 : 4);
            if constexpr (kBf16) {
                const uint2 r = lds_u2(qp);
                qv[0] = bf16_lo(r.x), qv[1] = bf16_hi(r.x), qv[2] = bf16_lo(r.y), qv[3] = bf16_hi(r.y);
            } else {
                const uint4 r = lds_u4(qp);
                qv[0] = __uint_as_float(r.x), qv[1] = __uint_as_float(r.y);
                qv[2] = __uint_as_float(r.z), qv[3] = __uint_as_float(r.w);
            }
        }
        const int t = 2 * k + h;
        const bool active = t < cnt;
        const int32_t slot = __shfl_sync(0xffffffffu, sl_cur, t & 31);
        int32_t pt = 0;
        if constexpr (kRope) pt = __shfl_sync(0xffffffffu, p_cur, t & 31);
        issue(k + D);  // refill the ring (the slot of pair k-1) while this pair is computed

        if constexpr (kNorm) {
            float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < kBlock; e += 4) {
                sa = ffma2(make_float2(v[e], v[e + 1]), make_float2(v[e], v[e + 1]), sa);
                sb = ffma2(make_float2(v[e + 2], v[e + 3]), make_float2(v[e + 2], v[e + 3]), sb);
            }
            float ss = bi < kOwn ? (sa.x + sa.y) + (sb.x + sb.y) : 0.f;
            if constexpr (kRope) {
                const float2 qa = fmul2(make_float2(qv[0], qv[1]), make_float2(qv[0], qv[1]));
                const float2 qb = ffma2(make_float2(qv[2], qv[3]), make_float2(qv[2], qv[3]), qa);
                ss += qb.x + qb.y;
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrt_approx(__fadd_rn(ss * (1.0f / kD), a.eps));
            const float2 inv2 = make_float2(inv, inv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 wv = *reinterpret_cast<const float4 *>(s_w + 4 * swz<8>(bi, j));
                const float2 a0 = fmul2(fmul2(make_float2(v[4 * j], v[4 * j + 1]), inv2), make_float2(wv.x, wv.y));
                const float2 a1 = fmul2(fmul2(make_float2(v[4 * j + 2], v[4 * j + 3]), inv2), make_float2(wv.z, wv.w));
                v[4 * j] = a0.x, v[4 * j + 1] = a0.y, v[4 * j + 2] = a1.x, v[4 * j + 3] = a1.y;
            }
            if constexpr (kRope) {
                const float4 wq = *reinterpret_cast<const float4 *>(s_w + 4 * swz<8>(kRopeBlk0 + (bi >> 3), bi & 7));
                const float2 a0 = fmul2(fmul2(make_float2(qv[0], qv[1]), inv2), make_float2(wq.x, wq.y));
                const float2 a1 = fmul2(fmul2(make_float2(qv[2], qv[3]), inv2), make_float2(wq.z, wq.w));
                qv[0] = a0.x, qv[1] = a0.y, qv[2] = a1.x, qv[3] = a1.y;
            }
        }

        // the blocks this lane owns: round, absmax, quantise, store
        if constexpr (kRoundBlk) round_bf16_n<kBlock>(v);
        const float am = amax32(v);
        const bool bad_pos = kRope && pt < 0;
        const bool ok = active && !bad_pos && slot >= 0;
        if (active && !ok && bi == 0) raise_err(a.err, bad_pos ? KVQ_DEVERR_POS : KVQ_DEVERR_SLOT);
        uint8_t *crow = nullptr, *srow = nullptr;
        if (ok) {
            const int64_t page = int64_t(slot >> PageBits) * PK::kPageBytes;
            const int row_i = slot & int(PK::kPage - 1);
            crow = a.pool + page + row_i * T::kCodeBytes;
            srow = a.pool + page + PK::kPage * T::kCodeBytes + row_i * T::kScaleBytes;
            if constexpr (L == Layout::V41) {
                const uint32_t sbyte = v41_scale_byte(__float_as_uint(am));
                const float mult = v41_multiplier(sbyte);
                if (bi < kOwn) {
                    uint32_t wd[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) wd[q] = v41_word(v + 4 * q, mult);
                    if (pool32) {
                        st_v8(crow + bi * 32, wd);
                    } else {
                        st_u4(crow + bi * 32, make_uint4(wd[0], wd[1], wd[2], wd[3]));
                        st_u4(crow + bi * 32 + 16, make_uint4(wd[4], wd[5], wd[6], wd[7]));
                    }
                    srow[bi] = uint8_t(sbyte);
                }
            } else {
                const uint32_t sbyte = fp4_scale_byte_fast(am);
                if (bi < kOwn) {
                    const float inv = s_rcp[sbyte];
                    uint32_t wd[4] = {0u, 0u, 0u, 0u};
                    if (sbyte != 0u) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) wd[q] = fp4_word(v + 8 * q, inv);
                    }
                    st_u4(crow + bi * 16, make_uint4(wd[0], wd[1], wd[2], wd[3]));
                    srow[bi] = uint8_t(sbyte);
                }
                if (bi == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
            }
        }

        // the rotated quads, once this pair's cos/sin rows have landed
        if constexpr (kRope) {
            cp_async_wait<2 * D>();  // (a refill of two groups was committed since)
            __syncwarp();
            const uint32_t cs = slot_sm + 2 * SM::XB + h * SM::CSB;
            const uint2 cc = lds_u2(cs + 8 * bi), ss = lds_u2(cs + kRopeD * 2 + 8 * bi);
            const float cq[2] = {__uint_as_float(cc.x), __uint_as_float(cc.y)};
            const float sq[2] = {__uint_as_float(ss.x), __uint_as_float(ss.y)};
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // pairs 2i and 2i+1 of the rotation
                const float2 xv = make_float2(qv[2 * q], qv[2 * q + 1]);
                const float2 p = fmul2(xv, make_float2(cq[q], sq[q]));  // (a*c, b*s)
                const float2 r = fmul2(xv, make_float2(sq[q], cq[q]));  // (a*s, b*c)
                qv[2 * q] = __fsub_rn(p.x, p.y);
                qv[2 * q + 1] = __fadd_rn(r.x, r.y);
            }
            if constexpr (kRoundQuad) round_bf16_n<4>(qv);
            float amq = fmaxf(fmax3(fabsf(qv[0]), fabsf(qv[1]), fabsf(qv[2])), fabsf(qv[3]));
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) amq = fmaxf(amq, __shfl_xor_sync(0xffffffffu, amq, off));
            if (ok) {
                if constexpr (L == Layout::V41) {
                    const uint32_t sbq = v41_scale_byte(__float_as_uint(amq));
                    *reinterpret_cast<uint32_t *>(crow + kRopeStart + 4 * bi) = v41_word(qv, v41_multiplier(sbq));
                    if ((bi & 7) == 0) srow[kRopeBlk0 + (bi >> 3)] = uint8_t(sbq);
                } else {
                    const uint32_t sbq = fp4_scale_byte_fast(amq);
                    const float inv = s_rcp[sbq];
                    uint32_t w2 = 0;
                    if (sbq != 0u) {
                        const float2 y0 = fmul2(make_float2(qv[0], qv[1]), make_float2(inv, inv));
                        const float2 y1 = fmul2(make_float2(qv[2], qv[3]), make_float2(inv, inv));
                        w2 = cvt_e2m1x2(y0.x, y0.y) | (cvt_e2m1x2(y1.x, y1.y) << 8);
                    }
                    *reinterpret_cast<uint16_t *>(crow + kRopeStart / 2 + 2 * bi) = uint16_t(w2);
                    if ((bi & 7) == 0) srow[kRopeBlk0 + (bi >> 3)] = uint8_t(sbq);
                }
            }
        }
    }
    cp_async_wait<0>();
}

// Contiguous token ranges for `warps` warps, computed on the host so that no
// warp divides.  The first warps take the remainder: when a launch follows
// another under PDL, the lowest CTAs become resident (and prefetch) first,
// so front-loading them evens out the finish times.  `skew` moves one more
// token from each of the last `skew` warps to the first ones (only when
// every warp holds four tokens or more).
inline StoreArgs partition(const StoreArgs &a, int64_t warps, int64_t skew) {
    StoreArgs b = a;
    b.warps = warps;
    b.per_warp = a.n / warps;
    b.extra = a.n % warps;
    if (b.per_warp < 4) skew = 0;  // small batches: one pair per warp is the latency
    if (b.extra + 2 * skew > warps) skew = (warps - b.extra) / 2;
    b.skew = skew;
    return b;
}

template <auto Kernel, int Warps, size_t Smem>
kvq_status launch_persistent(const StoreArgs &a, int64_t tokens_per_warp, int skew_div, cudaStream_t stream) {
    int64_t cap = 0;
    kvq_status st = resident_grid<Kernel, 32 * Warps>(Smem, &cap);
    if (st != KVQ_OK) return st;
    const int64_t want = (a.n + tokens_per_warp * Warps - 1) / (tokens_per_warp * Warps);
    const int64_t grid = want < cap ? want : cap;
    const int64_t warps = grid * Warps;
    return launch_pdl_smem(Kernel, dim3(unsigned(grid)), dim3(32 * Warps), Smem, stream,
                           partition(a, warps, skew_div > 0 ? warps / skew_div : 0));
}

// Which kernel serves which instance (past the one-CTA-per-token batches):
//  * Large V41 batches, from kPlainHalfMin tokens without the norm and from
//    kNormHalfMin with it: the half-warp kernel in four-warp CTAs (plain:
//    equal at 16384 tokens, 8-11% faster at 20480-32768; norm + RoPE: 3%
//    slower at 32768, 1-3% faster at 65536-262144).
//  * Below, V41 without RoPE, and the fused norm + RoPE: one warp per token.  The
//    norm + RoPE instance launches one-warp CTAs from two and a half tokens
//    per resident warp up, so that a finished warp frees its slot at once
//    and the next launch's warps become resident (and prefetch) sooner
//    (12288 tokens: 5.55 against 5.92 us); with fewer tokens per warp the
//    four times larger CTA count costs more in dispatch than it saves (8192
//    tokens: 6.34 against 4.52 us).
//  * V41 with RoPE only: from kRopeHalfMin tokens the half-warp kernel (the
//    rotation spread over all 16 lanes), one-warp CTAs, half the warps'
//    remainder front-loaded; below, one warp per token in four-warp CTAs
//    (4096 tokens: 2.65 against 3.46 us, 8192: 4.00 against 4.60 us; equal
//    at 12288, and 15% slower at 16384).
//  * V41_FP4: the half-warp kernel (each block's e4m3 scale, division and
//    reciprocal computed once), four-warp CTAs.
constexpr int64_t kRopeHalfMin = 12288;   // V41 store + RoPE
constexpr int64_t kPlainHalfMin = 16384;  // V41 store
constexpr int64_t kNormHalfMin = 65536;   // V41 store with the norm

template <Layout L, int PB, bool B16, bool L64, bool N, bool R>
kvq_status launch_store(const StoreArgs &a, cudaStream_t stream) {
    if constexpr (L == Layout::V41 && !(R && !N)) {
        if (a.n >= (N ? kNormHalfMin : kPlainHalfMin)) {
            using SMh = StoreSmem<L, B16, R, N>;
            return launch_persistent<store_half_kernel<L, PB, B16, L64, N, R, 4>, 4, SMh::bytes(4)>(a, 2, 0, stream);
        }
        constexpr size_t wsm = WarpStoreSmem<B16, R>::kWarpBytes;
        constexpr auto kern4 = store_warp_kernel<L, PB, B16, L64, N, R, 4>;
        if constexpr (N && R) {
            constexpr auto kern1 = store_warp_kernel<L, PB, B16, L64, N, R, 1>;
            constexpr auto kern1d2 = store_warp_kernel<L, PB, B16, L64, N, R, 1, 2>;
            int64_t cap1 = 0, cap4 = 0;
            kvq_status st = resident_grid<kern1, 32>(wsm, &cap1);
            if (st == KVQ_OK) st = resident_grid<kern4, 128>(4 * wsm, &cap4);
            if (st != KVQ_OK) return st;
            if (cap1 >= 4 * cap4 && 2 * a.n >= 5 * cap1) {
                // Up to four tokens per warp, two in flight instead of three
                // (a smaller first burst: 16384 tokens 6.61 -> 6.46 us; at 32768
                // tokens three are faster, 10.96 against 11.96 us).
                if (a.n <= 4 * cap1) {
                    int64_t cap1d2 = 0;
                    st = resident_grid<kern1d2, 32>(wsm, &cap1d2);
                    if (st != KVQ_OK) return st;
                    if (cap1d2 == cap1) return launch_persistent<kern1d2, 1, wsm>(a, 1, 0, stream);
                }
                return launch_persistent<kern1, 1, wsm>(a, 1, 0, stream);
            }
        }
        return launch_persistent<kern4, 4, 4 * wsm>(a, 1, 0, stream);
    } else if constexpr (L == Layout::V41) {
        if (a.n < kRopeHalfMin) {
            constexpr size_t wsm = WarpStoreSmem<B16, R>::kWarpBytes;
            return launch_persistent<store_warp_kernel<L, PB, B16, L64, N, R, 4>, 4, 4 * wsm>(a, 1, 0, stream);
        }
        using SM = StoreSmem<L, B16, R, N>;
        return launch_persistent<store_half_kernel<L, PB, B16, L64, N, R, 1>, 1, SM::bytes(1)>(a, 2, 2, stream);
    } else {
        using SM = StoreSmem<L, B16, R, N>;
        return launch_persistent<store_half_kernel<L, PB, B16, L64, N, R, 4>, 4, SM::bytes(4)>(a, 2, 0, stream);
    }
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
    if (pool_slots > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;  // slots are held as int32
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
    if (const int tpc = store_small_tokens_per_cta(layout, norm, rope, n))
        return launch_store_small(layout, page_bits, x_dtype == KVQ_BF16, loc_dtype == KVQ_I64, norm, rope, tpc, a, s);
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
