// kvq_store.cu -- fused (K RMSNorm) + (RoPE) + block quantisation + paged
// scatter of new K rows: the store / store + RoPE / fused K norm + RoPE
// kernels of "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats"
// (section 1 store_row, and the store-latency table).
//
// Both kernels are persistent (as many CTAs of four warps as are resident at
// once; the fused norm + RoPE V41 instance switches to one-warp CTAs from
// three tokens per resident warp up); warp w of W owns the contiguous token
// range [n*w/W, n*(w+1)/W) and
// keeps its next rows in flight in a per-warp shared-memory ring filled with
// cp.async (one commit group per ring slot; the V41 kernel with RoPE commits
// a token's cos/sin values as a second group, so that everything but the
// rotated chunk is finished while they land).  Before the PDL wait each warp
// prefetches its first rows into L2.  Slot indices and positions of
// 32 tokens sit one per lane, validated once, and are fetched with a
// shuffle.  Math is fp32; the products of the RMSNorm and of the rotation are
// rounded one by one, as in the definition.
//
//  * store_warp_kernel (V41): one warp per token.  Lane l owns the 16-byte
//    chunks l, l+32, ... of the row, so every warp load / store instruction
//    covers one contiguous span; a 32-value quant block is 32/(values per
//    chunk) adjacent lanes, reduced with xor shuffles.  Each lane copies and
//    reads back only its own chunks: no cross-lane waits.
//  * store_pair_kernel (V41_FP4): two tokens per warp; half-warp h holds
//    token 2k+h and lane i of the half owns quant block i.  The block
//    absmax needs no shuffle and each block's e4m3 scale and reciprocal are
//    computed once.  Rows land block-swizzled in shared memory so the
//    block-per-lane reads are bank-conflict-free.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kStoreWarps = 4;
constexpr int kStoreThreads = kStoreWarps * 32;

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

template <bool kBf16, bool kRope>
struct WarpStoreSmem {
    static constexpr int XB = kD * (kBf16 ? 2 : 4);    // input row bytes
    static constexpr int CSB = kRope ? kRopeD * 4 : 0;  // this token's cos/sin values
    static constexpr int D = 3;                         // tokens in flight per warp
    static constexpr int NS = D + 1;                    // ring slots per warp (a power of two)
    static_assert((NS & (NS - 1)) == 0, "ring index by mask");
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
        float m[E / 2];
#pragma unroll
        for (int e = 0; e < E / 2; ++e) m[e] = fmaxf(fabsf(v[k][2 * e]), fabsf(v[k][2 * e + 1]));
#pragma unroll
        for (int w = E / 4; w >= 1; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e) m[e] = fmaxf(m[e], m[e + w]);
        float mm = m[0];
#pragma unroll
        for (int off = 1; off < LPB; off <<= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
        am[k] = mm;
    }
}

// Quantise chunks K0 .. K1-1 with their block absmax into the token's code
// row and scale row.  The lane that leads a quant block writes its scale byte.
template <Layout L, int E, int K, int K0, int K1>
__device__ __forceinline__ void quant_store(float (&v)[K][E], const float (&am)[K], uint8_t *crow, uint8_t *srow,
                                            int lane) {
    constexpr int LPB = kBlock / E;
#pragma unroll
    for (int k = K0; k < K1; ++k) {
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
        if (lane % LPB == 0) srow[c / LPB] = uint8_t(sbyte);
    }
    if constexpr (LayoutTraits<L>::kScaleBytes == 32 && K1 == K) {
        if (lane == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
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

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope, int kWarps>
__global__ void __launch_bounds__(32 * kWarps, 8 * (kStoreWarps / kWarps)) store_warp_kernel(const StoreArgs a) {
    using SM = WarpStoreSmem<kBf16, kRope>;
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
    uint8_t *wsm = smem + warp * SM::kWarpBytes;
    const int64_t W = int64_t(gridDim.x) * kWarps;
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    const int64_t start = a.n * gw / W;
    const int cnt = int(a.n * (gw + 1) / W - start);

    // While the upstream grid drains: pull this warp's first NS rows and its
    // slot / position lines into L2 (hints only; the loads come after the wait).
    if (lane < cnt && lane < NS) prefetch_l2_bulk(a.x + (start + lane) * a.row_stride_bytes, SM::XB);
    if (lane == 0 && cnt > 0) {
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + start)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + start));
        if constexpr (kRope) prefetch_l2(a.pos + start);
    }
    pdl_wait();

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
    const uint8_t *src_next = a.x + start * a.row_stride_bytes + lane * 16;
    int ring_in = 0;
    auto issue = [&](int j) {
        if (j < cnt) {
            uint8_t *slot = wsm + ring_in * SM::SLOT + lane * 16;
#pragma unroll
            for (int k = 0; k < K; ++k) cp_async16(slot + k * 512, src_next + k * 512);
            if constexpr (kRope) {
                cp_async_commit();
                const int32_t pj = __shfl_sync(0xffffffffu, (j >> 5) == cur_b ? p_cur : p_nxt, j & 31);
                if (lane >= kRopeLane0 && pj >= 0) {
                    const int i0 = ((K - 1) * 32 + lane) * E / 2 - kRopeStart / 2;
                    const float *cs = a.cs + int64_t(pj) * kRopeD;
                    uint8_t *dst = wsm + ring_in * SM::SLOT + SM::XB + (lane - kRopeLane0) * E * 4;
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
        // row is what holds the warp up (store + RoPE at 16384 tokens:
        // 6.44 -> 6.26 us).  Warps with a single token, and the plain store,
        // are faster without the wait.
        issue(0);
        pdl_trigger();
        cp_async_wait<kGroups - 1>();
#pragma unroll
        for (int j = 1; j < D; ++j) issue(j);
    } else {
#pragma unroll
        for (int j = 0; j < D; ++j) issue(j);
        pdl_trigger();
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
        const uint8_t *slot_sm = wsm + ring_out * SM::SLOT;
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
            float ss = ((ss2[0].x + ss2[0].y) + (ss2[1].x + ss2[1].y)) + ((ss2[2].x + ss2[2].y) + (ss2[3].x + ss2[3].y));
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
                const uint8_t *cs = slot_sm + SM::XB + (lane - kRopeLane0) * E * 4;
                if constexpr (E == 8) {
                    const uint4 c4 = lds_u4(cs), s4 = lds_u4(cs + 16);
                    cosv[0] = __uint_as_float(c4.x), cosv[1] = __uint_as_float(c4.y);
                    cosv[2] = __uint_as_float(c4.z), cosv[3] = __uint_as_float(c4.w);
                    sinv[0] = __uint_as_float(s4.x), sinv[1] = __uint_as_float(s4.y);
                    sinv[2] = __uint_as_float(s4.z), sinv[3] = __uint_as_float(s4.w);
                } else {
                    const float2 c2 = *reinterpret_cast<const float2 *>(cs);
                    const float2 s2 = *reinterpret_cast<const float2 *>(cs + 8);
                    cosv[0] = c2.x, cosv[1] = c2.y, sinv[0] = s2.x, sinv[1] = s2.y;
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

template <bool kBf16, bool kRope, bool kNorm>
struct PairStoreSmem {
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
    static constexpr int kW = kStoreWarps * kWarpBytes;  // norm weights, swizzled
    static constexpr int kBytes = kW + (kNorm ? kD * 4 : 0);
    static_assert(SLOT % 16 == 0, "16-byte aligned slots");
    static_assert((2 * CPR) % 32 == 0, "a pair is whole chunks per lane");
};

template <Layout L, int PageBits, bool kBf16, bool kLoc64, bool kNorm, bool kRope>
__global__ void __launch_bounds__(kStoreThreads, 4) store_pair_kernel(const StoreArgs a) {
    using SM = PairStoreSmem<kBf16, kRope, kNorm>;
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int D = SM::D, NS = SM::NS, E = SM::E, SUBS = SM::SUBS, CPR = SM::CPR;
    constexpr int NC = 2 * CPR / 32;          // chunks each lane copies per pair
    constexpr int kRopeBlk0 = kRopeStart / kBlock;  // first rotated block (14)
    static_assert(kRopeD == 2 * kBlock, "the rotated dims are the last two blocks");
    static_assert(D < 16, "a pair's slot index is in the current or the next batch of 32");

    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h = lane >> 4;   // token of the pair
    const int bi = lane & 15;  // quant block owned
    uint8_t *wsm = smem + warp * SM::kWarpBytes;
    const float *s_w = reinterpret_cast<const float *>(smem + SM::kW);
    const int64_t W = int64_t(gridDim.x) * kStoreWarps;
    const int64_t gw = int64_t(blockIdx.x) * kStoreWarps + warp;
    const int64_t start = a.n * gw / W;
    const int cnt = int(a.n * (gw + 1) / W - start);
    const int npairs = (cnt + 1) >> 1;

    // While the upstream grid drains: L2 hints for this warp's first NS pairs
    // and its slot / position lines (the loads come after the wait).
    if (lane < cnt && lane < 2 * NS) prefetch_l2_bulk(a.x + (start + lane) * a.row_stride_bytes, SM::XB);
    if (lane == 0 && cnt > 0) {
        prefetch_l2(kLoc64 ? static_cast<const void *>(static_cast<const int64_t *>(a.loc) + start)
                           : static_cast<const void *>(static_cast<const int32_t *>(a.loc) + start));
        if constexpr (kRope) prefetch_l2(a.pos + start);
    }
    pdl_wait();

    if constexpr (kNorm) {  // the weight row, block-swizzled like fp32 rows
        float *w = reinterpret_cast<float *>(smem + SM::kW);
        for (int c = threadIdx.x; c < kD / 4; c += kStoreThreads)
            *reinterpret_cast<float4 *>(w + 4 * swz<8>(c >> 3, c & 7)) =
                __ldg(reinterpret_cast<const float4 *>(a.w) + c);
        __syncthreads();
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

    // copies of token pair p (tokens 2p, 2p+1) into the next ring slot
    int ring_in = 0;
    auto issue = [&](int p) {
        if (p < npairs) {
            uint8_t *slot = wsm + ring_in * SM::SLOT;
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                const int c = lane + 32 * m;
                const int r = c / CPR, cc = c % CPR;
                if (2 * p + r < cnt)
                    cp_async16(slot + (r * CPR + swz<SUBS>(cc / SUBS, cc % SUBS)) * 16,
                               a.x + (start + 2 * p + r) * a.row_stride_bytes + cc * 16);
            }
            if constexpr (kRope) {
                const int t = 2 * p + h;
                const int32_t pt = __shfl_sync(0xffffffffu, (t >> 5) == cur_b ? p_cur : p_nxt, t & 31);
                if (t < cnt && pt >= 0)
                    cp_async16(slot + 2 * SM::XB + h * SM::CSB + bi * 16, a.cs + int64_t(pt) * kRopeD + bi * 4);
            }
            ring_in = (ring_in + 1) & (NS - 1);
        }
        cp_async_commit();
    };

    if (npairs > 1) {
        // The first pair lands before the next ones are requested: every warp
        // starts at once, and the first pair is what holds it up (FP4 store
        // at 16384 tokens: 5.07 -> 4.82 us).
        issue(0);
        pdl_trigger();
        cp_async_wait<0>();
#pragma unroll
        for (int p = 1; p < D; ++p) issue(p);
    } else {
#pragma unroll
        for (int p = 0; p < D; ++p) issue(p);
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
        cp_async_wait<D - 1>();  // this lane's copies of pair k have landed ...
        __syncwarp();            // ... and so have the other lanes'
        const uint8_t *slot_sm = wsm + ring_out * SM::SLOT;
        ring_out = (ring_out + 1) & (NS - 1);

        float v[kBlock];
        {
            const uint8_t *row = slot_sm + h * SM::XB;
#pragma unroll
            for (int j = 0; j < SUBS; ++j) unpack_chunk<kBf16>(lds_u4(row + swz<SUBS>(bi, j) * 16), v + j * E);
        }
        const int t = 2 * k + h;
        const bool active = t < cnt;
        const int32_t slot = __shfl_sync(0xffffffffu, sl_cur, t & 31);
        int32_t pt = 0;
        if constexpr (kRope) pt = __shfl_sync(0xffffffffu, p_cur, t & 31);

        if constexpr (kNorm) {
            float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < kBlock; e += 2) {
                const float2 t2 = make_float2(v[e], v[e + 1]);
                ss2 = ffma2(t2, t2, ss2);
            }
            float ss = ss2.x + ss2.y;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrt_approx(__fadd_rn(ss * (1.0f / kD), a.eps));
            const float2 inv2 = make_float2(inv, inv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 wv = *reinterpret_cast<const float4 *>(s_w + 4 * swz<8>(bi, j));
                const float2 a0 = fmul2(fmul2(make_float2(v[4 * j], v[4 * j + 1]), inv2), make_float2(wv.x, wv.y));
                const float2 a1 = fmul2(fmul2(make_float2(v[4 * j + 2], v[4 * j + 3]), inv2), make_float2(wv.z, wv.w));
                v[4 * j] = a0.x;
                v[4 * j + 1] = a0.y;
                v[4 * j + 2] = a1.x;
                v[4 * j + 3] = a1.y;
            }
        }
        if constexpr (kRope) {
            if (bi >= kRopeBlk0) {  // pairs (bi - 14) * 16 .. +15 of the rotation
                const float *cs = reinterpret_cast<const float *>(slot_sm + 2 * SM::XB + h * SM::CSB);
                const int q0 = (bi - kRopeBlk0) * (kBlock / 2);
#pragma unroll
                for (int g = 0; g < kBlock / 8; ++g) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(cs + q0 + 4 * g);
                    const float4 s4 = *reinterpret_cast<const float4 *>(cs + kRopeD / 2 + q0 + 4 * g);
                    const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xv = make_float2(v[8 * g + 2 * q], v[8 * g + 2 * q + 1]);
                        const float2 p = fmul2(xv, make_float2(cc[q], sn[q]));  // (a*c, b*s)
                        const float2 r = fmul2(xv, make_float2(sn[q], cc[q]));  // (a*s, b*c)
                        v[8 * g + 2 * q] = __fsub_rn(p.x, p.y);
                        v[8 * g + 2 * q + 1] = __fadd_rn(r.x, r.y);
                    }
                }
            }
        }
        issue(k + D);  // refill the ring while this pair is computed

        if constexpr (kNorm || kRope) {
#pragma unroll
            for (int e = 0; e < kBlock; e += 2) {
                const uint32_t b = pack_bf16x2(v[e], v[e + 1]);
                v[e] = bf16_lo(b);
                v[e + 1] = bf16_hi(b);
            }
        }
        // block absmax (this lane holds the whole block): four running maxima
        float m0 = fabsf(v[0]), m1 = fabsf(v[1]), m2 = fabsf(v[2]), m3 = fabsf(v[3]);
#pragma unroll
        for (int e = 4; e < kBlock; e += 4) {
            m0 = fmaxf(m0, fabsf(v[e]));
            m1 = fmaxf(m1, fabsf(v[e + 1]));
            m2 = fmaxf(m2, fabsf(v[e + 2]));
            m3 = fmaxf(m3, fabsf(v[e + 3]));
        }
        const uint32_t amax = __float_as_uint(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));

        const bool bad_pos = kRope && pt < 0;
        if (!active || bad_pos || slot < 0) {
            if (active && bi == 0) raise_err(a.err, bad_pos ? KVQ_DEVERR_POS : KVQ_DEVERR_SLOT);
            continue;
        }
        const int64_t page = int64_t(slot >> PageBits) * PK::kPageBytes;
        const int row = slot & int(PK::kPage - 1);
        uint8_t *crow = a.pool + page + row * T::kCodeBytes;
        uint8_t *srow = a.pool + page + PK::kPage * T::kCodeBytes + row * T::kScaleBytes;
        uint32_t sbyte;
        if constexpr (L == Layout::V41) {
            sbyte = v41_scale_byte(amax);
            const float mult = v41_multiplier(sbyte);
            const float2 mult2 = make_float2(mult, mult);
            uint32_t wd[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float2 lo = fmul2(make_float2(v[4 * q], v[4 * q + 1]), mult2);
                const float2 hi = fmul2(make_float2(v[4 * q + 2], v[4 * q + 3]), mult2);
                wd[q] = cvt_e4m3x2(lo.x, lo.y) | (cvt_e4m3x2(hi.x, hi.y) << 16);
            }
            st_u4(crow + bi * 32, make_uint4(wd[0], wd[1], wd[2], wd[3]));
            st_u4(crow + bi * 32 + 16, make_uint4(wd[4], wd[5], wd[6], wd[7]));
        } else {
            sbyte = fp4_scale_byte(amax);
            const float S = e4m3x2_to_f32x2(sbyte).x;
            const float inv = __frcp_rn(S);
            uint32_t wd[4] = {0u, 0u, 0u, 0u};
            if (S != 0.0f) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float2 y = fmul2(make_float2(v[2 * q], v[2 * q + 1]), make_float2(inv, inv));
                    wd[q >> 2] |= cvt_e2m1x2(y.x, y.y) << (8 * (q & 3));
                }
            }
            st_u4(crow + bi * 16, make_uint4(wd[0], wd[1], wd[2], wd[3]));
            if (bi == 0) st_u4(srow + 16, make_uint4(0u, 0u, 0u, 0u));
        }
        srow[bi] = uint8_t(sbyte);
    }
    cp_async_wait<0>();
}

// V41 rows use the warp-per-token kernel (fewer instructions for the
// norm / RoPE paths); V41_FP4 rows use the pair kernel, which computes each
// block's e4m3 scale and its reciprocal once per block instead of once per
// lane of the block.
template <Layout L, int PB, bool B16, bool L64, bool N, bool R>
kvq_status launch_store(const StoreArgs &a, cudaStream_t stream) {
    if constexpr (L == Layout::V41) {
        constexpr size_t wsm = WarpStoreSmem<B16, R>::kWarpBytes;
        constexpr auto kern4 = store_warp_kernel<L, PB, B16, L64, N, R, kStoreWarps>;
        int64_t cap4 = 0;
        kvq_status st = resident_grid<kern4, kStoreThreads>(kStoreWarps * wsm, &cap4);
        if (st != KVQ_OK) return st;
        if constexpr (N && R) {
            // The fused norm + RoPE instance also has a one-warp-CTA form.
            // With each warp holding at least three tokens, a finished warp
            // then frees its slot at once, so the next launch's warps become
            // resident, and start their L2 prefetch, sooner (norm + RoPE at
            // 16384 tokens: 7.45 -> 7.15 us).  With fewer tokens per warp the
            // four times larger CTA count costs more in dispatch than it
            // saves (2.97 -> 5.56 us at 4096 tokens).
            constexpr auto kern1 = store_warp_kernel<L, PB, B16, L64, N, R, 1>;
            int64_t cap1 = 0;
            st = resident_grid<kern1, 32>(wsm, &cap1);
            if (st != KVQ_OK) return st;
            if (cap1 >= kStoreWarps * cap4 && a.n >= 3 * cap1)
                return launch_pdl_smem(kern1, dim3(unsigned(cap1)), dim3(32), wsm, stream, a);
        }
        const int64_t want = (a.n + kStoreWarps - 1) / kStoreWarps;
        const int64_t grid = want < cap4 ? want : cap4;
        return launch_pdl_smem(kern4, dim3(unsigned(grid)), dim3(kStoreThreads), kStoreWarps * wsm, stream, a);
    } else {
        constexpr auto kern = store_pair_kernel<L, PB, B16, L64, N, R>;
        constexpr size_t smem = PairStoreSmem<B16, R, N>::kBytes;
        int64_t cap = 0;
        kvq_status st = resident_grid<kern, kStoreThreads>(smem, &cap);
        if (st != KVQ_OK) return st;
        const int64_t want = (a.n + 2 * kStoreWarps - 1) / (2 * kStoreWarps);
        const int64_t grid = want < cap ? want : cap;
        return launch_pdl_smem(kern, dim3(unsigned(grid)), dim3(kStoreThreads), smem, stream, a);
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
