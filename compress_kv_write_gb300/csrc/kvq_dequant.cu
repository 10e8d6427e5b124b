// kvq_dequant.cu -- paged dequant of V41 / V41_FP4 pages into a contiguous
// bf16 workspace, the job of dequant_k_cache.py in "[sglang] DeepSeek V4.1
// Paged KV Cache: V41 and FP4 formats" (section 4).
//
// Mapping: one CTA per logical page.  The page's code area is cut into
// pieces of 8 values (8 bytes of e4m3 or 4 bytes of e2m1); thread i takes
// pieces i, i+256, ...  Each piece becomes 16 bytes of bf16, so the 32 lanes
// of a warp write 512 contiguous bytes per store instruction.  Every code
// load of the CTA is issued first; the page's scale rows are staged in
// shared memory meanwhile.  Every product code * scale has at most 6
// significant bits, so the bf16 result is exact.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kDqThreads = 256;

struct DequantArgs {
    const uint8_t *pool;
    int64_t pool_pages;
    const int32_t *page_table;
    uint8_t *out;
    int64_t out_stride_bytes;
    int32_t *err;
};

template <Layout L, int PageBits>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const DequantArgs a) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int64_t P = PK::kPage;
    constexpr int kPieceBytes = L == Layout::V41 ? 8 : 4;        // 8 values
    constexpr int kPiecesPerRow = T::kCodeBytes / kPieceBytes;     // 64
    constexpr int64_t kPieces = P * kPiecesPerRow;
    constexpr int ITER = int((kPieces + kDqThreads - 1) / kDqThreads);
    constexpr int kScaleArea = int(P * T::kScaleBytes);           // bytes
    static_assert(kPiecesPerRow == 64, "a row is 64 pieces of 8 values");
    static_assert(kScaleArea % 16 == 0, "scale area is whole 16-byte chunks");

    __shared__ __align__(16) uint8_t s_scale[kScaleArea];

    const int64_t lp = blockIdx.x;
    pdl_wait();
    const int64_t phys = __ldg(a.page_table + lp);
    if (phys < 0 || phys >= a.pool_pages) {
        if (threadIdx.x == 0) raise_err(a.err, KVQ_DEVERR_PAGE);
        return;
    }
    const uint8_t *codes = a.pool + phys * PK::kPageBytes;
    const uint8_t *scales = codes + P * T::kCodeBytes;

    uint2 raw[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
        const int64_t q = int64_t(it) * kDqThreads + threadIdx.x;
        if (q < kPieces) {
            if constexpr (kPieceBytes == 8) {
                raw[it] = __ldg(reinterpret_cast<const uint2 *>(codes) + q);
            } else {
                raw[it].x = __ldg(reinterpret_cast<const uint32_t *>(codes) + q);
                raw[it].y = 0;
            }
        }
    }
    for (int c = threadIdx.x; c < kScaleArea / 16; c += kDqThreads)
        *reinterpret_cast<uint4 *>(s_scale + c * 16) = __ldg(reinterpret_cast<const uint4 *>(scales) + c);
    __syncthreads();
    pdl_trigger();

#pragma unroll
    for (int it = 0; it < ITER; ++it) {
        const int64_t q = int64_t(it) * kDqThreads + threadIdx.x;
        if (q >= kPieces) break;
        const int64_t row = q / kPiecesPerRow;
        const int j = int(q % kPiecesPerRow);                 // values 8j .. 8j+7
        const uint32_t sb = s_scale[row * T::kScaleBytes + j / 4];
        uint32_t o[4];
        if constexpr (L == Layout::V41) {
            const float sc = ue8m0_to_f32(sb);
            const uint32_t w[2] = {raw[it].x, raw[it].y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float2 f0 = e4m3x2_to_f32x2(w[h] & 0xFFFFu);
                const float2 f1 = e4m3x2_to_f32x2(w[h] >> 16);
                const float2 g0 = fmul2(f0, make_float2(sc, sc));
                const float2 g1 = fmul2(f1, make_float2(sc, sc));
                o[2 * h] = pack_bf16x2(g0.x, g0.y);
                o[2 * h + 1] = pack_bf16x2(g1.x, g1.y);
            }
        } else {
            const float S = e4m3x2_to_f32x2(sb).x;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float2 f = e2m1x2_to_f32x2((raw[it].x >> (8 * b)) & 0xFFu);
                const float2 g = fmul2(f, make_float2(S, S));
                o[b] = pack_bf16x2(g.x, g.y);
            }
        }
        st_u4(a.out + (lp * P + row) * a.out_stride_bytes + j * 16, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

template <Layout L, int PB>
kvq_status launch_dequant(const DequantArgs &a, int64_t n_pages, cudaStream_t stream) {
    if (n_pages > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    return launch_pdl(dequant_kernel<L, PB>, dim3(unsigned(n_pages)), dim3(kDqThreads), stream, a);
}

// ---------------------------------------------------------------------------
// Selected-token dequant: the rows a sparse attention picks, gathered by slot.
// One warp per token, TPW tokens per warp with every load issued first.  A
// row is 64 pieces of 8 values; lane l decodes pieces l and l+32, so each
// warp store instruction writes 512 contiguous bytes of the output row.

constexpr int kDsThreads = 256;
constexpr int kDsTPW = 4;

struct DequantSlotsArgs {
    const uint8_t *pool;
    int64_t pool_slots;
    const void *slots;
    int64_t n;
    uint8_t *out;
    int64_t out_stride_bytes;
    int32_t *err;
};

template <Layout L, int PageBits, bool kIdx64>
__global__ void __launch_bounds__(kDsThreads) dequant_slots_kernel(const DequantSlotsArgs a) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int kPieceBytes = L == Layout::V41 ? 8 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t(blockIdx.x) * (kDsThreads / 32) + (threadIdx.x >> 5)) * kDsTPW;

    pdl_wait();
    int64_t slot[kDsTPW];
    uint2 raw[kDsTPW][2];
    uint4 sc[kDsTPW];
#pragma unroll
    for (int j = 0; j < kDsTPW; ++j) {
        slot[j] = -2;
        if (t0 + j < a.n)
            slot[j] = kIdx64 ? __ldg(static_cast<const int64_t *>(a.slots) + t0 + j)
                             : int64_t(__ldg(static_cast<const int32_t *>(a.slots) + t0 + j));
    }
#pragma unroll
    for (int j = 0; j < kDsTPW; ++j) {
        if (slot[j] >= 0 && slot[j] < a.pool_slots) {
            const uint8_t *crow = PK::code_row(const_cast<uint8_t *>(a.pool), slot[j]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int p = lane + 32 * h;
                if constexpr (kPieceBytes == 8) {
                    raw[j][h] = __ldg(reinterpret_cast<const uint2 *>(crow) + p);
                } else {
                    raw[j][h] = make_uint2(__ldg(reinterpret_cast<const uint32_t *>(crow) + p), 0u);
                }
            }
            sc[j] = __ldg(reinterpret_cast<const uint4 *>(PK::scale_row(const_cast<uint8_t *>(a.pool), slot[j])));
        }
    }
    pdl_trigger();

#pragma unroll
    for (int j = 0; j < kDsTPW; ++j) {
        const int64_t t = t0 + j;
        if (t >= a.n) break;
        uint8_t *orow = a.out + t * a.out_stride_bytes;
        if (slot[j] == -1) {  // padding: a zero row
            st_u4(orow + lane * 16, make_uint4(0u, 0u, 0u, 0u));
            st_u4(orow + 512 + lane * 16, make_uint4(0u, 0u, 0u, 0u));
            continue;
        }
        if (slot[j] < 0 || slot[j] >= a.pool_slots) {
            if (lane == 0) raise_err(a.err, KVQ_DEVERR_SLOT);
            continue;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // piece p = lane + 32h covers values 8p .. 8p+7, quant block p / 4
            const uint32_t word = h == 0 ? (lane < 16 ? sc[j].x : sc[j].y) : (lane < 16 ? sc[j].z : sc[j].w);
            const uint32_t sb = (word >> (8 * ((lane >> 2) & 3))) & 0xFFu;
            uint32_t o[4];
            if constexpr (L == Layout::V41) {
                const float s = ue8m0_to_f32(sb);
                const uint32_t w[2] = {raw[j][h].x, raw[j][h].y};
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 g0 = fmul2(e4m3x2_to_f32x2(w[q] & 0xFFFFu), make_float2(s, s));
                    const float2 g1 = fmul2(e4m3x2_to_f32x2(w[q] >> 16), make_float2(s, s));
                    o[2 * q] = pack_bf16x2(g0.x, g0.y);
                    o[2 * q + 1] = pack_bf16x2(g1.x, g1.y);
                }
            } else {
                const float S = e4m3x2_to_f32x2(sb).x;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float2 g = fmul2(e2m1x2_to_f32x2((raw[j][h].x >> (8 * b)) & 0xFFu), make_float2(S, S));
                    o[b] = pack_bf16x2(g.x, g.y);
                }
            }
            st_u4(orow + (lane + 32 * h) * 16, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

template <Layout L, int PB, bool I64>
kvq_status launch_dequant_slots(const DequantSlotsArgs &a, cudaStream_t stream) {
    const int64_t warps = (a.n + kDsTPW - 1) / kDsTPW;
    const int64_t blocks = (warps + kDsThreads / 32 - 1) / (kDsThreads / 32);
    if (blocks > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    return launch_pdl(dequant_slots_kernel<L, PB, I64>, dim3(unsigned(blocks)), dim3(kDsThreads), stream, a);
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_dequant(kvq_layout layout, int page_bits, const uint8_t *pool,
                                  int64_t pool_pages, const int32_t *page_table, int64_t n_tokens,
                                  void *out_bf16, int64_t out_row_stride, int32_t *err,
                                  struct CUstream_st *stream) {
    if (layout != KVQ_LAYOUT_V41 && layout != KVQ_LAYOUT_V41_FP4) return KVQ_ERR_INVALID_ARG;
    if (page_bits < 1 || page_bits > 16) return KVQ_ERR_INVALID_ARG;
    if (!page_bits_supported(page_bits)) return KVQ_ERR_UNSUPPORTED;
    if (!pool || !aligned(pool, 16) || pool_pages <= 0) return KVQ_ERR_INVALID_ARG;
    if (n_tokens < 0 || (n_tokens & ((int64_t(1) << page_bits) - 1)) != 0) return KVQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return KVQ_OK;  // nothing to enqueue; the table / output may be empty
    if (!page_table || !aligned(page_table, 4)) return KVQ_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned(out_bf16, 16) || out_row_stride < kD || (out_row_stride * 2) % 16 != 0)
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;

    DequantArgs a;
    a.pool = pool;
    a.pool_pages = pool_pages;
    a.page_table = page_table;
    a.out = static_cast<uint8_t *>(out_bf16);
    a.out_stride_bytes = out_row_stride * 2;
    a.err = err;
    const int64_t n_pages = n_tokens >> page_bits;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return launch_dequant<decltype(Lc)::value, decltype(PBc)::value>(a, n_pages, s);
        });
    });
}

extern "C" kvq_status kvq_dequant_slots(kvq_layout layout, int page_bits, const uint8_t *pool,
                                        int64_t pool_slots, const void *slots, kvq_index_dtype slot_dtype,
                                        int64_t n, void *out_bf16, int64_t out_row_stride, int32_t *err,
                                        struct CUstream_st *stream) {
    kvq_status st = check_pool(layout, page_bits, pool, pool_slots);
    if (st != KVQ_OK) return st;
    if (slot_dtype != KVQ_I32 && slot_dtype != KVQ_I64) return KVQ_ERR_INVALID_ARG;
    if (n < 0) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;  // nothing to enqueue; slots / output may be empty
    if (!slots || !aligned(slots, slot_dtype == KVQ_I64 ? 8 : 4)) return KVQ_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned(out_bf16, 16) || out_row_stride < kD || (out_row_stride * 2) % 16 != 0)
        return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;

    DequantSlotsArgs a;
    a.pool = pool;
    a.pool_slots = pool_slots;
    a.slots = slots;
    a.n = n;
    a.out = static_cast<uint8_t *>(out_bf16);
    a.out_stride_bytes = out_row_stride * 2;
    a.err = err;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return with_layout(layout, [&](auto Lc) {
        return with_page_bits(page_bits, [&](auto PBc) {
            return with_bool(slot_dtype == KVQ_I64, [&](auto I64) {
                return launch_dequant_slots<decltype(Lc)::value, decltype(PBc)::value, decltype(I64)::value>(a, s);
            });
        });
    });
}
