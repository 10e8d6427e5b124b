// kvq_dequant.cu -- paged dequant of V41 / V41_FP4 pages into a contiguous
// bf16 workspace, the job of dequant_k_cache.py in "[sglang] DeepSeek V4.1
// Paged KV Cache: V41 and FP4 formats" (section 4).
//
// Mapping: one CTA per logical page.  The page's code area is contiguous, so
// the CTA sweeps it in 16-byte chunks (thread i takes chunks i, i+256, ...),
// all loads issued before any conversion; each chunk's scale byte comes from
// the page's scale area.  V41: a chunk is 16 codes of one row (half a quant
// block) -> 32 bytes of bf16.  V41_FP4: a chunk is one whole 32-value block
// -> 64 bytes of bf16.  Every product code * scale has at most 6 significant
// bits, so the bf16 result is exact.
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

__device__ __forceinline__ uint8_t ld_byte(const uint8_t *p) {
    uint16_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return uint8_t(r);
}

template <Layout L, int PageBits>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const DequantArgs a) {
    using PK = PagedKV<L, PageBits>;
    using T = LayoutTraits<L>;
    constexpr int64_t P = PK::kPage;
    constexpr int kChunksPerRow = T::kCodeBytes / 16;       // 32 (V41) or 16 (FP4)
    constexpr int64_t kChunks = P * kChunksPerRow;
    constexpr int ITER = int((kChunks + kDqThreads - 1) / kDqThreads);

    const int64_t lp = blockIdx.x;
    pdl_wait();
    const int64_t phys = __ldg(a.page_table + lp);
    if (phys < 0 || phys >= a.pool_pages) {
        if (threadIdx.x == 0) raise_err(a.err, KVQ_DEVERR_PAGE);
        return;
    }
    const uint8_t *codes = a.pool + phys * PK::kPageBytes;
    const uint8_t *scales = codes + P * T::kCodeBytes;

    uint4 raw[ITER];
    uint8_t sb[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
        const int64_t c = int64_t(it) * kDqThreads + threadIdx.x;
        if (c < kChunks) {
            raw[it] = ld_stream_u4(codes + c * 16);
            const int64_t row = c / kChunksPerRow;
            const int blk = L == Layout::V41 ? int(c % kChunksPerRow) / 2 : int(c % kChunksPerRow);
            sb[it] = ld_byte(scales + row * T::kScaleBytes + blk);
        }
    }
    pdl_trigger();

#pragma unroll
    for (int it = 0; it < ITER; ++it) {
        const int64_t c = int64_t(it) * kDqThreads + threadIdx.x;
        if (c >= kChunks) break;
        const int64_t row = c / kChunksPerRow;
        const int j = int(c % kChunksPerRow);
        uint8_t *orow = a.out + (lp * P + row) * a.out_stride_bytes;
        const uint32_t w[4] = {raw[it].x, raw[it].y, raw[it].z, raw[it].w};
        if constexpr (L == Layout::V41) {
            const float sc = ue8m0_to_f32(sb[it]);
            uint32_t o[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f0 = e4m3x2_to_f32x2(w[q] & 0xFFFFu);
                const float2 f1 = e4m3x2_to_f32x2(w[q] >> 16);
                o[2 * q] = pack_bf16x2(__fmul_rn(f0.x, sc), __fmul_rn(f0.y, sc));
                o[2 * q + 1] = pack_bf16x2(__fmul_rn(f1.x, sc), __fmul_rn(f1.y, sc));
            }
            st_u4(orow + j * 32, make_uint4(o[0], o[1], o[2], o[3]));
            st_u4(orow + j * 32 + 16, make_uint4(o[4], o[5], o[6], o[7]));
        } else {
            const float S = e4m3x2_to_f32x2(sb[it]).x;
            uint32_t o[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float2 f = e2m1x2_to_f32x2((w[q] >> (8 * b)) & 0xFFu);
                    o[4 * q + b] = pack_bf16x2(__fmul_rn(f.x, S), __fmul_rn(f.y, S));
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_u4(orow + j * 64 + 16 * q, make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
        }
    }
}

template <Layout L, int PB>
kvq_status launch_dequant(const DequantArgs &a, int64_t n_pages, cudaStream_t stream) {
    if (n_pages > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    return launch_pdl(dequant_kernel<L, PB>, dim3(unsigned(n_pages)), dim3(kDqThreads), stream, a);
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
