// kvq_store.cuh -- the arguments of the KV store kernels ("[sglang] DeepSeek
// V4.1 Paged KV Cache: V41 and FP4 formats", section 1 store_row), shared by
// the persistent kernels of kvq_store.cu and the small-batch kernel of
// kvq_store_small.cu.
#pragma once
#include "kvq_launch.cuh"

namespace kvq {

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
    // token ranges of the persistent kernels (set by partition()): per_warp
    // tokens per warp, one more for the first extra + skew warps, one fewer
    // for the last skew warps
    int64_t per_warp;
    int64_t extra;
    int64_t skew;
    int64_t warps;
};

// Batches up to this many tokens take one four-warp CTA per token
// (kvq_store_small.cu), larger ones the persistent kernels: measured at 512,
// 1024 and 2048 tokens, the CTA per token wins up to 1024 with RoPE or the
// norm and for V41_FP4, and ties at 512 for the plain V41 store.
constexpr int64_t kStoreSmallMax = 1024;
constexpr int64_t kStoreSmallMaxPlainV41 = 512;
inline int64_t store_small_max(int layout, bool norm, bool rope) {
    return (layout == KVQ_LAYOUT_V41 && !norm && !rope) ? kStoreSmallMaxPlainV41 : kStoreSmallMax;
}

// One CTA per token: layout, page_bits, input dtype, index dtype and flags
// as validated by kvq_store.
kvq_status launch_store_small(int layout, int page_bits, bool bf16, bool loc64, bool norm, bool rope,
                              const StoreArgs &a, cudaStream_t stream);

}  // namespace kvq
