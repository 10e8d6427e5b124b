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

// Small batches take the small-batch kernel (kvq_store_small.cu): one
// four-warp CTA per token, or per two tokens in the middle range, where one
// CTA per token costs more to schedule and one warp per token has the longer
// chain.  Larger ones take the persistent kernels.  Measured from 64 to 4096
// tokens; the limits are the last sizes at which each form wins:
constexpr int64_t kSmallNormMax = 1024;     // with the norm: one token per CTA up to here
constexpr int64_t kSmallRopeOneMax = 512;   // V41 store + RoPE: one token per CTA ...
constexpr int64_t kSmallRopeTwoMax = 3072;  // ... then two, up to here
constexpr int64_t kSmallOneMax = 256;       // plain V41 and V41_FP4 without the norm: one ...
constexpr int64_t kSmallTwoMax = 1536;      // ... then two, up to here
// Tokens per CTA of the small-batch kernel for a batch of n tokens (0: the
// persistent kernels).
inline int store_small_tokens_per_cta(int layout, bool norm, bool rope, int64_t n) {
    if (norm) return n <= kSmallNormMax ? 1 : 0;
    if (layout == KVQ_LAYOUT_V41 && rope) return n <= kSmallRopeOneMax ? 1 : n <= kSmallRopeTwoMax ? 2 : 0;
    return n <= kSmallOneMax ? 1 : n <= kSmallTwoMax ? 2 : 0;
}

// One four-warp CTA per token (tokens_per_cta 1) or per two tokens (2):
// layout, page_bits, input dtype, index dtype and flags as validated by
// kvq_store.
kvq_status launch_store_small(int layout, int page_bits, bool bf16, bool loc64, bool norm, bool rope,
                              int tokens_per_cta, const StoreArgs &a, cudaStream_t stream);

}  // namespace kvq
