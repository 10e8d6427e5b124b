// kvq_capi.cu -- size queries and status strings of the C ABI.
// Sizes: "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats",
// section 1 (528 / 288 B per token) and section 2 (kv_page_bytes).
#include "kvq_launch.cuh"

using namespace kvq;

extern "C" size_t kvq_bytes_per_token(kvq_layout layout) {
    switch (layout) {
        case KVQ_LAYOUT_V41: return size_t(kTokenBytes<Layout::V41>);
        case KVQ_LAYOUT_V41_FP4: return size_t(kTokenBytes<Layout::FP4>);
        default: return 0;
    }
}

extern "C" size_t kvq_page_bytes(kvq_layout layout, int page_bits) {
    if (page_bits < 1 || page_bits > 16) return 0;
    return (size_t(1) << page_bits) * kvq_bytes_per_token(layout);
}

extern "C" int kvq_page_bits_supported(int page_bits) { return page_bits_supported(page_bits) ? 1 : 0; }

extern "C" const char *kvq_status_string(kvq_status status) {
    switch (status) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_UNSUPPORTED: return "unsupported (no compiled instance)";
        case KVQ_ERR_CAPACITY: return "n exceeds the output capacity";
        case KVQ_ERR_LAUNCH: return "kernel launch failed";
        default: return "unknown status";
    }
}
