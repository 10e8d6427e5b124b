// kvq_translate.cu -- the full -> SWA slot translation, hoisted to once per
// step ("[sglang] Hoist DSv4 draft-extend SWA write locs", sections 1-2):
// out[i] = full_to_swa[full_loc[i]] as int32 for i < n, out[n:capacity] = 0,
// so the same preallocated buffer serves every layer's store of the step.
#include "kvq_launch.cuh"

namespace kvq {
namespace {

constexpr int kTrThreads = 256;
constexpr int kTrPerThread = 4;

struct TranslateArgs {
    const void *loc;
    int64_t n;
    const int32_t *table;
    int64_t full_slots;
    int32_t *out;
    int64_t capacity;
    int32_t *err;
};

template <bool kLoc64>
__global__ void __launch_bounds__(kTrThreads) translate_kernel(const TranslateArgs a) {
    const int64_t base = (int64_t(blockIdx.x) * kTrThreads + threadIdx.x) * kTrPerThread;
    pdl_wait();
    int64_t l[kTrPerThread];
#pragma unroll
    for (int q = 0; q < kTrPerThread; ++q) {
        const int64_t i = base + q;
        l[q] = -2;
        if (i < a.n)
            l[q] = kLoc64 ? __ldg(static_cast<const int64_t *>(a.loc) + i)
                          : int64_t(__ldg(static_cast<const int32_t *>(a.loc) + i));
    }
    int32_t v[kTrPerThread];
    bool bad = false;
#pragma unroll
    for (int q = 0; q < kTrPerThread; ++q) {
        v[q] = 0;
        if (base + q < a.n) {
            if (l[q] >= 0 && l[q] < a.full_slots) {
                v[q] = __ldg(a.table + l[q]);
            } else {
                v[q] = -1;
                bad = true;
            }
        }
    }
    pdl_trigger();
    if (bad) raise_err(a.err, KVQ_DEVERR_LOC);
#pragma unroll
    for (int q = 0; q < kTrPerThread; ++q)
        if (base + q < a.capacity) a.out[base + q] = v[q];
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_translate_loc(const void *full_loc, kvq_index_dtype loc_dtype, int64_t n,
                                        const int32_t *full_to_swa, int64_t full_slots, int32_t *out,
                                        int64_t out_capacity, int32_t *err,
                                        struct CUstream_st *stream) {
    if (loc_dtype != KVQ_I32 && loc_dtype != KVQ_I64) return KVQ_ERR_INVALID_ARG;
    if (n < 0 || out_capacity < 0 || full_slots < 0) return KVQ_ERR_INVALID_ARG;
    if (n > out_capacity) return KVQ_ERR_CAPACITY;
    if (n > 0 && (!full_loc || !aligned(full_loc, loc_dtype == KVQ_I64 ? 8 : 4)))
        return KVQ_ERR_INVALID_ARG;
    if (n > 0 && full_slots > 0 && (!full_to_swa || !aligned(full_to_swa, 4))) return KVQ_ERR_INVALID_ARG;
    if (out_capacity > 0 && (!out || !aligned(out, 4))) return KVQ_ERR_INVALID_ARG;
    if (err && !aligned(err, 4)) return KVQ_ERR_INVALID_ARG;
    if (out_capacity == 0) return KVQ_OK;

    TranslateArgs a;
    a.loc = full_loc;
    a.n = n;
    a.table = full_to_swa;
    a.full_slots = full_slots;
    a.out = out;
    a.capacity = out_capacity;
    a.err = err;
    const int64_t per_block = int64_t(kTrThreads) * kTrPerThread;
    const int64_t blocks = (out_capacity + per_block - 1) / per_block;
    if (blocks > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return with_bool(loc_dtype == KVQ_I64, [&](auto L64) {
        return launch_pdl(translate_kernel<decltype(L64)::value>, dim3(unsigned(blocks)),
                          dim3(kTrThreads), s, a);
    });
}
