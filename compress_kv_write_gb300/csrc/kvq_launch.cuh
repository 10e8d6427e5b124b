// kvq_launch.cuh -- host-side helpers of the C ABI: argument checks, the
// runtime-enum -> template-instance dispatch, and PDL launches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "kvq_device.cuh"

namespace kvq {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch with programmatic stream serialisation, so a kernel can start its
// prologue while its predecessor drains (it waits with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
kvq_status launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return KVQ_ERR_LAUNCH;
    }
    return KVQ_OK;
}

template <typename... KArgs, typename... Args>
kvq_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                      Args &&...args) {
    return launch_pdl_smem(kernel, grid, block, 0, stream, std::forward<Args>(args)...);
}

// Per-device launch limits of a kernel instance launched with CTAs of
// `Threads` threads: opts it into `smem` bytes of dynamic shared memory (once
// per device) and returns the largest grid that is resident at once (blocks
// per SM x SMs).
constexpr int kMaxDevices = 64;

template <auto Kernel, int Threads>
kvq_status resident_grid(size_t smem, int64_t *grid_cap) {
    constexpr int threads = Threads;
    static std::atomic<int> cap[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return KVQ_ERR_LAUNCH;
    }
    int c = cap[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess) {
            (void)cudaGetLastError();
            return KVQ_ERR_LAUNCH;
        }
        int bps = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, Kernel, threads, smem) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return KVQ_ERR_LAUNCH;
        }
        c = (bps > 0 ? bps : 1) * (sms > 0 ? sms : 1);
        cap[dev].store(c, std::memory_order_relaxed);
    }
    *grid_cap = c;
    return KVQ_OK;
}

// page_bits values with compiled instances: pages of 4, 16, 64 and 256 tokens.
inline bool page_bits_supported(int pb) { return pb == 2 || pb == 4 || pb == 6 || pb == 8; }

template <typename F>
kvq_status with_page_bits(int pb, F &&f) {
    switch (pb) {
        case 2: return f(std::integral_constant<int, 2>{});
        case 4: return f(std::integral_constant<int, 4>{});
        case 6: return f(std::integral_constant<int, 6>{});
        case 8: return f(std::integral_constant<int, 8>{});
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

// Compressor ratios compiled in.
template <typename F>
kvq_status with_ratio(int r, F &&f) {
    switch (r) {
        case 1: return f(std::integral_constant<int, 1>{});
        case 2: return f(std::integral_constant<int, 2>{});
        case 4: return f(std::integral_constant<int, 4>{});
        case 128: return f(std::integral_constant<int, 128>{});
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

template <typename F>
kvq_status with_layout(int layout, F &&f) {
    switch (layout) {
        case KVQ_LAYOUT_V41: return f(std::integral_constant<Layout, Layout::V41>{});
        case KVQ_LAYOUT_V41_FP4: return f(std::integral_constant<Layout, Layout::FP4>{});
        default: return KVQ_ERR_INVALID_ARG;
    }
}

template <typename F>
kvq_status with_bool(bool b, F &&f) {
    if (b) return f(std::true_type{});
    return f(std::false_type{});
}

// Common checks of (layout, page_bits) and the pool.
inline kvq_status check_pool(int layout, int page_bits, const void *pool, int64_t pool_slots) {
    if (layout != KVQ_LAYOUT_V41 && layout != KVQ_LAYOUT_V41_FP4) return KVQ_ERR_INVALID_ARG;
    if (page_bits < 1 || page_bits > 16) return KVQ_ERR_INVALID_ARG;
    if (!page_bits_supported(page_bits)) return KVQ_ERR_UNSUPPORTED;
    if (!pool || !aligned(pool, 16)) return KVQ_ERR_INVALID_ARG;
    if (pool_slots <= 0 || (pool_slots & ((int64_t(1) << page_bits) - 1)) != 0)
        return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

}  // namespace kvq
