// kvq_device.cuh -- compile-time layout traits, paged addressing and the
// sm_103a conversion / memory primitives shared by the write-path kernels.
//
// Layouts: "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats",
// section 1 (KVLayoutTraits / PagedKV: page, row and scale-row addresses as
// compile-time constants) and section 2 (kv_page_bytes).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kD = 512;        // head dim
constexpr int kRopeD = 64;     // rotated dims: the last 64
constexpr int kRopeStart = kD - kRopeD;
constexpr int kBlock = 32;     // values per quant block
constexpr int kNBlk = kD / kBlock;

static_assert(kD % kBlock == 0, "quant blocks must tile the head dim");
static_assert(kRopeD <= kD && kRopeD % 2 == 0, "rope dims are pairs inside the head");
static_assert(kRopeStart % kBlock == 0, "rope dims start on a block boundary");

enum class Layout : int { V41 = KVQ_LAYOUT_V41, FP4 = KVQ_LAYOUT_V41_FP4 };

template <Layout L>
struct LayoutTraits;

// V41: 512 e4m3 codes, then (in the scale area) 16 ue8m0 bytes.
template <>
struct LayoutTraits<Layout::V41> {
    static constexpr int kCodeBytes = kD;
    static constexpr int kScaleBytes = kNBlk;
};

// V41_FP4: 256 bytes of packed e2m1 codes, then a 32-byte scale row:
// 16 e4m3 scales and 16 bytes of zero padding (288 B/token in all).
template <>
struct LayoutTraits<Layout::FP4> {
    static constexpr int kCodeBytes = kD / 2;
    static constexpr int kScaleBytes = 2 * kNBlk;
};

template <Layout L>
constexpr int kTokenBytes = LayoutTraits<L>::kCodeBytes + LayoutTraits<L>::kScaleBytes;
static_assert(kTokenBytes<Layout::V41> == 528, "V41 is 528 B/token");
static_assert(kTokenBytes<Layout::FP4> == 288, "V41_FP4 is 288 B/token");

// A page of P = 2^PageBits tokens: P code rows, then P scale rows.
template <Layout L, int PageBits>
struct PagedKV {
    static_assert(PageBits >= 1 && PageBits <= 16, "page_bits out of range");
    using T = LayoutTraits<L>;
    static constexpr int64_t kPage = int64_t(1) << PageBits;
    static constexpr int64_t kPageBytes = kPage * kTokenBytes<L>;
    static_assert(kPageBytes % 16 == 0, "pages keep 16-byte alignment");

    __device__ __forceinline__ static uint8_t *code_row(uint8_t *pool, int64_t slot) {
        return pool + (slot >> PageBits) * kPageBytes + (slot & (kPage - 1)) * T::kCodeBytes;
    }
    __device__ __forceinline__ static uint8_t *scale_row(uint8_t *pool, int64_t slot) {
        return pool + (slot >> PageBits) * kPageBytes + kPage * T::kCodeBytes +
               (slot & (kPage - 1)) * T::kScaleBytes;
    }
};

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: wait for the predecessor grid's memory
// before the first global read; let the successor grid start launching once
// this CTA's loads are issued.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- memory
// Streaming (read-once) 16-byte loads of input rows: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_u4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// One 32-byte store per lane (p 32-byte aligned).
__device__ __forceinline__ void st_v8(void *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// ---------------------------------------------------------------- conversions
// Two fp32 -> packed e4m3x2, round to nearest even, saturating to +-448.
// The first operand of cvt goes to the upper byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> packed e2m1x2 (lo in bits 0-3), round to nearest even,
// saturating to +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "mov.b32 %0, {t, 0, 0, 0};\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Packed e4m3x2 (low byte first) -> two fp32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t v) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v));
    float2 f;
    asm("{\n\t.reg .f16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t"
        "cvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f.x), "=f"(f.y)
        : "r"(h));
    return f;
}

// Packed e2m1x2 (low nibble first) -> two fp32 (exact).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t v) {
    uint32_t h;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h)
        : "r"(v));
    float2 f;
    asm("{\n\t.reg .f16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t"
        "cvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f.x), "=f"(f.y)
        : "r"(h));
    return f;
}

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 rounded to the nearest bf16 (ties to even), returned as fp32.
__device__ __forceinline__ float round_bf16(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return __uint_as_float(uint32_t(r) << 16);
}

// 2^(byte - 127) for a ue8m0 scale byte; 0xFF is NaN (OCP MX).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t byte) {
    if (byte == 0u) return __uint_as_float(0x00400000u);  // 2^-127, subnormal
    if (byte == 255u) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(byte << 23);
}

// max(a, b, c) in one instruction (three-operand fp32 max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// |x| bits, so that an unsigned max is the magnitude max (finite inputs).
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// 2^x with the hardware approximation (softmax weights only).
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// 1/sqrt(x) with the hardware approximation (relative error below 2^-22),
// for x >= eps > 0: the RMSNorm scale.
__device__ __forceinline__ float rsqrt_approx(float x) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void raise_err(int32_t *err, int32_t bit) {
    if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- packed fp32x2
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pr, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pr, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pc, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pr, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Per-thread async copies global -> shared (LSU path, no register cost),
// grouped per thread with commit / wait_group; dst is a shared-window
// address (32 bits, from smem_addr).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One fp32 float4 from a streamed (read-once) row.
__device__ __forceinline__ float4 ld_f4(const float *p) {
    uint4 r = ld_stream_u4(p);
    return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z),
                       __uint_as_float(r.w));
}

constexpr float kLog2e = 1.4426950408889634f;

// L2 prefetch hints.  They move lines into L2 only (never into L1 or
// registers), and every write of any grid reaches L2, so issuing them before
// griddepcontrol.wait cannot make a later load see stale data.
// Bulk form: p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Into this SM's L1 as well; issue it only after griddepcontrol.wait.
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Shared-memory loads from a shared-window address.
__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}

// ---------------------------------------------------------------- scales
// V41: scale byte = exponent field of amax - 8, clamped at 0 (OCP MX shared
// exponent floor(log2 amax) - emax(E4M3)); the values are then multiplied by
// 2^(127 - byte), exact for every byte the rule can produce (<= 246).
__device__ __forceinline__ uint32_t v41_scale_byte(uint32_t amax_bits) {
    int e = int((amax_bits >> 23) & 0xFFu) - 8;
    return uint32_t(e < 0 ? 0 : e);
}
__device__ __forceinline__ float v41_multiplier(uint32_t byte) {
    return __uint_as_float((254u - byte) << 23);
}

// V41_FP4: scale = e4m3(amax / 6) with a correctly rounded division.
__device__ __forceinline__ uint32_t fp4_scale_byte(uint32_t amax_bits) {
    float s = __fdiv_rn(__uint_as_float(amax_bits), 6.0f);
    return cvt_e4m3x2(s, 0.0f) & 0xFFu;
}

}  // namespace kvq
