// kvq_device.cuh -- device-side building blocks shared by the kernels:
// error flags, 16-byte cp.async copies with L2 policies, exact code -> float
// conversions, mixed-precision and dp4a dot-product steps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start before the kernel ahead of it in the stream has
// finished; grid_dependency_wait() returns once that kernel has completed and
// its memory operations are visible (at once if there is no such kernel).
// grid_launch_dependents() lets the kernel after this one be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// 16-byte asynchronous copy global -> shared (bypassing L1).  No L2
// cache-policy operand: on sm_103a the cache-hinted form of this copy raised
// "illegal instruction" in a minimal streaming kernel whose unhinted twin ran
// clean, so no copy in this library carries one.  Completion is tracked per
// thread (commit / wait groups, or an mbarrier arrival).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// Brings the line holding `p` into L2 (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// 8-byte asynchronous copy global -> shared (through L1; both addresses
// 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- exact conversions of stored codes to fp32 -----------------------------

// Four int8 codes (one 32-bit word, little-endian) -> four floats, exactly.
// Each byte is made unsigned by flipping its top bit (c + 128), placed in the
// low mantissa byte of 2^23 (the float 8388608 + c + 128), and the bias is
// subtracted: the result is the integer c, with no conversion instruction.
__device__ __forceinline__ void s8x4_to_float(uint32_t w, float f[4]) {
    const uint32_t u = w ^ 0x80808080u;
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - 8388736.0f;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - 8388736.0f;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - 8388736.0f;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - 8388736.0f;
}

// Four E4M3 codes -> four floats, exactly (via two half2 conversions).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float f[4]) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

// Two mixed-precision FMAs: acc0 += lo(q2) * lo(c2), acc1 += hi(q2) * hi(c2),
// fp16 operands, fp32 accumulation (the product is exact in fp32).
__device__ __forceinline__ void mfma_h2(uint32_t q2, uint32_t c2, float& acc0, float& acc1) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %2;\n\t"
        "mov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(q2), "r"(c2));
}

// The same two products accumulated into one fp32 value.
__device__ __forceinline__ void mfma_h2_1(uint32_t q2, uint32_t c2, float& acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(q2), "r"(c2));
}

// 4-way byte dot products accumulated in int32 (dp4a).  Suffixes give the
// signedness of (a, b): s = signed bytes, u = unsigned bytes.
__device__ __forceinline__ int dp4a_ss(int a, int b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(int a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two E4M3 codes (low 16 bits) -> exact fp16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t w16) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w16 & 0xFFFFu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

}  // namespace kvq
