// kvq_quant.cuh -- the quantization rule of one cache row, shared by the
// quantize-append kernel (kvq_append.cu) and the decode that appends its
// step's token itself (kvq_alu.cuh), so that both write the same bytes.
//
// The rule ("Dynamic KV Cache Quantization for Fast LLM Inference", section
// "Understanding Dynamic Quantization Techniques for KV Caches (e.g., INT8,
// INT4)"): the scale comes from the row's (or 32-channel group's) own
// largest magnitude at run time and the code is the rounded quotient.
// Every fp32 step is an explicitly rounded IEEE operation (__fdiv_rn,
// __fsub_rn, cvt.rni), so the codes do not depend on compiler contraction.
//
// Lane layout: a row (head_dim channels) is held by LPR = head_dim / 16
// consecutive lanes, 16 channels (two 16-byte words of bf16) each; the
// absmax (or min/max) is a shuffle reduction among them (INT4: a 32-channel
// group is two lanes, xor 1).  Every lane of the warp must call these
// functions together (full-mask shuffles).
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// Round-half-even of fl(x_i / s), for |x_i / s| <= 128, into q_i.  With r
// within 2 ulps of 1/s (the hardware reciprocal), y = RN(x r) lies within
// 1.25 * 2^-22 * |x / s| (< 2^-14.6 here) of x / s, and fl(x / s) within
// 2^-17 of it, so unless y is within 2^-14 of a half-integer both round to
// the same integer.  If any element of the warp is that close, or r overflowed
// (a row of tiny magnitudes: x r is then infinite or NaN), the warp takes the
// exact quotient for those elements (a warp-uniform branch: rare, and the
// division is not evaluated otherwise).
// The hardware reciprocal (rcp.approx: within one ulp), for the fast
// quotients above; a zero or subnormal s gives inf, which takes the exact path.
__device__ __forceinline__ float approx_rcp(float s) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
    return r;
}

// INT8: the same rounding as rne_quotients, with each code left as the low
// byte of t = RN(y + 1.5 * 2^23) (whose low mantissa bits hold the integer
// RNE(y) for |y| < 2^22), packed four to a word.  Pairs of elements go through
// the packed fp32 operations (each half one correctly rounded IEEE operation,
// the same bits as the scalar ones): y = x r, t = y + M, and the rounding
// residual y - (t - M), exact for |y| < 2^22.
template <int N>
__device__ __forceinline__ void rne_codes_s8(const float* x, float s, float r, uint32_t* wd) {
    constexpr float M = 12582912.0f;  // 1.5 * 2^23
    uint32_t t[N];
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 y = __fmul2_rn(make_float2(x[i], x[i + 1]), make_float2(r, r));
        const float2 tf = __fadd2_rn(y, make_float2(M, M));
        const float2 back = __fadd2_rn(tf, make_float2(-M, -M));
        const float2 d = __fadd2_rn(y, make_float2(-back.x, -back.y));
        t[i] = __float_as_uint(tf.x);
        t[i + 1] = __float_as_uint(tf.y);
        dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
    }
    const bool r_inf = !(r <= 0x1.fffffep127f);
    if (__any_sync(0xffffffffu, !(dmax < 0.5f - 0x1p-14f) || r_inf)) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float y = __fmul_rn(x[i], r);
            if (r_inf || !(fabsf(__fsub_rn(y, rintf(y))) < 0.5f - 0x1p-14f))
                t[i] = (uint32_t)__float2int_rn(__fdiv_rn(x[i], s));
        }
    }
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
        wd[k] = __byte_perm(__byte_perm(t[4 * k], t[4 * k + 1], 0x0040), __byte_perm(t[4 * k + 2], t[4 * k + 3], 0x0040),
                            0x5410);
}

// The same rounding as integers: q_i = the bits of t = RN(y + 1.5 * 2^23)
// less those of 1.5 * 2^23 (the two's-complement integer RNE(y) for
// |y| < 2^22), by the packed operations as above.
template <int N>
__device__ __forceinline__ void rne_quotients(const float* x, float s, float r, int* q) {
    constexpr float M = 12582912.0f;  // 1.5 * 2^23
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 y = __fmul2_rn(make_float2(x[i], x[i + 1]), make_float2(r, r));
        const float2 tf = __fadd2_rn(y, make_float2(M, M));
        const float2 back = __fadd2_rn(tf, make_float2(-M, -M));
        const float2 d = __fadd2_rn(y, make_float2(-back.x, -back.y));
        q[i] = (int)(__float_as_uint(tf.x) - __float_as_uint(M));
        q[i + 1] = (int)(__float_as_uint(tf.y) - __float_as_uint(M));
        dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
    }
    const bool r_inf = !(r <= 0x1.fffffep127f);
    if (__any_sync(0xffffffffu, !(dmax < 0.5f - 0x1p-14f) || r_inf)) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float y = __fmul_rn(x[i], r);
            if (r_inf || !(fabsf(__fsub_rn(y, rintf(y))) < 0.5f - 0x1p-14f)) q[i] = __float2int_rn(__fdiv_rn(x[i], s));
        }
    }
}

// fl(x_i / s) where only its E4M3 rounding matters: with r within 2 ulps of
// 1/s, y = RN(x r) is within 1.25 * 2^-22 relative (6 fp32 ulps) of
// fl(x / s); E4M3 rounding (3 mantissa bits) can only differ if y is within
// 8 ulps of a midpoint between E4M3 values (fp32 mantissa bits 19..0 =
// 0x80000) or in the E4M3 subnormal range; there the exact
// quotient is used, and for every element if r overflowed (a warp-uniform
// branch, as above).
__device__ __forceinline__ bool e4m3_needs_exact(float y) {
    const uint32_t bits = __float_as_uint(y);
    const int e = (int)((bits >> 23) & 0xFFu);
    const int low = (int)(bits & 0xFFFFFu);
    return abs(low - 0x80000) <= 8 || (e < 127 - 6 && y != 0.0f);
}
template <int N>
__device__ __forceinline__ void e4m3_quotients(const float* x, float s, float r, float* y) {
    const bool r_inf = !(r <= 0x1.fffffep127f);
    bool slow = r_inf;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        y[i] = __fmul_rn(x[i], r);
        slow |= e4m3_needs_exact(y[i]);
    }
    if (__any_sync(0xffffffffu, slow)) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (r_inf || e4m3_needs_exact(y[i])) y[i] = __fdiv_rn(x[i], s);
    }
}

// The codes of one lane's 16 channels and its row's (or group's) scale:
//   8-bit schemes: w[0..3] = 16 codes (one byte each), scale (fp32);
//   INT4: w[0..1] = 16 nibbles (even channel low), scale (symmetric: fp32)
//   or sh, zh (asymmetric: the fp16 bits of the group's scale and zero).
struct LaneCodes {
    uint32_t w[4];
    float scale;
    __half sh, zh;
};

template <int SCHEME, int LPR>
__device__ __forceinline__ LaneCodes quantize_lane(const uint4 (&raw)[2]) {
    LaneCodes out;
    float x[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {raw[h].x, raw[h].y, raw[h].z, raw[h].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[8 * h + 2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
            x[8 * h + 2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
        }
    }
    if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN || SCHEME == KVQ_FP8E4M3_TOKEN) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        constexpr float QMAX = SCHEME == KVQ_INT8_SYM_TOKEN ? 127.0f : 448.0f;
        const bool zero_row = (a == 0.0f);
        const float scale = zero_row ? 1.0f : __fdiv_rn(a, QMAX);
        const float rcp = approx_rcp(scale);
        if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN) {
            // |x| <= a gives |x / scale| <= 127 (1 + 2^-24) < 127.5: codes in
            // [-127, 127] without clamping; a zero row's x are +-0: codes 0
            rne_codes_s8<16>(x, scale, rcp, out.w);
        } else {
            float y[16];
            e4m3_quotients<16>(x, scale, rcp, y);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[4 * k], y[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
                const uint32_t hi =
                    __nv_cvt_float2_to_fp8x2(make_float2(y[4 * k + 2], y[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
                out.w[k] = zero_row ? 0u : (lo | (hi << 16));  // a zero row (even of -0) codes +0
            }
        }
        out.scale = scale;
    } else if constexpr (SCHEME == KVQ_INT4_SYM_G32) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        // scale = a / 7 in fp32 (1 for an all-zero group, whose x are +-0
        // and so round to code 0); |x / scale| <= 7 (1 + 2^-24): codes in
        // [-7, 7] without clamping
        const float sc = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 7.0f);
        const float rcp = approx_rcp(sc);
        int q[16];
        rne_quotients<16>(x, sc, rcp, q);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) w |= ((uint32_t)q[8 * h + i] & 0xFu) << (4 * i);
            out.w[h] = w;
        }
        out.scale = sc;
    } else {
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            mn = fminf(mn, x[i]);
            mx = fmaxf(mx, x[i]);
        }
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        const __half zh = __float2half_rd(mn);
        const float zf = __half2float(zh);
        __half sh = __float2half_ru(__fdiv_rn(__fsub_rn(mx, zf), 15.0f));
        if (__half2float(sh) == 0.0f) sh = __float2half(1.0f);
        const float sf = __half2float(sh);
        const float rcp = approx_rcp(sf);
        float d[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) d[i] = __fsub_rn(x[i], zf);
        // zf <= mn and sf >= (mx - zf) / 15 (both rounded outwards): the
        // quotients lie in [0, 15] up to the last place; clamp anyway
        int q[16];
        rne_quotients<16>(d, sf, rcp, q);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) w |= (uint32_t)max(0, min(15, q[8 * h + i])) << (4 * i);
            out.w[h] = w;
        }
        out.sh = sh;
        out.zh = zh;
    }
    return out;
}

// Stores a lane's codes and (from the lanes that own them) the scales and
// zero-points of row `row` of pools laid out as the cache's: codes
// [row][code bytes per token], scales / zeros [row][per-token entries].  The
// same layout serves a page pool and a shared-memory stage of the decode.
// `li` is the lane's index in its row.
template <int SCHEME, int D>
__device__ __forceinline__ void store_lane(const LaneCodes& c, uint8_t* codes, void* scales, void* zeros,
                                           int64_t row, int li) {
    if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN || SCHEME == KVQ_FP8E4M3_TOKEN) {
        *reinterpret_cast<uint4*>(codes + row * D + li * 16) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
        if (li == 0) static_cast<float*>(scales)[row] = c.scale;
    } else {
        *reinterpret_cast<uint2*>(codes + row * (D / 2) + li * 8) = make_uint2(c.w[0], c.w[1]);
        if ((li & 1) == 0) {
            const int64_t gi = row * (D / 32) + li / 2;
            if constexpr (SCHEME == KVQ_INT4_SYM_G32) {
                static_cast<float*>(scales)[gi] = c.scale;
            } else {
                static_cast<__half*>(scales)[gi] = c.sh;
                static_cast<__half*>(zeros)[gi] = c.zh;
            }
        }
    }
}

}  // namespace kvq
