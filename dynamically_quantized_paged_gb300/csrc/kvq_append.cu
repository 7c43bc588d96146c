// kvq_append.cu -- quantize-append (K1) and the table check (K4).
//
// Quantize-append follows "Dynamic KV Cache Quantization for Fast LLM
// Inference", section "Understanding Dynamic Quantization Techniques for KV
// Caches (e.g., INT8, INT4)": the scale comes from the row's own largest
// magnitude at run time, the code is the rounded quotient; and "What is KV
// Cache Optimization? ...", section "Technical Architecture": captured K/V
// rows are quantized and written into non-contiguous pages.
//
// Work layout: one row = the head_dim bf16 values of one (token, KV head,
// K-or-V).  A lane holds 16 channels (two 128-bit loads) of both the K row
// and the V row of one (token, KV head), so head_dim/16 lanes hold the pair
// and the slot, page and head arithmetic is shared by its two rows.  The
// absmax (or min/max) is a warp-shuffle reduction inside the row's lanes.  Every fp32 step is an
// explicitly rounded IEEE operation (__fdiv_rn, __fsub_rn, cvt.rni), so the
// codes do not depend on compiler contraction.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_UNROLL = 2;  // (token, head) pairs per lane whose loads are issued together

// n / d for 0 <= n < 2^31 as (n * mul) >> shift, with mul and shift from
// magic_divisor (below).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint64_t mul, int shift) {
    return (uint32_t)(((uint64_t)n * mul) >> shift);
}

// Round-half-even of fl(x_i / s), for |x_i / s| <= 128, into q_i.  With r =
// RN(1/s), y = RN(x r) lies within 1.5 * 2^-23 * |x / s| (< 2^-15 here) of
// fl(x / s), so unless y is within 2^-14 of a half-integer both round to the
// same integer.  If any element of the warp is that close, or r overflowed
// (a row of tiny magnitudes: x r is then infinite or NaN), the warp takes the
// exact quotient for those elements (a warp-uniform branch: rare, and the
// division is not evaluated otherwise).
template <int N>
__device__ __forceinline__ void rne_quotients(const float* x, float s, float r, int* q) {
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float y = __fmul_rn(x[i], r);
        const float c = rintf(y);
        q[i] = (int)c;
        dmax = fmaxf(dmax, fabsf(__fsub_rn(y, c)));
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

// fl(x_i / s) where only its E4M3 rounding matters: y = RN(x r) is within 3
// fp32 ulps of fl(x / s); E4M3 rounding (3 mantissa bits) can only differ
// if y is within a few ulps of a midpoint between E4M3 values (fp32 mantissa
// bits 19..0 = 0x80000) or in the E4M3 subnormal range; there the exact
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

// One lane's 16 channels of one row (K or V of a (token, head)), quantized
// and stored.  LPR lanes hold a row; `li` is this lane's index in it.
template <int SCHEME, int D, int LPR>
__device__ __forceinline__ void quantize_store(const AppendParams& p, const uint4 (&raw)[2], int kv, bool valid,
                                               int64_t prow, int li) {
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
        const float rcp = __frcp_rn(scale);
        uint32_t wd[4];
        if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN) {
            // |x| <= a gives |x / scale| <= 127 (1 + 2^-24) < 127.5: codes in
            // [-127, 127] without clamping; a zero row's x are +-0: codes 0
            int q[16];
            rne_quotients<16>(x, scale, rcp, q);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                wd[k] = (uint32_t)(q[4 * k] & 0xFF) | ((uint32_t)(q[4 * k + 1] & 0xFF) << 8) |
                        ((uint32_t)(q[4 * k + 2] & 0xFF) << 16) | ((uint32_t)(q[4 * k + 3] & 0xFF) << 24);
        } else {
            float y[16];
            e4m3_quotients<16>(x, scale, rcp, y);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[4 * k], y[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
                const uint32_t hi =
                    __nv_cvt_float2_to_fp8x2(make_float2(y[4 * k + 2], y[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
                wd[k] = zero_row ? 0u : (lo | (hi << 16));  // a zero row (even of -0) codes +0
            }
        }
        if (valid) {
            uint8_t* dst = (kv ? p.v_codes : p.k_codes) + prow * D + li * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            if (li == 0) static_cast<float*>(kv ? p.v_scales : p.k_scales)[prow] = scale;
        }
    } else {
        // INT4: a 32-channel group is two lanes (xor 1)
        uint32_t packed[2];
        if constexpr (SCHEME == KVQ_INT4_SYM_G32) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            // scale = a / 7 in fp32 (1 for an all-zero group, whose x are +-0
            // and so round to code 0); |x / scale| <= 7 (1 + 2^-24): codes in
            // [-7, 7] without clamping
            const float sc = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 7.0f);
            const float rcp = __frcp_rn(sc);
            int q[16];
            rne_quotients<16>(x, sc, rcp, q);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) w |= ((uint32_t)q[8 * h + i] & 0xFu) << (4 * i);
                packed[h] = w;
            }
            if (valid && (li & 1) == 0)
                static_cast<float*>(kv ? p.v_scales : p.k_scales)[prow * (D / 32) + li / 2] = sc;
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
            const float rcp = __frcp_rn(sf);
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
                packed[h] = w;
            }
            if (valid && (li & 1) == 0) {
                const int64_t gi = prow * (D / 32) + li / 2;
                static_cast<__half*>(kv ? p.v_scales : p.k_scales)[gi] = sh;
                static_cast<__half*>(kv ? p.v_zeros : p.k_zeros)[gi] = zh;
            }
        }
        if (valid) {
            uint8_t* dst = (kv ? p.v_codes : p.k_codes) + prow * (D / 2) + li * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
        }
    }
}

// One lane holds 16 channels (two 16-byte loads) of both the K row and the V
// row of a (token, KV head) pair; LPR = D / 16 lanes hold a pair, a warp
// 32 / LPR pairs.  The slot, page and head arithmetic is done once for the
// two rows.
template <int SCHEME, int D>
__global__ void __launch_bounds__(APPEND_THREADS, 2) append_kernel(AppendParams p) {
    constexpr int LPR = D / 16;    // lanes per pair
    constexpr int PPW = 32 / LPR;  // pairs per warp
    // a decode launched next may be scheduled now (it waits for this grid to
    // complete before reading anything)
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int li = lane % LPR;
    const int H = p.num_kv_heads;
    const int64_t pairs = (int64_t)p.num_tokens * H;
    const int64_t warp_id = ((int64_t)blockIdx.x * APPEND_THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * APPEND_THREADS) >> 5;
    const int64_t stride = nwarps * PPW;

    // the trip count is the same for every lane of the warp (pairs past the
    // end are carried as invalid), so the warp collectives see all lanes
    for (int64_t pb = warp_id * PPW; pb < pairs; pb += stride * APPEND_UNROLL) {
        int64_t slot[APPEND_UNROLL];
        uint4 rk[APPEND_UNROLL][2], rv[APPEND_UNROLL][2];
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {
            const int64_t pi = pb + lane / LPR + u * stride;
            slot[u] = -1;
            rk[u][0] = rk[u][1] = rv[u][0] = rv[u][1] = make_uint4(0u, 0u, 0u, 0u);
            if (pi < pairs) {
                const uint32_t t = fast_div((uint32_t)pi, p.heads_mul, p.heads_shift);
                slot[u] = __ldg(p.slot_mapping + t);
                const uint4* ks = reinterpret_cast<const uint4*>(p.k + pi * D + li * 16);
                const uint4* vs = reinterpret_cast<const uint4*>(p.v + pi * D + li * 16);
                rk[u][0] = __ldg(ks);
                rk[u][1] = __ldg(ks + 1);
                rv[u][0] = __ldg(vs);
                rv[u][1] = __ldg(vs + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {
            const int64_t pi = pb + lane / LPR + u * stride;
            int64_t sl = pi < pairs ? slot[u] : -1;
            if (sl >= p.num_slots) {
                if (li == 0) flag_error(p.err, ERR_BAD_TABLE);
                sl = -1;
            }
            const bool valid = sl >= 0;
            const uint32_t t = fast_div((uint32_t)(pi < pairs ? pi : 0), p.heads_mul, p.heads_shift);
            const int h = (int)((uint32_t)(pi < pairs ? pi : 0) - t * (uint32_t)H);
            // pool row of this (slot, head): [page][head][offset]
            const uint32_t pg = valid ? fast_div((uint32_t)sl, p.page_mul, p.page_shift) : 0u;
            const uint32_t off = valid ? (uint32_t)sl - pg * (uint32_t)p.page_size : 0u;
            const int64_t prow = ((int64_t)pg * H + h) * p.page_size + off;
            quantize_store<SCHEME, D, LPR>(p, rk[u], 0, valid, prow, li);
            quantize_store<SCHEME, D, LPR>(p, rv[u], 1, valid, prow, li);
        }
    }
}

// K4: every page a sequence uses must lie in the pool, and the sequence must
// fit its table row.  Without seq_lens, every entry must be -1 or in the pool.
__global__ void validate_kernel(int num_pages, int page_size, const int32_t* block_table,
                                const int32_t* seq_lens, int B, int max_pages, unsigned* err) {
    const int64_t n = (int64_t)B * max_pages;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / max_pages);
        const int j = (int)(i % max_pages);
        const int32_t e = block_table[i];
        if (seq_lens) {
            const int32_t L = seq_lens[b];
            if (j == 0 && (L < 0 || (int64_t)L > (int64_t)max_pages * page_size))
                flag_error(err, ERR_BAD_TABLE);
            const int64_t used = (L <= 0) ? 0 : ((int64_t)L + page_size - 1) / page_size;
            if (j < used && (e < 0 || e >= num_pages)) flag_error(err, ERR_BAD_TABLE);
        } else if (e < -1 || e >= num_pages) {
            flag_error(err, ERR_BAD_TABLE);
        }
    }
}

// Division by a runtime divisor d >= 1 for dividends 0 <= n < 2^31 as one
// 64-bit product and shift: with l = ceil(log2 d) and m = ceil(2^(32+l) / d),
// floor(n m / 2^(32+l)) = floor(n / d), because m d - 2^(32+l) < d makes the
// product exceed n / d by less than n / 2^(32+l) < 1 / (2d), which cannot
// reach the next integer (Granlund and Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994, the round-up method).
void magic_divisor(uint32_t d, uint64_t* mul, int* shift) {
    int l = 0;
    while ((1ull << l) < d) ++l;
    const unsigned __int128 num = (unsigned __int128)1 << (32 + l);
    *mul = (uint64_t)((num + d - 1) / d);
    *shift = 32 + l;
}

template <int SCHEME, int D>
cudaError_t launch_append_t(AppendParams p, cudaStream_t s) {
    magic_divisor((uint32_t)p.num_kv_heads, &p.heads_mul, &p.heads_shift);
    magic_divisor((uint32_t)p.page_size, &p.page_mul, &p.page_shift);
    // as many CTAs as there are pair groups (small appends are latency-bound),
    // at most one wave of 2 resident CTAs per SM (then each lane group
    // loops, APPEND_UNROLL pairs at a time)
    constexpr int PPB = (APPEND_THREADS / 32) * (32 / (D / 16));
    const int64_t pairs = (int64_t)p.num_tokens * p.num_kv_heads;
    int64_t blocks = (pairs + PPB - 1) / PPB;
    const int64_t cap = (int64_t)device_sm_count() * 2;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    append_kernel<SCHEME, D><<<(unsigned)blocks, APPEND_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int scheme, int head_dim, cudaStream_t s) {
    if (head_dim == 128) {
        if (scheme == KVQ_INT8_SYM_TOKEN) return launch_append_t<KVQ_INT8_SYM_TOKEN, 128>(p, s);
        if (scheme == KVQ_FP8E4M3_TOKEN) return launch_append_t<KVQ_FP8E4M3_TOKEN, 128>(p, s);
        if (scheme == KVQ_INT4_SYM_G32) return launch_append_t<KVQ_INT4_SYM_G32, 128>(p, s);
        return launch_append_t<KVQ_INT4_ASYM_G32, 128>(p, s);
    }
    if (scheme == KVQ_INT8_SYM_TOKEN) return launch_append_t<KVQ_INT8_SYM_TOKEN, 64>(p, s);
    if (scheme == KVQ_FP8E4M3_TOKEN) return launch_append_t<KVQ_FP8E4M3_TOKEN, 64>(p, s);
    if (scheme == KVQ_INT4_SYM_G32) return launch_append_t<KVQ_INT4_SYM_G32, 64>(p, s);
    return launch_append_t<KVQ_INT4_ASYM_G32, 64>(p, s);
}

cudaError_t launch_validate(const CacheView& c, const int32_t* block_table,
                            const int32_t* seq_lens, int B, int max_pages, unsigned* err,
                            cudaStream_t s) {
    const int64_t n = (int64_t)B * max_pages;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    validate_kernel<<<(unsigned)blocks, 256, 0, s>>>(c.num_pages, c.page_size, block_table,
                                                     seq_lens, B, max_pages, err);
    return cudaGetLastError();
}

}  // namespace kvq
