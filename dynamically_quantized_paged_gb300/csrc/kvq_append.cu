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
// K-or-V).  A row is spread over head_dim/8 lanes, 16 bytes (8 values) per
// lane, so that a warp loads whole rows with 128-bit loads; K and V of the
// same (token, head) sit in the same warp.  The absmax (or min/max) is a
// warp-shuffle reduction inside the row's lanes.  Every fp32 step is an
// explicitly rounded IEEE operation (__fdiv_rn, __fsub_rn, cvt.rni), so the
// codes do not depend on compiler contraction.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_UNROLL = 4;  // rows per lane group whose loads are issued together

// RNE(fl(x_i / s)) as integers, for |x_i / s| <= 128.  With r = RN(1/s),
// y = RN(x r) lies within 1.5 * 2^-23 * |x / s| (< 2^-15 here) of fl(x / s),
// so unless y is within 2^-14 of a half-integer both round to the same
// integer.  Near one, the quotient is computed exactly; that branch is taken
// by the whole warp or not at all (it is rare), so that the division is not
// evaluated for every element.
template <int N>
__device__ __forceinline__ void rne_quotients(const float* x, float s, float r, int* q) {
    bool slow = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float y = __fmul_rn(x[i], r);
        const float c = rintf(y);
        q[i] = (int)c;
        slow |= !(fabsf(__fsub_rn(y, c)) < 0.5f - 0x1p-14f);
    }
    if (__any_sync(0xffffffffu, slow)) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float y = __fmul_rn(x[i], r);
            if (!(fabsf(__fsub_rn(y, rintf(y))) < 0.5f - 0x1p-14f)) q[i] = __float2int_rn(__fdiv_rn(x[i], s));
        }
    }
}

// fl(x_i / s) where only its E4M3 rounding matters: y = RN(x r) is within 3
// fp32 ulps of fl(x / s); E4M3 rounding (3 mantissa bits) can only differ
// if y is within a few ulps of a midpoint between E4M3 values (fp32 mantissa
// bits 19..0 = 0x80000) or in the E4M3 subnormal range; there the exact
// quotient is used (a warp-uniform branch, as above).
__device__ __forceinline__ bool e4m3_needs_exact(float y) {
    const uint32_t bits = __float_as_uint(y);
    const int e = (int)((bits >> 23) & 0xFFu);
    const int low = (int)(bits & 0xFFFFFu);
    return abs(low - 0x80000) <= 8 || (e < 127 - 6 && y != 0.0f);
}
template <int N>
__device__ __forceinline__ void e4m3_quotients(const float* x, float s, float r, float* y) {
    bool slow = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        y[i] = __fmul_rn(x[i], r);
        slow |= e4m3_needs_exact(y[i]);
    }
    if (__any_sync(0xffffffffu, slow)) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (e4m3_needs_exact(y[i])) y[i] = __fdiv_rn(x[i], s);
    }
}

template <int SCHEME, int D>
__global__ void __launch_bounds__(APPEND_THREADS, 4) append_kernel(AppendParams p) {
    constexpr int LPR = D / 8;     // lanes per row
    constexpr int RPW = 32 / LPR;  // rows per warp
    // a decode launched next may be scheduled now (it waits for this grid to
    // complete before reading anything)
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int li = lane % LPR;
    const int H = p.num_kv_heads;
    const int64_t rows = (int64_t)p.num_tokens * H * 2;
    const int64_t warp_id = ((int64_t)blockIdx.x * APPEND_THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * APPEND_THREADS) >> 5;
    const int64_t stride = nwarps * RPW;

    // the trip count is the same for every lane of the warp (rows past the
    // end are carried as invalid), so the warp collectives below see all lanes
    for (int64_t rb = warp_id * RPW; rb < rows; rb += stride * APPEND_UNROLL) {
        const int64_t r0 = rb + lane / LPR;
        // issue every load of APPEND_UNROLL rows before using any of them
        int64_t slot[APPEND_UNROLL];
        uint4 raw[APPEND_UNROLL];
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {
            const int64_t r = r0 + u * stride;
            slot[u] = -1;
            raw[u] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows) {
                const uint32_t th = (uint32_t)r >> 1;  // token * H + head
                const int64_t t = th / (uint32_t)H;
                const int h = (int)(th - (uint32_t)t * (uint32_t)H);
                const int kv = (int)(r & 1);
                slot[u] = __ldg(p.slot_mapping + t);
                raw[u] = __ldg(reinterpret_cast<const uint4*>((kv ? p.v : p.k) + (t * H + h) * D + li * 8));
            }
        }
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {
            const int64_t r = r0 + u * stride;
            const uint32_t th = (uint32_t)r >> 1;
            const int h = (int)(th % (uint32_t)H);
            const int kv = (int)(r & 1);
            int64_t sl = r < rows ? slot[u] : -1;
            if (sl >= p.num_slots) {
                if (li == 0) flag_error(p.err, ERR_BAD_TABLE);
                sl = -1;
            }
            const bool valid = sl >= 0;
            float x[8];
            {
                const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
                    x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
                }
            }
            // pool row of this (slot, head): [page][head][offset]
            const uint32_t pg = valid ? (uint32_t)sl / (uint32_t)p.page_size : 0u;
            const uint32_t off = valid ? (uint32_t)sl - pg * (uint32_t)p.page_size : 0u;
            const int64_t prow = ((int64_t)pg * H + h) * p.page_size + off;

            if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN || SCHEME == KVQ_FP8E4M3_TOKEN) {
                float a = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
                constexpr float QMAX = SCHEME == KVQ_INT8_SYM_TOKEN ? 127.0f : 448.0f;
                const bool zero_row = (a == 0.0f);
                const float scale = zero_row ? 1.0f : __fdiv_rn(a, QMAX);
                const float rcp = __frcp_rn(scale);
                // (a zero row's x are all +-0: codes 0 with scale 1)
                uint32_t lo = 0, hi = 0;
                if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN) {
                    int q[8];
                    rne_quotients<8>(x, scale, rcp, q);
                    uint32_t b[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) b[i] = (uint32_t)(max(-127, min(127, q[i])) & 0xFF);
                    lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
                    hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
                } else {
                    float y[8];
                    e4m3_quotients<8>(x, scale, rcp, y);
                    uint32_t pr[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pr[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(y[2 * i], y[2 * i + 1]), __NV_SATFINITE,
                                                                    __NV_E4M3);
                    lo = zero_row ? 0u : (pr[0] | (pr[1] << 16));  // a zero row (even of -0) codes +0
                    hi = zero_row ? 0u : (pr[2] | (pr[3] << 16));
                }
                if (valid) {
                    uint8_t* dst = (kv ? p.v_codes : p.k_codes) + prow * D + li * 8;
                    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
                    if (li == 0) static_cast<float*>(kv ? p.v_scales : p.k_scales)[prow] = scale;
                }
            } else if constexpr (SCHEME == KVQ_INT4_SYM_G32) {  // symmetric INT4, groups of 32 channels = 4 lanes
                float a = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
                for (int off = 2; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
                // scale = a / 7 in fp32 (1 for an all-zero group, whose x are
                // +-0 and so round to code 0 as well); |x / scale| <= 7
                const float sc = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 7.0f);
                const float rcp = __frcp_rn(sc);
                int q[8];
                rne_quotients<8>(x, sc, rcp, q);
                uint32_t packed = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) packed |= ((uint32_t)max(-7, min(7, q[i])) & 0xFu) << (4 * i);
                if (valid) {
                    uint8_t* dst = (kv ? p.v_codes : p.k_codes) + prow * (D / 2) + li * 4;
                    *reinterpret_cast<uint32_t*>(dst) = packed;
                    if ((li & 3) == 0) static_cast<float*>(kv ? p.v_scales : p.k_scales)[prow * (D / 32) + li / 4] = sc;
                }
            } else {  // INT4 asymmetric, groups of 32 channels = 4 lanes
                float mn = x[0], mx = x[0];
#pragma unroll
                for (int i = 1; i < 8; ++i) {
                    mn = fminf(mn, x[i]);
                    mx = fmaxf(mx, x[i]);
                }
#pragma unroll
                for (int off = 2; off >= 1; off >>= 1) {
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                }
                const __half zh = __float2half_rd(mn);
                const float zf = __half2float(zh);
                __half sh = __float2half_ru(__fdiv_rn(__fsub_rn(mx, zf), 15.0f));
                if (__half2float(sh) == 0.0f) sh = __float2half(1.0f);
                const float sf = __half2float(sh);
                const float rcp = __frcp_rn(sf);
                float d[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) d[i] = __fsub_rn(x[i], zf);
                int q[8];
                rne_quotients<8>(d, sf, rcp, q);
                uint32_t packed = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) packed |= (uint32_t)max(0, min(15, q[i])) << (4 * i);
                if (valid) {
                    uint8_t* dst = (kv ? p.v_codes : p.k_codes) + prow * (D / 2) + li * 4;
                    *reinterpret_cast<uint32_t*>(dst) = packed;
                    if ((li & 3) == 0) {
                        const int64_t gi = prow * (D / 32) + li / 4;
                        static_cast<__half*>(kv ? p.v_scales : p.k_scales)[gi] = sh;
                        static_cast<__half*>(kv ? p.v_zeros : p.k_zeros)[gi] = zh;
                    }
                }
            }
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

template <int SCHEME, int D>
cudaError_t launch_append_t(const AppendParams& p, cudaStream_t s) {
    // as many CTAs as there are row groups (small appends are latency-bound),
    // at most one wave of 4 resident CTAs per SM (then each lane group loops,
    // APPEND_UNROLL rows at a time)
    constexpr int RPB = (APPEND_THREADS / 32) * (32 / (D / 8));
    const int64_t rows = (int64_t)p.num_tokens * p.num_kv_heads * 2;
    int64_t blocks = (rows + RPB - 1) / RPB;
    const int64_t cap = (int64_t)device_sm_count() * 4;
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
