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
#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_STAGES = 4;  // per-warp ring of items: APPEND_STAGES - 1 in flight

// n / d for 0 <= n < 2^31 as (n * mul) >> shift, with mul and shift from
// magic_divisor (below).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint64_t mul, int shift) {
    return (uint32_t)(((uint64_t)n * mul) >> shift);
}

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
// RNE(y) for |y| < 2^22), packed four to a word.
template <int N>
__device__ __forceinline__ void rne_codes_s8(const float* x, float s, float r, uint32_t* wd) {
    constexpr float M = 12582912.0f;  // 1.5 * 2^23
    uint32_t t[N];
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float y = __fmul_rn(x[i], r);
        const float tf = __fadd_rn(y, M);
        t[i] = __float_as_uint(tf);
        dmax = fmaxf(dmax, fabsf(__fsub_rn(y, __fsub_rn(tf, M))));
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

// One lane's 16 channels of one row (K or V of a (token, head)), quantized
// and stored.  LPR lanes hold a row; `li` is this lane's index in it.
template <int SCHEME, int D, int LPR>
__device__ __forceinline__ void quantize_store(const AppendParams& p, const uint4 (&raw)[2], int kv, bool valid,
                                               bool host, int64_t prow, int li) {
    // the pools of this row's tier (device, or host for page ids >= num_pages)
    uint8_t* const codes = host ? (kv ? p.hv_codes : p.hk_codes) : (kv ? p.v_codes : p.k_codes);
    void* const scales = host ? (kv ? p.hv_scales : p.hk_scales) : (kv ? p.v_scales : p.k_scales);
    void* const zeros = host ? (kv ? p.hv_zeros : p.hk_zeros) : (kv ? p.v_zeros : p.k_zeros);
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
        uint32_t wd[4];
        if constexpr (SCHEME == KVQ_INT8_SYM_TOKEN) {
            // |x| <= a gives |x / scale| <= 127 (1 + 2^-24) < 127.5: codes in
            // [-127, 127] without clamping; a zero row's x are +-0: codes 0
            rne_codes_s8<16>(x, scale, rcp, wd);
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
            uint8_t* dst = codes + prow * D + li * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            if (li == 0) static_cast<float*>(scales)[prow] = scale;
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
            const float rcp = approx_rcp(sc);
            int q[16];
            rne_quotients<16>(x, sc, rcp, q);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) w |= ((uint32_t)q[8 * h + i] & 0xFu) << (4 * i);
                packed[h] = w;
            }
            if (valid && (li & 1) == 0) static_cast<float*>(scales)[prow * (D / 32) + li / 2] = sc;
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
                packed[h] = w;
            }
            if (valid && (li & 1) == 0) {
                const int64_t gi = prow * (D / 32) + li / 2;
                static_cast<__half*>(scales)[gi] = sh;
                static_cast<__half*>(zeros)[gi] = zh;
            }
        }
        if (valid) {
            uint8_t* dst = codes + prow * (D / 2) + li * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
        }
    }
}

// One lane holds 16 channels of both the K row and the V row of a (token, KV
// head) pair; LPR = D / 16 lanes hold a pair, and a warp's item is PPW =
// 32 / LPR consecutive pairs (their K rows, V rows and slots are contiguous
// runs).  Each warp streams its items (item j of warp w is item w + j * nwarps
// of the launch) through its own ring of APPEND_STAGES shared-memory stages
// with cp.async, keeping APPEND_STAGES - 1 items in flight, so that a chunk of
// many tokens has its whole input in flight from the start.  The slot, page
// and head arithmetic is done once for the two rows of a pair.
template <int D>
struct AppendCfg {
    static constexpr int LPR = D / 16;               // lanes per pair
    static constexpr int PPW = 32 / LPR;             // pairs per item
    static constexpr int ROW = D * 2;                // bytes of one bf16 row
    static constexpr int K_OFF = 0;                  // [PPW][D] bf16
    static constexpr int V_OFF = PPW * ROW;          // [PPW][D] bf16
    static constexpr int S_OFF = 2 * PPW * ROW;      // [PPW] int64 slots
    static constexpr int ITEM = S_OFF + PPW * 8;     // bytes of one stage
    static constexpr int PIECES = PPW * ROW / 16;    // 16-byte pieces of one row run
    static constexpr int WARPS = APPEND_THREADS / 32;
    static constexpr int SMEM = WARPS * APPEND_STAGES * ITEM;
    static_assert(ITEM % 16 == 0 && PIECES % 32 == 0, "whole 16-byte pieces, one set per lane");
};

template <int SCHEME, int D>
__global__ void __launch_bounds__(APPEND_THREADS, 2) append_kernel(AppendParams p) {
    using C = AppendCfg<D>;
    constexpr int LPR = C::LPR;
    constexpr int PPW = C::PPW;
    extern __shared__ __align__(16) uint8_t smem[];
    // a decode launched next may be scheduled now (it waits for this grid to
    // complete before reading anything)
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int li = lane % LPR;
    const int H = p.num_kv_heads;
    const int64_t pairs = (int64_t)p.num_tokens * H;
    const int64_t items = (pairs + PPW - 1) / PPW;
    const int64_t warp_id = (int64_t)blockIdx.x * C::WARPS + warp;
    const int64_t nwarps = (int64_t)gridDim.x * C::WARPS;
    uint8_t* ring = smem + (size_t)warp * APPEND_STAGES * C::ITEM;
    // items of this warp: warp_id, warp_id + nwarps, ...  (the same count for
    // every lane, so the warp collectives below see all lanes)
    const int64_t n_items = warp_id < items ? (items - warp_id + nwarps - 1) / nwarps : 0;

    // issues item j of this warp into its stage and commits one group (empty
    // past the last item); a pair past the end of the chunk is not read
    auto issue = [&](int64_t j) {
        if (j < n_items) {
            uint8_t* stg = ring + (j % APPEND_STAGES) * C::ITEM;
            const int64_t pb = (warp_id + j * nwarps) * PPW;  // first pair of the item
            const uint8_t* ks = reinterpret_cast<const uint8_t*>(p.k + pb * D);
            const uint8_t* vs = reinterpret_cast<const uint8_t*>(p.v + pb * D);
#pragma unroll
            for (int k = 0; k < C::PIECES / 32; ++k) {
                const int i = k * 32 + lane;
                if (pb + (i * 16) / C::ROW < pairs) {
                    cp_async16(stg + C::K_OFF + 16 * i, ks + 16 * i);
                    cp_async16(stg + C::V_OFF + 16 * i, vs + 16 * i);
                }
            }
            if (lane < PPW && pb + lane < pairs) {
                const uint32_t t = fast_div((uint32_t)(pb + lane), p.heads_mul, p.heads_shift);
                cp_async8(stg + C::S_OFF + 8 * lane, p.slot_mapping + t);
            }
        }
        cp_async_commit();
    };

#pragma unroll 1
    for (int j = 0; j < APPEND_STAGES - 1; ++j) issue(j);
#pragma unroll 1
    for (int64_t j = 0; j < n_items; ++j) {
        issue(j + APPEND_STAGES - 1);
        cp_async_wait<APPEND_STAGES - 1>();  // item j has landed (this lane's copies)
        __syncwarp();                        // ... and every lane's
        const uint8_t* stg = ring + (j % APPEND_STAGES) * C::ITEM;
        const int pr = lane / LPR;  // this lane's pair in the item
        const int64_t pi = (warp_id + j * nwarps) * PPW + pr;
        const bool in_chunk = pi < pairs;
        uint4 rk[2], rv[2];
        int64_t sl = -1;
        if (in_chunk) {
            const uint4* kr = reinterpret_cast<const uint4*>(stg + C::K_OFF + pr * C::ROW + li * 32);
            const uint4* vr = reinterpret_cast<const uint4*>(stg + C::V_OFF + pr * C::ROW + li * 32);
            rk[0] = kr[0];
            rk[1] = kr[1];
            rv[0] = vr[0];
            rv[1] = vr[1];
            sl = *reinterpret_cast<const int64_t*>(stg + C::S_OFF + 8 * pr);
        } else {
            rk[0] = rk[1] = rv[0] = rv[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();  // the stage is read: the next issue may refill it
        if (sl >= p.num_slots) {
            if (li == 0) flag_error(p.err, ERR_BAD_TABLE);
            sl = -1;
        }
        const bool valid = sl >= 0;
        const uint32_t t = fast_div((uint32_t)(in_chunk ? pi : 0), p.heads_mul, p.heads_shift);
        const int h = (int)((uint32_t)(in_chunk ? pi : 0) - t * (uint32_t)H);
        // pool row of this (slot, head): [page][head][offset] in the page's tier
        const uint32_t pg = valid ? fast_div((uint32_t)sl, p.page_mul, p.page_shift) : 0u;
        const uint32_t off = valid ? (uint32_t)sl - pg * (uint32_t)p.page_size : 0u;
        const bool host = pg >= (uint32_t)p.num_pages;
        const uint32_t pi_t = host ? pg - (uint32_t)p.num_pages : pg;
        const int64_t prow = ((int64_t)pi_t * H + h) * p.page_size + off;
        quantize_store<SCHEME, D, LPR>(p, rk, 0, valid, host, prow, li);
        quantize_store<SCHEME, D, LPR>(p, rv, 1, valid, host, prow, li);
    }
    cp_async_wait<0>();
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
    // as many CTAs as there are items for their warps (small appends are
    // latency-bound), at most one wave of 2 resident CTAs per SM (then each
    // warp loops over its items)
    using C = AppendCfg<D>;
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(append_kernel<SCHEME, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    const int64_t pairs = (int64_t)p.num_tokens * p.num_kv_heads;
    const int64_t items = (pairs + C::PPW - 1) / C::PPW;
    int64_t blocks = (items + C::WARPS - 1) / C::WARPS;
    const int64_t cap = (int64_t)device_sm_count() * 2;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    append_kernel<SCHEME, D><<<(unsigned)blocks, APPEND_THREADS, C::SMEM, s>>>(p);
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
    validate_kernel<<<(unsigned)blocks, 256, 0, s>>>(c.num_pages + c.host_pages, c.page_size, block_table,
                                                     seq_lens, B, max_pages, err);
    return cudaGetLastError();
}

}  // namespace kvq
