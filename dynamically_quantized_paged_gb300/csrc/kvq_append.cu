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
// rule itself (absmax or min/max by warp shuffles, explicitly rounded IEEE
// steps) is kvq_quant.cuh's, shared with the decode that appends its step's
// token itself.
#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_STAGES = 4;  // per-warp ring of items: APPEND_STAGES - 1 in flight

// n / d for 0 <= n < 2^31 as (n * mul) >> shift, with mul and shift from
// magic_divisor (below).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint64_t mul, int shift) {
    return (uint32_t)(((uint64_t)n * mul) >> shift);
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
__global__ void __launch_bounds__(APPEND_THREADS, 3) append_kernel(AppendParams p) {
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
        bool valid = sl >= 0;
        const uint32_t t = fast_div((uint32_t)(in_chunk ? pi : 0), p.heads_mul, p.heads_shift);
        int32_t rs = -1;  // per-channel K: the token's residual slot
        if constexpr (SCHEME == KVQ_INT8_KCHAN) {
            if (valid && p.resid_slot) {
                rs = __ldg(p.resid_slot + t);
                if (rs >= p.resid_slots) {  // nothing is written for the token
                    if (li == 0) flag_error(p.err, ERR_BAD_TABLE);
                    valid = false;
                }
            }
        }
        const int h = (int)((uint32_t)(in_chunk ? pi : 0) - t * (uint32_t)H);
        // pool row of this (slot, head): [page][head][offset] in the page's tier
        const uint32_t pg = valid ? fast_div((uint32_t)sl, p.page_mul, p.page_shift) : 0u;
        const uint32_t off = valid ? (uint32_t)sl - pg * (uint32_t)p.page_size : 0u;
        const bool host = pg >= (uint32_t)p.num_pages;
        const uint32_t pi_t = host ? pg - (uint32_t)p.num_pages : pg;
        const int64_t prow = ((int64_t)pi_t * H + h) * p.page_size + off;
        // the per-channel K scheme stores an open page's rows by the INT8 token rule
        constexpr int QS = SCHEME == KVQ_INT8_KCHAN ? KVQ_INT8_SYM_TOKEN : SCHEME;
        const LaneCodes ck = quantize_lane<QS, LPR>(rk);
        const LaneCodes cv = quantize_lane<QS, LPR>(rv);
        if (valid) {  // into the pools of the page's tier
            store_lane<QS, D>(ck, host ? p.hk_codes : p.k_codes, host ? p.hk_scales : p.k_scales,
                              host ? p.hk_zeros : p.k_zeros, prow, li);
            store_lane<QS, D>(cv, host ? p.hv_codes : p.v_codes, host ? p.hv_scales : p.v_scales,
                              host ? p.hv_zeros : p.v_zeros, prow, li);
            if constexpr (SCHEME == KVQ_INT8_KCHAN) {
                if (off == 0) {  // the page's first token opens it: channel factors 1.0
                    const uint4 ones = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
                    uint4* f = reinterpret_cast<uint4*>((host ? p.hk_chan : p.k_chan) +
                                                        ((int64_t)pi_t * H + h) * D + li * 16);
                    f[0] = ones;
                    f[1] = ones;
                }
                if (rs >= 0) {  // the bf16 K row, kept for the page's seal
                    uint4* r = reinterpret_cast<uint4*>(p.k_resid +
                                                        (((int64_t)rs * H + h) * p.page_size + off) * D + li * 16);
                    r[0] = rk[0];
                    r[1] = rk[1];
                }
            }
        }
    }
    cp_async_wait<0>();
}

// Seal of the per-channel K scheme: one CTA per (pair i, KV head h), one
// thread per channel j.  The page rule down each channel of the residual
// slot's rows ("KV Cache Optimization: Strategies for Faster LLM Inference",
// section "KV Cache Quantization: When and How to Compress": per-channel
// scales; the absmax rule of "Dynamic KV Cache Quantization for Fast LLM
// Inference", section "Understanding Dynamic Quantization Techniques"):
// s_j = max_t |x| / 127, S = max_j s_j, factor r_j = fp16 round-up of
// s_j / S, code = round-half-even(x / (r_j S)), every token scale S; each
// step one correctly rounded IEEE operation (the quotients through the token
// rule's reciprocal with its exactness check, which gives the same codes).
template <int D>
__global__ void __launch_bounds__(D) seal_kernel(AppendParams p, const int32_t* pages, const int32_t* rslots) {
    const int i = blockIdx.x, h = blockIdx.y, j = threadIdx.x;
    const int H = p.num_kv_heads, P = p.page_size;
    const int32_t page = pages[i], rs = rslots[i];
    if (page < 0 || (int64_t)page * P >= p.num_slots || rs < 0 || rs >= p.resid_slots) {
        if (h == 0 && j == 0) flag_error(p.err, ERR_BAD_TABLE);
        return;
    }
    const uint16_t* x = p.k_resid + ((int64_t)rs * H + h) * P * D + j;
    // this channel's values, 16 tokens at a time (page_size is a multiple of
    // 16); the last 16 stay in registers for the codes below
    float xs[16];
    float amax = 0.0f;
    for (int t0 = 0; t0 < P; t0 += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) xs[i] = __uint_as_float((uint32_t)x[(int64_t)(t0 + i) * D] << 16);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(xs[i]));
    }
    const float sj = __fdiv_rn(amax, 127.0f);
    __shared__ float red[D / 32];
    float S = sj;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) S = fmaxf(S, __shfl_xor_sync(0xffffffffu, S, o));
    if ((j & 31) == 0) red[j >> 5] = S;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < D / 32; ++w) S = fmaxf(S, red[w]);
    const bool host = page >= p.num_pages;
    const int64_t pg = host ? page - p.num_pages : page;
    const int64_t row0 = (pg * H + h) * P;
    int8_t* codes = reinterpret_cast<int8_t*>(host ? p.hk_codes : p.k_codes) + row0 * D + j;
    float* tok = static_cast<float*>(host ? p.hk_scales : p.k_scales) + row0;
    uint16_t* chan = (host ? p.hk_chan : p.k_chan) + (pg * H + h) * D + j;
    if (S == 0.0f) {  // an all-zero block: the zero-row convention
        for (int t = 0; t < P; ++t) codes[(int64_t)t * D] = 0;
        *chan = 0x3C00;
        for (int t = j; t < P; t += D) tok[t] = 1.0f;
        return;
    }
    const __half r = __float2half_ru(__fdiv_rn(sj, S));
    const float e = __fmul_rn(__half2float(r), S);
    // round-half-even of fl(x / e), 16 tokens at a time (page_size is a
    // multiple of 16; every lane of the warp takes part): the reciprocal with
    // the exactness check of the token rule, since |x / e| <= 127 (1 + 2^-22)
    const float re = approx_rcp(e);
    for (int t0 = 0; t0 < P; t0 += 16) {
        int q[16];
        if (P > 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) xs[i] = __uint_as_float((uint32_t)x[(int64_t)(t0 + i) * D] << 16);
        }
        rne_quotients<16>(xs, e, re, q);
#pragma unroll
        for (int i = 0; i < 16; ++i)  // an all-zero channel (e = 0) has codes 0
            codes[(int64_t)(t0 + i) * D] = (int8_t)(e != 0.0f ? min(max(q[i], -127), 127) : 0);
    }
    *chan = __half_as_ushort(r);
    for (int t = j; t < P; t += D) tok[t] = S;
}

// Batched page copies: CTA-strided over the pairs; every pool of page src[i]
// to page dst[i], 16-byte words, four loads in flight per thread before
// their stores (a host-tier page is read over NVLink-C2C, whose latency the
// loads in flight cover).
__global__ void __launch_bounds__(256) copy_pages_kernel(PageCopyParams p) {
    for (int i = blockIdx.x; i < p.n; i += gridDim.x) {
        const int s = p.src[i], d = p.dst[i];
        if (s < 0 || s >= p.total_pages || d < 0 || d >= p.total_pages || s == d) {
            if (threadIdx.x == 0) flag_error(p.err, ERR_BAD_TABLE);
            continue;
        }
        const int ts = s >= p.num_pages, td = d >= p.num_pages;
        const int64_t is = s - (ts ? p.num_pages : 0), id = d - (td ? p.num_pages : 0);
#pragma unroll 1
        for (int k = 0; k < 7; ++k) {
            const uint8_t* from = p.base[k][ts];
            uint8_t* to = p.base[k][td];
            if (!from || !to) continue;
            const int64_t words = p.bytes[k] / 16;
            const uint4* f = reinterpret_cast<const uint4*>(from + is * p.bytes[k]);
            uint4* t = reinterpret_cast<uint4*>(to + id * p.bytes[k]);
            for (int64_t j0 = threadIdx.x; j0 < words; j0 += 4 * (int64_t)blockDim.x) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t j = j0 + u * (int64_t)blockDim.x;
                    if (j < words) v[u] = f[j];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t j = j0 + u * (int64_t)blockDim.x;
                    if (j < words) t[j] = v[u];
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
    // latency-bound), at most one wave of 3 resident CTAs per SM (then each
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
        // three resident CTAs need the largest shared-memory carveout
        e = cudaFuncSetAttribute(append_kernel<SCHEME, D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    const int64_t pairs = (int64_t)p.num_tokens * p.num_kv_heads;
    const int64_t items = (pairs + C::PPW - 1) / C::PPW;
    int64_t blocks = (items + C::WARPS - 1) / C::WARPS;
    const int64_t cap = (int64_t)device_sm_count() * 3;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    append_kernel<SCHEME, D><<<(unsigned)blocks, APPEND_THREADS, C::SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int scheme, int head_dim, cudaStream_t s) {
    if (scheme == KVQ_INT8_KCHAN)
        return head_dim == 128 ? launch_append_t<KVQ_INT8_KCHAN, 128>(p, s) : launch_append_t<KVQ_INT8_KCHAN, 64>(p, s);
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

cudaError_t launch_seal(const AppendParams& p, int head_dim, const int32_t* pages, const int32_t* rslots, int n,
                        cudaStream_t s) {
    const dim3 grid((unsigned)n, (unsigned)p.num_kv_heads);
    if (head_dim == 128) seal_kernel<128><<<grid, 128, 0, s>>>(p, pages, rslots);
    else seal_kernel<64><<<grid, 64, 0, s>>>(p, pages, rslots);
    return cudaGetLastError();
}

cudaError_t launch_copy_pages(const PageCopyParams& p, cudaStream_t s) {
    int64_t blocks = p.n;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    copy_pages_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// slots[b]: the physical slot of position seq_lens[b] - 1 of sequence b,
// for the two-launch form of the decode that appends its step's token.
__global__ void last_slots_kernel(int total_pages, int page_size, const int32_t* block_table,
                                  const int32_t* seq_lens, int B, int max_pages, int64_t* slots, unsigned* err) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
        const int32_t L = seq_lens[b];
        int64_t sl = -1;
        if (L > 0 && (int64_t)L <= (int64_t)max_pages * page_size) {
            const int32_t pg = block_table[(int64_t)b * max_pages + (L - 1) / page_size];
            if (pg >= 0 && pg < total_pages) sl = (int64_t)pg * page_size + (L - 1) % page_size;
            else flag_error(err, ERR_BAD_TABLE);
        } else if (L != 0) {
            flag_error(err, ERR_BAD_TABLE);
        }
        slots[b] = sl;
    }
}

cudaError_t launch_last_slots(const CacheView& c, const int32_t* block_table, const int32_t* seq_lens, int B,
                              int max_pages, int64_t* slots, unsigned* err, cudaStream_t s) {
    last_slots_kernel<<<(B + 255) / 256, 256, 0, s>>>(c.num_pages + c.host_pages, c.page_size, block_table,
                                                      seq_lens, B, max_pages, slots, err);
    return cudaGetLastError();
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
