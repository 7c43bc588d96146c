// kvq_internal.h -- launch parameters and launcher entry points shared by the
// host API (kvq_api.cu) and the kernel translation units.  Not public.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

// Bits of the per-device error word (see kvq_last_device_error).
constexpr unsigned ERR_BAD_TABLE = 1u;
constexpr unsigned ERR_TIMEOUT = 2u;

// Tokens per pipeline stage ("unit").  Pages are a multiple of it, so a unit
// never straddles two pages and split boundaries fall on unit boundaries.
constexpr int UNIT = 16;
// Threads of the two-launch form's merge kernel (one CTA per segment).
constexpr int MERGE_THREADS = 128;
constexpr int MAX_SEQS = 4096;     // per decode call (the plan lives in shared memory)
constexpr int MIN_SLICE_UNITS = 8; // smallest per-CTA share of the work, in units (one tile)

struct CacheView {
    int scheme, num_pages, page_size, num_kv_heads, head_dim, group;
    const uint8_t* k_codes;
    const uint8_t* v_codes;
    const void* k_scales;
    const void* v_scales;
    const void* k_zeros;
    const void* v_zeros;
    // host tier: page ids [num_pages, num_pages + host_pages) live in these
    // pools (page-locked host memory the device reads in place)
    int host_pages;
    const uint8_t* hk_codes;
    const uint8_t* hv_codes;
    const void* hk_scales;
    const void* hv_scales;
    const void* hk_zeros;
    const void* hv_zeros;
    // per-channel K scheme: channel factors of the two tiers (fp16 [page][head][D])
    const void* k_chan;
    const void* hk_chan;
};

// The pools that hold page id `page` (the device tier below num_pages, the
// host tier from there on) and the page's index within them.  `page` must
// lie in [0, num_pages + host_pages).
struct PagePools {
    const uint8_t* k_codes;
    const uint8_t* v_codes;
    const uint8_t* k_scales;
    const uint8_t* v_scales;
    const uint8_t* k_zeros;
    const uint8_t* v_zeros;
    const uint8_t* k_chan;
    int index;
};
__host__ __device__ inline PagePools page_pools(const CacheView& c, int page) {
    const bool host = page >= c.num_pages;
    PagePools r;
    r.k_codes = host ? c.hk_codes : c.k_codes;
    r.v_codes = host ? c.hv_codes : c.v_codes;
    r.k_scales = static_cast<const uint8_t*>(host ? c.hk_scales : c.k_scales);
    r.v_scales = static_cast<const uint8_t*>(host ? c.hv_scales : c.v_scales);
    r.k_zeros = static_cast<const uint8_t*>(host ? c.hk_zeros : c.k_zeros);
    r.v_zeros = static_cast<const uint8_t*>(host ? c.hv_zeros : c.v_zeros);
    r.k_chan = static_cast<const uint8_t*>(host ? c.hk_chan : c.k_chan);
    r.index = host ? page - c.num_pages : page;
    return r;
}

struct AppendParams {
    uint8_t* k_codes;
    uint8_t* v_codes;
    void* k_scales;
    void* v_scales;
    void* k_zeros;
    void* v_zeros;
    // host tier (pages num_pages .. num_pages + host_pages - 1)
    uint8_t* hk_codes;
    uint8_t* hv_codes;
    void* hk_scales;
    void* hv_scales;
    void* hk_zeros;
    void* hv_zeros;
    // per-channel K scheme: channel factors of the two tiers (fp16 bits),
    // the residual pool (bf16 [resid_slots][H][page_size][D]) and each
    // token's residual slot (null: none)
    uint16_t* k_chan;
    uint16_t* hk_chan;
    uint16_t* k_resid;
    const int32_t* resid_slot;
    int resid_slots;
    int num_pages;
    const int64_t* slot_mapping;
    const uint16_t* k;  // bf16 bits
    const uint16_t* v;
    int64_t num_slots;  // (num_pages + host_pages) * page_size: both tiers
    int num_tokens, num_kv_heads, page_size;
    unsigned* err;
    // n / num_kv_heads and n / page_size for 0 <= n < 2^31 as
    // (n * mul) >> shift (filled in by launch_append)
    uint64_t heads_mul, page_mul;
    int heads_shift, page_shift;
};

struct DecodeParams {
    CacheView c;
    const uint16_t* q;  // bf16 bits [B][Hq][D]
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;          // [B][Hq][D]: fp32, or bf16 when out_bf16
    float* ws_o;  // [2 * n_ctas][G][D]
    float* ws_m;  // [2 * n_ctas][G]
    float* ws_l;  // [2 * n_ctas][G]
    float* wp_o;  // CUDA-core kernel only: per-warp partials [2 * n_ctas * warps][G][D]
    float* wp_m;  // [2 * n_ctas * warps][G]
    float* wp_l;  // [2 * n_ctas * warps][G]
    int B, Hq, max_pages;
    int n_ctas;
    float q_scale;  // softmax scale * log2(e), folded into q
    unsigned* err;
    int fuse_merge;                     // 1: the last CTA of a split segment merges it in place
    int out_bf16;                       // 1: the output rows are bf16 (round to nearest even), else fp32
    uint32_t gen;                       // call generation tagging the arrival counters
    unsigned long long* seg_ctr;        // [B * Hkv] arrival counters: (gen << 32) | arrivals
    // the step's appended token (CUDA-core kernel): bf16 [B][Hkv][D] key and
    // value of each sequence's last position (seq_lens[b] - 1), quantized by
    // the warp that reads that position and written to the cache by it; null
    // when the call appends nothing
    const uint16_t* k_new;
    const uint16_t* v_new;
};

// The CUDA-core kernel (kvq_alu.cuh) serves GQA ratios up to 4 of the INT8,
// FP8 and asymmetric INT4 schemes, the tensor-core kernel (kvq_tc.cuh) the
// rest; decode_alu_warps gives the former's warps per CTA, 0 for the latter.
constexpr int decode_alu_warps(int scheme, int G) {
    return !(G <= 4 && (scheme == KVQ_INT8_SYM_TOKEN || scheme == KVQ_FP8E4M3_TOKEN ||
                        scheme == KVQ_INT4_ASYM_G32))
               ? 0
               : ((scheme == KVQ_INT8_SYM_TOKEN || scheme == KVQ_INT4_ASYM_G32) ? 16 : 12);
}

// Workspace layout for n_ctas persistent CTAs (two partial slots per CTA):
// partials o [2 n_ctas][G][D], m [2 n_ctas][G], l [2 n_ctas][G] (fp32); the
// published plan: int64 U, int64 S, int32 prefix[B + 1]; then (8-byte
// aligned) one uint64 arrival counter per (sequence, KV head) segment; then,
// for the CUDA-core kernel of `warps` warps per CTA (16-byte aligned), the
// warp partials o [2 n_ctas warps][G][D], m and l [2 n_ctas warps][G].
inline size_t decode_plan_offset(int n_ctas, int G, int D) {
    const size_t slots = 2 * (size_t)n_ctas;
    return slots * G * D * sizeof(float) + 2 * slots * G * sizeof(float);
}
inline size_t decode_counter_offset(int n_ctas, int G, int D, int B) {
    const size_t end_plan = decode_plan_offset(n_ctas, G, D) + 16 + ((size_t)B + 1) * sizeof(int32_t);
    return (end_plan + 7) / 8 * 8;
}
inline size_t decode_warp_partial_offset(int n_ctas, int G, int D, int B, int Hkv) {
    const size_t end = decode_counter_offset(n_ctas, G, D, B) + (size_t)B * Hkv * sizeof(unsigned long long);
    return (end + 15) / 16 * 16;
}
inline size_t decode_workspace_bytes(int n_ctas, int G, int D, int B, int Hkv, int warps) {
    const size_t slots = 2 * (size_t)n_ctas * warps;
    return decode_warp_partial_offset(n_ctas, G, D, B, Hkv) + slots * G * D * sizeof(float) +
           2 * slots * G * sizeof(float);
}

// Batched page copies (kvq_copy_pages): pool k of tier t (0 device, 1 host)
// starts at base[k][t] (null: the scheme has no such pool) and holds bytes[k]
// bytes per page (a multiple of 16); page id >= num_pages is host-tier.
struct PageCopyParams {
    uint8_t* base[7][2];
    int64_t bytes[7];
    int num_pages, total_pages;
    const int32_t* src;
    const int32_t* dst;
    int n;
    unsigned* err;
};
cudaError_t launch_copy_pages(const PageCopyParams& p, cudaStream_t s);

cudaError_t launch_append(const AppendParams& p, int scheme, int head_dim, cudaStream_t s);
// Per-channel K: seals pages[i] from residual slot rslots[i], i < n.
cudaError_t launch_seal(const AppendParams& p, int head_dim, const int32_t* pages, const int32_t* rslots, int n,
                        cudaStream_t s);
// slots[b] = the physical slot of position seq_lens[b] - 1 of sequence b (from
// its block-table row), -1 for an empty sequence or a page id outside the
// pool (flagged)
cudaError_t launch_last_slots(const CacheView& c, const int32_t* block_table, const int32_t* seq_lens, int B,
                              int max_pages, int64_t* slots, unsigned* err, cudaStream_t s);
cudaError_t launch_decode_partial(const DecodeParams& p, int G, cudaStream_t s);
cudaError_t launch_decode_merge(const DecodeParams& p, int G, cudaStream_t s);
// Resident decode CTAs per SM for this configuration (0 if the query fails).
int decode_ctas_per_sm(int scheme, int head_dim, int G, int B);
cudaError_t launch_validate(const CacheView& c, const int32_t* block_table,
                            const int32_t* seq_lens, int B, int max_pages, unsigned* err,
                            cudaStream_t s);

// Byte offset and length, inside a decode workspace for this problem, of the
// per-segment arrival counters (host only; kvq_api.cu).
kvq_status decode_counter_region(const kvq_cache* cache, int B, int Hq, size_t* offset, size_t* bytes);

// Per-device error word (device address) and SM count.
unsigned* device_error_word();
int device_sm_count();

}  // namespace kvq
