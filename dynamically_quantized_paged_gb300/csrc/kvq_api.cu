// kvq_api.cu -- the C ABI declared in include/kvq.h: argument checks on the
// host, dispatch to the kernels, the per-device error word, and the host page
// allocator.  Nothing here allocates device memory.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <chrono>
#include <mutex>
#include <new>
#include <vector>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

constexpr int MAX_DEVICES = 64;

// Per-device error word written by the kernels (atomicOr of kvq::ERR_* bits).
__device__ unsigned g_error_word;

std::mutex g_mu;
unsigned* g_err_ptr[MAX_DEVICES];
int g_sm_count[MAX_DEVICES];

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1;
    return dev;
}

kvq_status check_cache(const kvq_cache* c) {
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (c->scheme < KVQ_INT8_SYM_TOKEN || c->scheme > KVQ_INT8_KCHAN) return KVQ_ERR_INVALID_ARG;
    if (c->num_pages < 1 || c->page_size < 1 || c->num_kv_heads < 1 || c->head_dim < 1)
        return KVQ_ERR_INVALID_ARG;
    if (c->page_size % kvq::UNIT != 0) return KVQ_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if ((c->scheme == KVQ_INT4_ASYM_G32 || c->scheme == KVQ_INT4_SYM_G32) && c->group != 32)
        return KVQ_ERR_UNSUPPORTED;
    const void* need[4] = {c->k_codes, c->v_codes, c->k_scales, c->v_scales};
    for (const void* p : need)
        if (!p || !aligned(p, 16)) return KVQ_ERR_INVALID_ARG;
    if (c->scheme == KVQ_INT4_ASYM_G32) {
        if (!c->k_zeros || !c->v_zeros || !aligned(c->k_zeros, 16) || !aligned(c->v_zeros, 16))
            return KVQ_ERR_INVALID_ARG;
    }
    if (c->scheme == KVQ_INT8_KCHAN) {  // channel factors; the residual pool when it has slots
        if (!c->k_chan || !aligned(c->k_chan, 16) || c->resid_slots < 0) return KVQ_ERR_INVALID_ARG;
        if (c->resid_slots > 0 && (!c->k_resid || !aligned(c->k_resid, 16))) return KVQ_ERR_INVALID_ARG;
        if (c->host_pages > 0 && (!c->host_k_chan || !aligned(c->host_k_chan, 16))) return KVQ_ERR_INVALID_ARG;
    }
    if (c->host_pages < 0) return KVQ_ERR_INVALID_ARG;
    if (c->host_pages > 0) {  // the host tier's pools, as the device tier's
        const void* hneed[4] = {c->host_k_codes, c->host_v_codes, c->host_k_scales, c->host_v_scales};
        for (const void* p : hneed)
            if (!p || !aligned(p, 16)) return KVQ_ERR_INVALID_ARG;
        if (c->scheme == KVQ_INT4_ASYM_G32 && (!c->host_k_zeros || !c->host_v_zeros ||
                                               !aligned(c->host_k_zeros, 16) || !aligned(c->host_v_zeros, 16)))
            return KVQ_ERR_INVALID_ARG;
    }
    // the pools must be addressable with 64-bit row arithmetic and int32 page
    // ids (both tiers)
    const int64_t pages = (int64_t)c->num_pages + c->host_pages;
    if (pages > INT32_MAX) return KVQ_ERR_INVALID_ARG;
    const int64_t rows = pages * c->num_kv_heads * c->page_size;
    if (rows <= 0 || rows > ((int64_t)1 << 40)) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

kvq::CacheView view_of(const kvq_cache* c) {
    kvq::CacheView v;
    v.scheme = c->scheme;
    v.num_pages = c->num_pages;
    v.page_size = c->page_size;
    v.num_kv_heads = c->num_kv_heads;
    v.head_dim = c->head_dim;
    v.group = c->group;
    v.k_codes = static_cast<const uint8_t*>(c->k_codes);
    v.v_codes = static_cast<const uint8_t*>(c->v_codes);
    v.k_scales = c->k_scales;
    v.v_scales = c->v_scales;
    v.k_zeros = c->k_zeros;
    v.v_zeros = c->v_zeros;
    const bool ht = c->host_pages > 0;
    v.host_pages = ht ? c->host_pages : 0;
    v.hk_codes = ht ? static_cast<const uint8_t*>(c->host_k_codes) : nullptr;
    v.hv_codes = ht ? static_cast<const uint8_t*>(c->host_v_codes) : nullptr;
    v.hk_scales = ht ? c->host_k_scales : nullptr;
    v.hv_scales = ht ? c->host_v_scales : nullptr;
    v.hk_zeros = ht ? c->host_k_zeros : nullptr;
    v.hv_zeros = ht ? c->host_v_zeros : nullptr;
    const bool kc = c->scheme == KVQ_INT8_KCHAN;
    v.k_chan = kc ? c->k_chan : nullptr;
    v.hk_chan = kc && ht ? c->host_k_chan : nullptr;
    return v;
}

int gqa_ratio(const kvq_cache* c, int32_t Hq) {
    if (Hq < 1 || Hq % c->num_kv_heads != 0) return -1;
    const int G = Hq / c->num_kv_heads;
    return (G == 1 || G == 2 || G == 4 || G == 8) ? G : 0;
}

// Generation tag of a decode call: the fused merge counts arrivals per
// segment in workspace words tagged with it, so the workspace needs no
// zeroing.  Starts from a clock-derived odd value and never repeats
// within 2^31 calls of one process.
uint32_t next_generation() {
    static std::atomic<uint32_t> g{0};
    static std::atomic<bool> seeded{false};
    if (!seeded.exchange(true)) {
        const uint32_t seed = (uint32_t)std::chrono::steady_clock::now().time_since_epoch().count();
        g.store(seed | 1u);
    }
    uint32_t v = g.fetch_add(2);
    return v ? v : g.fetch_add(2);
}

// The persistent decode grid: resident CTAs per SM (occupancy of this kernel
// configuration at this batch size) times the SM count.
int n_ctas_for(const kvq_cache* c, int G, int B) {
    return kvq::device_sm_count() * kvq::decode_ctas_per_sm(c->scheme, c->head_dim, G, B);
}

// Shared argument checks of the three decode entry points; fills p.
kvq_status prepare_decode(const kvq_cache* cache, const void* q, const int32_t* block_table,
                          const int32_t* seq_lens, void* out, int32_t B, int32_t Hq,
                          int32_t max_pages, float softmax_scale, void* workspace,
                          size_t workspace_bytes, kvq::DecodeParams& p, int& G) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (B < 0 || B > kvq::MAX_SEQS || max_pages < 1) return KVQ_ERR_INVALID_ARG;
    G = gqa_ratio(cache, Hq);
    if (G < 0) return KVQ_ERR_INVALID_ARG;
    if (G == 0) return KVQ_ERR_UNSUPPORTED;
    if (B == 0) return KVQ_OK;
    if (!q || !block_table || !seq_lens || !out || !workspace) return KVQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return KVQ_ERR_INVALID_ARG;
    // all per-head unit counts must fit int32 (the plan's prefix sums)
    const int64_t units_per_seq = ((int64_t)max_pages * cache->page_size + kvq::UNIT - 1) / kvq::UNIT;
    if (units_per_seq * B * cache->num_kv_heads >= ((int64_t)1 << 31)) return KVQ_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return KVQ_ERR_CUDA;
    const int n_ctas = n_ctas_for(cache, G, B);
    if (n_ctas <= 0) return KVQ_ERR_CUDA;
    const int warps = kvq::decode_alu_warps(cache->scheme, G);
    const size_t need = kvq::decode_workspace_bytes(n_ctas, G, cache->head_dim, B, cache->num_kv_heads, warps);
    if (workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    unsigned* err = kvq::device_error_word();
    if (!err) return KVQ_ERR_CUDA;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)cache->head_dim);
    p.c = view_of(cache);
    p.q = static_cast<const uint16_t*>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_m = p.ws_o + (size_t)2 * n_ctas * G * cache->head_dim;
    p.ws_l = p.ws_m + (size_t)2 * n_ctas * G;
    if (warps > 0) {
        p.wp_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          kvq::decode_warp_partial_offset(n_ctas, G, cache->head_dim, B,
                                                                          cache->num_kv_heads));
        p.wp_m = p.wp_o + (size_t)2 * n_ctas * warps * G * cache->head_dim;
        p.wp_l = p.wp_m + (size_t)2 * n_ctas * warps * G;
    } else {
        p.wp_o = p.wp_m = p.wp_l = nullptr;
    }
    p.B = B;
    p.Hq = Hq;
    p.max_pages = max_pages;
    p.n_ctas = n_ctas;
    p.q_scale = scale * 1.4426950408889634f;  // log2(e): the kernel works in base 2
    p.err = err;
    p.fuse_merge = 0;
    p.out_bf16 = 0;
    p.gen = next_generation();
    p.seg_ctr = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) +
                                                      kvq::decode_counter_offset(n_ctas, G, cache->head_dim, B));
    p.k_new = p.v_new = nullptr;
    return KVQ_OK;
}

}  // namespace

namespace kvq {

kvq_status decode_counter_region(const kvq_cache* cache, int B, int Hq, size_t* offset, size_t* bytes) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    const int G = gqa_ratio(cache, Hq);
    if (G < 0) return KVQ_ERR_INVALID_ARG;
    if (G == 0) return KVQ_ERR_UNSUPPORTED;
    const int n_ctas = n_ctas_for(cache, G, B);
    if (n_ctas <= 0) return KVQ_ERR_CUDA;
    *offset = decode_counter_offset(n_ctas, G, cache->head_dim, B);
    *bytes = (size_t)B * cache->num_kv_heads * sizeof(unsigned long long);
    return KVQ_OK;
}

unsigned* device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(ptr);
    }
    return g_err_ptr[dev];
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace kvq

struct kvq_allocator {
    int32_t num_pages;
    std::vector<int32_t> stack;  // free pages; allocation pops from the back
    std::vector<int32_t> refs;   // references per page (0: free)
};

namespace {

// Occurrences of each page id among pages[0..n) into cnt (num_pages entries),
// after checking that every id is inside the pool and held (refs > 0).
bool count_held(const kvq_allocator* a, int32_t n, const int32_t* pages, std::vector<int32_t>& cnt) {
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = pages[i];
        if (p < 0 || p >= a->num_pages || a->refs[p] <= 0) return false;
    }
    try {
        cnt.assign(a->num_pages, 0);
    } catch (...) {
        return false;
    }
    for (int32_t i = 0; i < n; ++i) ++cnt[pages[i]];
    return true;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_SCHEME_MISMATCH: return "scheme does not match the cache";
        case KVQ_ERR_OUT_OF_PAGES: return "out of pages";
        case KVQ_ERR_BAD_TABLE: return "page, slot or sequence length outside the pool";
        case KVQ_ERR_CUDA: return "CUDA error";
        case KVQ_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case KVQ_ERR_UNSUPPORTED: return "unsupported shape";
        case KVQ_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

kvq_status kvq_cache_bytes(int32_t scheme, int32_t num_pages, int32_t page_size,
                           int32_t num_kv_heads, int32_t head_dim, size_t* code_bytes,
                           size_t* scale_bytes, size_t* zero_bytes) {
    if (scheme < KVQ_INT8_SYM_TOKEN || scheme > KVQ_INT8_KCHAN) return KVQ_ERR_INVALID_ARG;
    if (num_pages < 1 || page_size < 1 || num_kv_heads < 1 || head_dim < 1) return KVQ_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    const size_t rows = (size_t)num_pages * num_kv_heads * page_size;
    const bool int4 = scheme == KVQ_INT4_ASYM_G32, int4s = scheme == KVQ_INT4_SYM_G32;
    if (code_bytes) *code_bytes = rows * (int4 || int4s ? head_dim / 2 : head_dim);
    if (scale_bytes) *scale_bytes = rows * (int4 ? (head_dim / 32) * 2 : int4s ? (head_dim / 32) * 4 : 4);
    if (zero_bytes) *zero_bytes = int4 ? rows * (head_dim / 32) * 2 : 0;
    return KVQ_OK;
}

kvq_status kvq_kchan_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
                           int32_t resid_slots, size_t* chan_bytes, size_t* resid_bytes) {
    if (num_pages < 1 || page_size < 1 || num_kv_heads < 1 || resid_slots < 0) return KVQ_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if (chan_bytes) *chan_bytes = (size_t)num_pages * num_kv_heads * head_dim * 2;
    if (resid_bytes) *resid_bytes = (size_t)resid_slots * num_kv_heads * page_size * head_dim * 2;
    return KVQ_OK;
}

// The append kernel's arguments for num_tokens rows of k, v into the slots
// slot_mapping of the cache (both tiers).
static kvq::AppendParams append_params(const kvq_cache* cache, const int64_t* slot_mapping, const void* k, const void* v,
                                int32_t num_tokens, unsigned* err) {
    kvq::AppendParams p;
    p.k_codes = static_cast<uint8_t*>(cache->k_codes);
    p.v_codes = static_cast<uint8_t*>(cache->v_codes);
    p.k_scales = cache->k_scales;
    p.v_scales = cache->v_scales;
    p.k_zeros = cache->k_zeros;
    p.v_zeros = cache->v_zeros;
    p.slot_mapping = slot_mapping;
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.num_slots = ((int64_t)cache->num_pages + cache->host_pages) * cache->page_size;
    p.num_pages = cache->num_pages;
    const bool ht = cache->host_pages > 0;
    p.hk_codes = ht ? static_cast<uint8_t*>(cache->host_k_codes) : nullptr;
    p.hv_codes = ht ? static_cast<uint8_t*>(cache->host_v_codes) : nullptr;
    p.hk_scales = ht ? cache->host_k_scales : nullptr;
    p.hv_scales = ht ? cache->host_v_scales : nullptr;
    p.hk_zeros = ht ? cache->host_k_zeros : nullptr;
    p.hv_zeros = ht ? cache->host_v_zeros : nullptr;
    const bool kc = cache->scheme == KVQ_INT8_KCHAN;
    p.k_chan = kc ? static_cast<uint16_t*>(cache->k_chan) : nullptr;
    p.hk_chan = kc && ht ? static_cast<uint16_t*>(cache->host_k_chan) : nullptr;
    p.k_resid = kc ? static_cast<uint16_t*>(cache->k_resid) : nullptr;
    p.resid_slots = kc ? cache->resid_slots : 0;
    p.resid_slot = nullptr;
    p.num_tokens = num_tokens;
    p.num_kv_heads = cache->num_kv_heads;
    p.page_size = cache->page_size;
    p.err = err;
    return p;
}

// kvq_append and kvq_append_kchan (resid_slot: per-channel K only, may be null)
static kvq_status append_impl(const kvq_cache* cache, const int32_t* block_table, int32_t num_seqs,
                              int32_t max_pages_per_seq, const int64_t* slot_mapping, const int32_t* resid_slot,
                              const void* k, const void* v, int32_t num_tokens, int32_t scheme,
                              kvq_stream_t stream) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (scheme != cache->scheme) return KVQ_ERR_SCHEME_MISMATCH;
    if (resid_slot && (!aligned(resid_slot, 4) || cache->resid_slots < 1)) return KVQ_ERR_INVALID_ARG;
    if (num_tokens < 0) return KVQ_ERR_INVALID_ARG;
    // slots and rows are indexed in 32 bits on the device
    if (((int64_t)cache->num_pages + cache->host_pages) * cache->page_size >= ((int64_t)1 << 31) ||
        (int64_t)num_tokens * cache->num_kv_heads * 2 >= ((int64_t)1 << 31))
        return KVQ_ERR_INVALID_ARG;
    if (block_table && (num_seqs < 0 || max_pages_per_seq < 1 || !aligned(block_table, 4)))
        return KVQ_ERR_INVALID_ARG;
    if (num_tokens > 0) {
        if (!slot_mapping || !k || !v || !aligned(slot_mapping, 8) || !aligned(k, 16) ||
            !aligned(v, 16))
            return KVQ_ERR_INVALID_ARG;
    }
    if (num_tokens == 0 && !(block_table && num_seqs > 0)) return KVQ_OK;
    unsigned* err = kvq::device_error_word();
    if (!err) return KVQ_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (block_table && num_seqs > 0) {
        if (kvq::launch_validate(view_of(cache), block_table, nullptr, num_seqs, max_pages_per_seq,
                                 err, s) != cudaSuccess)
            return KVQ_ERR_CUDA;
    }
    if (num_tokens == 0) return KVQ_OK;
    kvq::AppendParams p = append_params(cache, slot_mapping, k, v, num_tokens, err);
    p.resid_slot = resid_slot;
    if (kvq::launch_append(p, cache->scheme, cache->head_dim, s) != cudaSuccess) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_append(const kvq_cache* cache, const int32_t* block_table, int32_t num_seqs,
                      int32_t max_pages_per_seq, const int64_t* slot_mapping, const void* k,
                      const void* v, int32_t num_tokens, int32_t scheme, kvq_stream_t stream) {
    return append_impl(cache, block_table, num_seqs, max_pages_per_seq, slot_mapping, nullptr, k, v, num_tokens,
                       scheme, stream);
}

kvq_status kvq_append_kchan(const kvq_cache* cache, const int32_t* block_table, int32_t num_seqs,
                            int32_t max_pages_per_seq, const int64_t* slot_mapping, const int32_t* resid_slot,
                            const void* k, const void* v, int32_t num_tokens, kvq_stream_t stream) {
    return append_impl(cache, block_table, num_seqs, max_pages_per_seq, slot_mapping, resid_slot, k, v, num_tokens,
                       KVQ_INT8_KCHAN, stream);
}

kvq_status kvq_seal_pages(const kvq_cache* cache, const int32_t* pages, const int32_t* resid_slots, int32_t n,
                          kvq_stream_t stream) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (cache->scheme != KVQ_INT8_KCHAN) return KVQ_ERR_SCHEME_MISMATCH;
    if (n < 0 || cache->resid_slots < 1 || !cache->k_resid) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;
    if (!pages || !resid_slots || !aligned(pages, 4) || !aligned(resid_slots, 4)) return KVQ_ERR_INVALID_ARG;
    if (((int64_t)cache->num_pages + cache->host_pages) * cache->page_size >= ((int64_t)1 << 31))
        return KVQ_ERR_INVALID_ARG;
    unsigned* err = kvq::device_error_word();
    if (!err) return KVQ_ERR_CUDA;
    const kvq::AppendParams p = append_params(cache, nullptr, nullptr, nullptr, 0, err);
    if (kvq::launch_seal(p, cache->head_dim, pages, resid_slots, n, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_pages_per_seq,
                                      size_t* bytes) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (!bytes || num_seqs < 0 || num_seqs > kvq::MAX_SEQS || max_pages_per_seq < 1)
        return KVQ_ERR_INVALID_ARG;
    const int G = gqa_ratio(cache, num_q_heads);
    if (G < 0) return KVQ_ERR_INVALID_ARG;
    if (G == 0) return KVQ_ERR_UNSUPPORTED;
    const int n_ctas = n_ctas_for(cache, G, num_seqs);
    if (n_ctas <= 0) return KVQ_ERR_CUDA;
    *bytes = kvq::decode_workspace_bytes(n_ctas, G, cache->head_dim, num_seqs, cache->num_kv_heads,
                                         kvq::decode_alu_warps(cache->scheme, G));
    return KVQ_OK;
}

kvq_status kvq_decode_partial(const kvq_cache* cache, const void* q, const int32_t* block_table,
                              const int32_t* seq_lens, float* out, int32_t num_seqs,
                              int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                              void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
    kvq::DecodeParams p;
    int G = 0;
    kvq_status st = prepare_decode(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads,
                                   max_pages_per_seq, softmax_scale, workspace, workspace_bytes, p, G);
    if (st != KVQ_OK || num_seqs == 0) return st;
    if (kvq::launch_decode_partial(p, G, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_decode_merge(const kvq_cache* cache, const void* q, const int32_t* block_table,
                            const int32_t* seq_lens, float* out, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                            void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
    kvq::DecodeParams p;
    int G = 0;
    kvq_status st = prepare_decode(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads,
                                   max_pages_per_seq, softmax_scale, workspace, workspace_bytes, p, G);
    if (st != KVQ_OK || num_seqs == 0) return st;
    if (kvq::launch_decode_merge(p, G, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_decode_attn(const kvq_cache* cache, const void* q, const int32_t* block_table,
                           const int32_t* seq_lens, float* out, int32_t num_seqs,
                           int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                           void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
    kvq::DecodeParams p;
    int G = 0;
    kvq_status st = prepare_decode(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads,
                                   max_pages_per_seq, softmax_scale, workspace, workspace_bytes, p, G);
    if (st != KVQ_OK || num_seqs == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    p.fuse_merge = 1;  // one launch: splits are merged by the CTA that finishes them last
    if (kvq::launch_decode_partial(p, G, s) != cudaSuccess) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_decode_attn_out(const kvq_cache* cache, const void* q, const int32_t* block_table,
                               const int32_t* seq_lens, void* out, int32_t out_dtype, int32_t num_seqs,
                               int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                               void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
    if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return KVQ_ERR_INVALID_ARG;
    kvq::DecodeParams p;
    int G = 0;
    kvq_status st = prepare_decode(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads,
                                   max_pages_per_seq, softmax_scale, workspace, workspace_bytes, p, G);
    if (st != KVQ_OK || num_seqs == 0) return st;
    p.fuse_merge = 1;
    p.out_bf16 = out_dtype == KVQ_OUT_BF16;
    if (kvq::launch_decode_partial(p, G, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_decode_attn_append(const kvq_cache* cache, const void* k_new, const void* v_new, const void* q,
                                  const int32_t* block_table, const int32_t* seq_lens, void* out,
                                  int32_t out_dtype, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_pages_per_seq, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, kvq_stream_t stream) {
    if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return KVQ_ERR_INVALID_ARG;
    if (cache && cache->scheme == KVQ_INT8_KCHAN) return KVQ_ERR_UNSUPPORTED;  // its append takes residual slots
    kvq::DecodeParams p;
    int G = 0;
    kvq_status st = prepare_decode(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads,
                                   max_pages_per_seq, softmax_scale, workspace, workspace_bytes, p, G);
    if (st != KVQ_OK || num_seqs == 0) return st;
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return KVQ_ERR_INVALID_ARG;
    if (((int64_t)cache->num_pages + cache->host_pages) * cache->page_size >= ((int64_t)1 << 31))
        return KVQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    p.fuse_merge = 1;
    p.out_bf16 = out_dtype == KVQ_OUT_BF16;
    if (kvq::decode_alu_warps(cache->scheme, G) > 0) {
        // one launch: the warp that reads a sequence's last position quantizes
        // its new token there and writes it to the cache
        p.k_new = static_cast<const uint16_t*>(k_new);
        p.v_new = static_cast<const uint16_t*>(v_new);
        if (kvq::launch_decode_partial(p, G, s) != cudaSuccess) return KVQ_ERR_CUDA;
        return KVQ_OK;
    }
    // the tensor-core kernel: the append kernel first (slots from the tables,
    // kept in the partials area of the workspace, which the decode writes only
    // after the append has completed), then the decode
    int64_t* slots = reinterpret_cast<int64_t*>(p.ws_o);
    if (kvq::launch_last_slots(p.c, block_table, seq_lens, num_seqs, max_pages_per_seq, slots, p.err, s) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    const kvq::AppendParams ap = append_params(cache, slots, k_new, v_new, num_seqs, p.err);
    if (kvq::launch_append(ap, cache->scheme, cache->head_dim, s) != cudaSuccess) return KVQ_ERR_CUDA;
    if (kvq::launch_decode_partial(p, G, s) != cudaSuccess) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_validate_tables(const kvq_cache* cache, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t num_seqs,
                               int32_t max_pages_per_seq, kvq_stream_t stream) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (num_seqs < 0 || max_pages_per_seq < 1) return KVQ_ERR_INVALID_ARG;
    if (num_seqs == 0) return KVQ_OK;
    if (!block_table || !seq_lens || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return KVQ_ERR_INVALID_ARG;
    unsigned* err = kvq::device_error_word();
    if (!err) return KVQ_ERR_CUDA;
    if (kvq::launch_validate(view_of(cache), block_table, seq_lens, num_seqs, max_pages_per_seq, err,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_copy_page(const kvq_cache* cache, int32_t src, int32_t dst, kvq_stream_t stream) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    const int64_t total = (int64_t)cache->num_pages + cache->host_pages;
    if (src < 0 || src >= total || dst < 0 || dst >= total || src == dst) return KVQ_ERR_INVALID_ARG;
    if (current_device() < 0) return KVQ_ERR_CUDA;
    // every pool is page-major: a page's rows ([Hkv][page_size], any interleave
    // inside) are one contiguous block of the same size in each
    const size_t rows = (size_t)cache->num_kv_heads * cache->page_size;
    const bool int4 = cache->scheme == KVQ_INT4_ASYM_G32, int4s = cache->scheme == KVQ_INT4_SYM_G32;
    const size_t code_b = rows * (int4 || int4s ? cache->head_dim / 2 : cache->head_dim);
    const size_t meta_b = rows * (int4 ? (cache->head_dim / 32) * 2 : int4s ? (cache->head_dim / 32) * 4 : 4);
    // pool bases of each tier: device, host
    struct Pool { void* base[2]; size_t bytes; } pools[6] = {
        {{cache->k_codes, cache->host_k_codes}, code_b},
        {{cache->v_codes, cache->host_v_codes}, code_b},
        {{cache->k_scales, cache->host_k_scales}, meta_b},
        {{cache->v_scales, cache->host_v_scales}, meta_b},
        {{int4 ? cache->k_zeros : nullptr, int4 ? cache->host_k_zeros : nullptr}, meta_b},
        {{int4 ? cache->v_zeros : nullptr, int4 ? cache->host_v_zeros : nullptr}, meta_b}};
    const bool kc = cache->scheme == KVQ_INT8_KCHAN;  // the channel factors: [Hkv][head_dim] fp16 per page
    const Pool chan = {{kc ? cache->k_chan : nullptr, kc ? cache->host_k_chan : nullptr},
                       (size_t)cache->num_kv_heads * cache->head_dim * 2};
    const int ts = src >= cache->num_pages, td = dst >= cache->num_pages;
    const size_t is = (size_t)(src - (ts ? cache->num_pages : 0)), id = (size_t)(dst - (td ? cache->num_pages : 0));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int i = 0; i < 7; ++i) {
        const Pool& pl = i < 6 ? pools[i] : chan;
        if (!pl.base[0]) continue;
        const uint8_t* from = static_cast<const uint8_t*>(pl.base[ts]) + is * pl.bytes;
        uint8_t* to = static_cast<uint8_t*>(pl.base[td]) + id * pl.bytes;
        // the host tier is page-locked memory the device addresses (unified
        // addressing): the runtime infers each copy's direction
        if (cudaMemcpyAsync(to, from, pl.bytes, cudaMemcpyDefault, s) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

kvq_status kvq_copy_pages(const kvq_cache* cache, const int32_t* src, const int32_t* dst, int32_t n,
                          kvq_stream_t stream) {
    kvq_status st = check_cache(cache);
    if (st != KVQ_OK) return st;
    if (n < 0) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;
    if (!src || !dst || !aligned(src, 4) || !aligned(dst, 4)) return KVQ_ERR_INVALID_ARG;
    unsigned* err = kvq::device_error_word();
    if (!err) return KVQ_ERR_CUDA;
    // the same per-page pool sizes as kvq_copy_page
    const int64_t rows = (int64_t)cache->num_kv_heads * cache->page_size;
    const bool int4 = cache->scheme == KVQ_INT4_ASYM_G32, int4s = cache->scheme == KVQ_INT4_SYM_G32;
    const bool kc = cache->scheme == KVQ_INT8_KCHAN, ht = cache->host_pages > 0;
    const int64_t code_b = rows * (int4 || int4s ? cache->head_dim / 2 : cache->head_dim);
    const int64_t meta_b = rows * (int4 ? (cache->head_dim / 32) * 2 : int4s ? (cache->head_dim / 32) * 4 : 4);
    kvq::PageCopyParams p;
    void* const dev_tier[7] = {cache->k_codes, cache->v_codes, cache->k_scales, cache->v_scales,
                               int4 ? cache->k_zeros : nullptr, int4 ? cache->v_zeros : nullptr,
                               kc ? cache->k_chan : nullptr};
    void* const host_tier[7] = {cache->host_k_codes, cache->host_v_codes, cache->host_k_scales,
                                cache->host_v_scales, int4 ? cache->host_k_zeros : nullptr,
                                int4 ? cache->host_v_zeros : nullptr, kc ? cache->host_k_chan : nullptr};
    const int64_t bytes[7] = {code_b, code_b, meta_b, meta_b, meta_b, meta_b,
                              (int64_t)cache->num_kv_heads * cache->head_dim * 2};
    for (int k = 0; k < 7; ++k) {
        p.base[k][0] = static_cast<uint8_t*>(dev_tier[k]);
        // with no host tier every id is a device page: the host column is never chosen
        p.base[k][1] = ht ? static_cast<uint8_t*>(host_tier[k]) : static_cast<uint8_t*>(dev_tier[k]);
        p.bytes[k] = bytes[k];
    }
    p.num_pages = cache->num_pages;
    p.total_pages = cache->num_pages + cache->host_pages;
    p.src = src;
    p.dst = dst;
    p.n = n;
    p.err = err;
    if (kvq::launch_copy_pages(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

kvq_status kvq_last_device_error(kvq_stream_t stream) {
    if (current_device() < 0) return KVQ_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof v) != cudaSuccess) return KVQ_ERR_CUDA;
    const unsigned zero = 0;
    if (v && cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero) != cudaSuccess) return KVQ_ERR_CUDA;
    if (v & kvq::ERR_TIMEOUT) return KVQ_ERR_DEVICE_TIMEOUT;
    if (v & kvq::ERR_BAD_TABLE) return KVQ_ERR_BAD_TABLE;
    return KVQ_OK;
}

// ---- host page allocator -------------------------------------------------------

static uint64_t splitmix64(uint64_t* state) {
    // SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): golden-ratio increment,
    // then two xor-shift-multiply mixing rounds and a final xor-shift.
    uint64_t z = (*state += 0x9e3779b97f4a7c15ULL);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

kvq_allocator* kvq_allocator_create(int32_t num_pages, uint64_t seed) {
    if (num_pages < 1) return nullptr;
    kvq_allocator* a = new (std::nothrow) kvq_allocator;
    if (!a) return nullptr;
    try {
        a->num_pages = num_pages;
        a->stack.resize(num_pages);
        a->refs.assign(num_pages, 0);
    } catch (...) {
        delete a;
        return nullptr;
    }
    for (int32_t i = 0; i < num_pages; ++i) a->stack[i] = i;
    uint64_t st = seed;
    for (int32_t i = num_pages - 1; i >= 1; --i) {  // Fisher-Yates, Durstenfeld's order
        const uint64_t j = splitmix64(&st) % (uint64_t)(i + 1);
        const int32_t t = a->stack[i];
        a->stack[i] = a->stack[j];
        a->stack[j] = t;
    }
    return a;
}

void kvq_allocator_destroy(kvq_allocator* a) { delete a; }

kvq_status kvq_alloc_pages(kvq_allocator* a, int32_t n, int32_t* out) {
    if (!a || n < 0 || (n > 0 && !out)) return KVQ_ERR_INVALID_ARG;
    if ((size_t)n > a->stack.size()) return KVQ_ERR_OUT_OF_PAGES;
    for (int32_t i = 0; i < n; ++i) {
        out[i] = a->stack.back();
        a->stack.pop_back();
        a->refs[out[i]] = 1;
    }
    return KVQ_OK;
}

kvq_status kvq_free_pages(kvq_allocator* a, int32_t n, const int32_t* pages) {
    if (!a || n < 0 || (n > 0 && !pages)) return KVQ_ERR_INVALID_ARG;
    std::vector<int32_t> cnt;
    if (!count_held(a, n, pages, cnt)) return KVQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (cnt[pages[i]] > a->refs[pages[i]]) return KVQ_ERR_INVALID_ARG;  // more drops than references
    try {
        a->stack.reserve(a->stack.size() + (size_t)n);
    } catch (...) {
        return KVQ_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i)
        if (--a->refs[pages[i]] == 0) a->stack.push_back(pages[i]);
    return KVQ_OK;
}

kvq_status kvq_share_pages(kvq_allocator* a, int32_t n, const int32_t* pages) {
    if (!a || n < 0 || (n > 0 && !pages)) return KVQ_ERR_INVALID_ARG;
    std::vector<int32_t> cnt;
    if (!count_held(a, n, pages, cnt)) return KVQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if ((int64_t)a->refs[pages[i]] + cnt[pages[i]] > INT32_MAX) return KVQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) ++a->refs[pages[i]];
    return KVQ_OK;
}

kvq_status kvq_page_refcount(const kvq_allocator* a, int32_t page, int32_t* refs) {
    if (!a || !refs || page < 0 || page >= a->num_pages) return KVQ_ERR_INVALID_ARG;
    *refs = a->refs[page];
    return KVQ_OK;
}

int32_t kvq_allocator_free_count(const kvq_allocator* a) {
    return a ? (int32_t)a->stack.size() : 0;
}

}  // extern "C"
