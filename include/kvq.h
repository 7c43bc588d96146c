/*
 * kvq.h -- dynamic KV-cache quantization with fused-dequantization paged
 * decode attention, for NVIDIA GB300 (sm_103a).  Plain C ABI.
 *
 * The operations follow three web pages on the subject:
 *  [P1] "Dynamic KV Cache Quantization for Fast LLM Inference"
 *  [P2] "What is KV Cache Optimization? Definition, Quantization & Memory
 *       Management in Enterprise AI?"
 *  [P3] "KV Cache Optimization: Strategies for Faster LLM Inference"
 * Their pipeline ([P2] section "Technical Architecture"): capture each
 * token's key/value projections, quantize them with a dynamically computed
 * scale, store the codes in fixed-size non-contiguous pages, and dequantize
 * inside the attention kernel while decoding.
 *
 * Conventions shared by every call:
 *  - Every pointer argument named as device memory must be device memory of
 *    the current CUDA device, allocated and owned by the caller (the one
 *    exception: the host-tier pools of kvq_cache, below, are page-locked
 *    host memory that the device addresses directly).  The library
 *    calls no allocator and keeps no pointer after a call returns; its own
 *    device memory is static: a per-device error word, and the fixed scratch
 *    array of kvq_decode_attn_noalloc.
 *  - Device buffers must start on a 16-byte boundary (kvq_append,
 *    kvq_decode_*: the page pools, q, k, v, out, workspace).
 *  - Calls that launch work are asynchronous on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream) and never synchronize, except
 *    kvq_last_device_error.
 *  - Every call returns a kvq_status; nothing throws across the ABI.  Argument
 *    errors are detected on the host before any launch, and then nothing is
 *    launched.  Errors that only the device can see (a page id outside the
 *    pool, a slot outside the pool, a sequence longer than its table row, a
 *    wait that timed out) are recorded in a per-device flag word, the
 *    offending access is skipped, and kvq_last_device_error reports them.
 *  - The kernels never trap and never wait without a time limit.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvq_stream_t; /* same type as cudaStream_t */

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, bad size or shape */
    KVQ_ERR_SCHEME_MISMATCH = 2, /* scheme argument differs from cache->scheme */
    KVQ_ERR_OUT_OF_PAGES = 3,    /* allocator exhausted ([P1]'s out-of-memory case) */
    KVQ_ERR_BAD_TABLE = 4,       /* device saw a page / slot / length outside the pool */
    KVQ_ERR_CUDA = 5,            /* a CUDA runtime call failed (no device, launch error) */
    KVQ_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait ran out */
    KVQ_ERR_UNSUPPORTED = 7,     /* valid but not implemented: head_dim, GQA ratio, page size */
    KVQ_ERR_WORKSPACE = 8        /* workspace smaller than kvq_decode_workspace_bytes */
} kvq_status;

/* Quantization schemes ([P1] section "Understanding Dynamic Quantization
 * Techniques for KV Caches (e.g., INT8, INT4)"; FP8 from [P2] "Technical
 * Architecture").  All scales are computed on the fly from the data. */
typedef enum kvq_scheme {
    /* per (token, KV head): scale = max|x| / 127 (fp32), code = round-half-
     * even(x / scale) in [-127, 127]; an all-zero row stores scale 1.0. */
    KVQ_INT8_SYM_TOKEN = 1,
    /* per (token, KV head): scale = max|x| / 448 (fp32), code = E4M3
     * round-to-nearest-even of x / scale with saturation to +-448. */
    KVQ_FP8E4M3_TOKEN = 2,
    /* per (token, KV head, 32-channel group): zero = fp16 round-down of the
     * group minimum, scale = fp16 round-up of (max - zero) / 15 (1.0 if that
     * is 0), code = round-half-even((x - zero) / scale) in [0, 15], two codes
     * per byte, even channel in the low nibble. */
    KVQ_INT4_ASYM_G32 = 3,
    /* per (token, KV head, 32-channel group): scale = max|x| / 7 (fp32; 1.0
     * for an all-zero group), code = round-half-even(x / scale) in [-7, 7],
     * stored as 4-bit two's complement, two codes per byte, even channel in
     * the low nibble; no zero-point ([P1] with bits = 4). */
    KVQ_INT4_SYM_G32 = 4,
    /* INT8 with per-channel K scales ([P3] section "KV Cache Quantization:
     * When and How to Compress": per-channel keeps more than per-tensor).
     * V is KVQ_INT8_SYM_TOKEN throughout.  K takes one scale per (page, KV
     * head, channel), fixed when the page is sealed (kvq_seal_pages) from
     * the page's bf16 rows, which the append keeps in a residual slot while
     * the page fills; until then the page's K rows are stored by the token
     * rule.  Dequantized K = code * k_chan[page][head][channel] (fp16) *
     * k_scales[page][head][token] (fp32).  An open page has channel factors
     * 1.0 (written by the append of the token at offset 0) and its tokens'
     * INT8 scales.  A sealed (page, head) block x[t][j] stores, with
     * s_j = max_t |x| / 127 and S = max_j s_j (fp32 divisions):
     *   k_chan[j]  = fp16 round-up of s_j / S (fp32 division), in [0, 1];
     *   code       = round-half-even(x / (k_chan[j] * S)) in [-127, 127], the
     *                product and the quotient fp32; 0 where k_chan[j] = 0;
     *   k_scales[t] = S for every token.
     * An all-zero block stores codes 0, factors 1.0 and scales 1.0. */
    KVQ_INT8_KCHAN = 5
} kvq_scheme;

/* One layer of the paged quantized cache ([P1] section "Integrating Dynamic
 * Quantization with PagedAttention ...": fixed-size blocks at scattered
 * physical locations; [P3] section "How vLLM Implements KV Cache
 * Optimization": 16 tokens per block by default).  All six pools are
 * caller-owned device memory, sized by kvq_cache_bytes.  Layout:
 *   codes   [num_pages][num_kv_heads][page_size][head_dim]    int8 / e4m3
 *           [num_pages][num_kv_heads][page_size][head_dim/2]  both INT4 (packed)
 *   scales  [num_pages][num_kv_heads][page_size]              fp32
 *           [num_pages][num_kv_heads][page_size][head_dim/32] fp16 (INT4 asym)
 *           [num_pages][num_kv_heads][page_size][head_dim/32] fp32 (INT4 sym)
 *   zeros   asymmetric INT4 only, same shape as its scales; NULL otherwise.
 * The token stored at physical slot s lives in page s / page_size at
 * offset s % page_size.  Supported: head_dim 64 or 128, page_size a positive
 * multiple of 16, num_kv_heads >= 1.  Several layers share one block table
 * by using one descriptor per layer.
 *
 * Cold-page tier ([P3] section "KV Cache Offloading: Moving Data Between GPU
 * and CPU": inactive cache kept in CPU RAM instead of GPU memory).  With
 * host_pages > 0 the page ids num_pages .. num_pages + host_pages - 1 name
 * pages of a second set of pools, host_k_codes .. host_v_zeros, laid out
 * exactly as above with host_pages pages and living in page-locked host
 * memory that the device can address (cudaHostAlloc / pinned memory: on
 * GB300 the GPU reads it over NVLink-C2C).  That id range is the residency
 * map: a block-table entry >= num_pages says the page is host-resident.
 * Every call treats both tiers alike: the append writes, and both decode
 * kernels read, host-resident pages in place (no staging copy), and
 * kvq_copy_page moves a page between the tiers (offload: device page to a
 * free host page; fetch: the reverse), after which the caller rewrites the
 * block-table entry.  host_pages = 0 (with NULL host pools) is the plain
 * device-only cache.  A slot s names page s / page_size in either tier.
 *
 * KVQ_INT8_KCHAN adds the channel factors, k_chan [num_pages][num_kv_heads]
 * [head_dim] fp16 (host_k_chan likewise for the host tier), and the residual
 * pool k_resid [resid_slots][num_kv_heads][page_size][head_dim] bf16 (device
 * memory; resid_slots may be 0 with k_resid NULL), sized by kvq_kchan_bytes.
 * These fields are ignored (and may be anything) for the other schemes. */
typedef struct kvq_cache {
    int32_t scheme;       /* kvq_scheme */
    int32_t num_pages;
    int32_t page_size;    /* tokens per page */
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t group;        /* channels per INT4 group (both INT4 schemes): must be 32; ignored otherwise */
    void* k_codes;
    void* v_codes;
    void* k_scales;
    void* v_scales;
    void* k_zeros;        /* INT4 only */
    void* v_zeros;        /* INT4 only */
    int32_t host_pages;   /* pages of the host tier (0: none) */
    void* host_k_codes;   /* host-tier pools, same layout with host_pages pages */
    void* host_v_codes;
    void* host_k_scales;
    void* host_v_scales;
    void* host_k_zeros;   /* asymmetric INT4 only */
    void* host_v_zeros;   /* asymmetric INT4 only */
    void* k_chan;         /* KVQ_INT8_KCHAN only: channel factors */
    void* host_k_chan;    /* KVQ_INT8_KCHAN only: host-tier channel factors */
    void* k_resid;        /* KVQ_INT8_KCHAN only: residual bf16 K rows of open pages */
    int32_t resid_slots;  /* KVQ_INT8_KCHAN only: slots of k_resid */
} kvq_cache;

/* Human-readable name of a status.  Never NULL; static storage. */
const char* kvq_status_string(kvq_status status);

/* Bytes of ONE of the K / V pools of each kind for the given geometry (the
 * V pools have the same sizes).  zero_bytes is 0 for the 8-bit schemes.
 * Per token and KV head this is head_dim code bytes (head_dim/2 for INT4)
 * plus 4 scale bytes (INT4: 2 + 2 bytes per 32-channel group): the
 * bytes-per-token rule of [P2] "Technical Architecture" (2 x layers x KV
 * heads x head_dim x bytes per element) with the scale overhead separate.
 * Host only; any output pointer may be NULL. */
kvq_status kvq_cache_bytes(int32_t scheme, int32_t num_pages, int32_t page_size,
                           int32_t num_kv_heads, int32_t head_dim, size_t* code_bytes,
                           size_t* scale_bytes, size_t* zero_bytes);

/* KVQ_INT8_KCHAN's extra pools: chan_bytes for k_chan with num_pages pages
 * (2 bytes per page, KV head and channel), resid_bytes for k_resid with
 * resid_slots slots (page_size bf16 rows per slot and KV head).  Its codes
 * and scales are sized by kvq_cache_bytes like KVQ_INT8_SYM_TOKEN.  Host
 * only; either output may be NULL. */
kvq_status kvq_kchan_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
                           int32_t resid_slots, size_t* chan_bytes, size_t* resid_bytes);

/* Quantize-append ([P2] "Key-Value Tensor Capture" and "Dynamic FP8/INT8
 * Quantization"; [P1] "Understanding Dynamic Quantization Techniques").
 *   k, v          device, bf16 [num_tokens][num_kv_heads][head_dim], the new
 *                 tokens' key / value projections.
 *   slot_mapping  device, int64 [num_tokens]: physical slot of each token
 *                 (page id * page_size + offset); a negative slot skips the
 *                 token.  A slot >= num_pages * page_size is skipped and
 *                 flagged KVQ_ERR_BAD_TABLE.
 *   block_table   device, int32 [num_seqs][max_pages_per_seq], or NULL.  When
 *                 given, its entries are checked (each must be -1 or a page id
 *                 of the pool) and violations flagged KVQ_ERR_BAD_TABLE; the
 *                 codes are written through slot_mapping either way.
 *   scheme        must equal cache->scheme (else KVQ_ERR_SCHEME_MISMATCH).
 *   num_pages * page_size and num_tokens * num_kv_heads * 2 must be below
 *   2^31 (else KVQ_ERR_INVALID_ARG): slots and rows are indexed in 32 bits.
 * Writes, for every token and KV head, the codes and scale (and INT4 zero)
 * at the slot.  num_tokens == 0 launches nothing. */
kvq_status kvq_append(const kvq_cache* cache, const int32_t* block_table, int32_t num_seqs,
                      int32_t max_pages_per_seq, const int64_t* slot_mapping, const void* k,
                      const void* v, int32_t num_tokens, int32_t scheme, kvq_stream_t stream);

/* Quantize-append for KVQ_INT8_KCHAN: kvq_append (same arguments, rules and
 * errors) plus, per token,
 *   resid_slot    device, int32 [num_tokens], or NULL (no residual rows): the
 *                 residual slot that keeps the token's bf16 K rows (every KV
 *                 head), at the token's page offset; -1 keeps none.  A slot
 *                 >= cache->resid_slots skips the token (nothing written) and
 *                 flags KVQ_ERR_BAD_TABLE.
 * The token at offset 0 of a page also sets that page's channel factors to
 * 1.0 (it opens the page; a page is appended to only while open).  Pages
 * whose bf16 rows are not all in one residual slot cannot be sealed and
 * keep the token rule.  KVQ_ERR_SCHEME_MISMATCH unless cache->scheme is
 * KVQ_INT8_KCHAN.  kvq_append on such a cache equals this call with
 * resid_slot NULL. */
kvq_status kvq_append_kchan(const kvq_cache* cache, const int32_t* block_table, int32_t num_seqs,
                            int32_t max_pages_per_seq, const int64_t* slot_mapping, const int32_t* resid_slot,
                            const void* k, const void* v, int32_t num_tokens, kvq_stream_t stream);

/* Seals pages of a KVQ_INT8_KCHAN cache: for each i < n, page pages[i] (in
 * either tier; every KV head) takes the per-channel K rule of the
 * page_size bf16 rows in residual slot resid_slots[i] (the rule under
 * KVQ_INT8_KCHAN): its K codes, channel factors and K token scales are
 * rewritten; V is left as it is.  The caller seals a page once the append
 * that fills it is on the stream (every offset of the slot written for
 * that page), and may then reuse the slot.  pages, resid_slots: device,
 * int32 [n].  An id outside its pool skips that pair and flags
 * KVQ_ERR_BAD_TABLE.  n == 0 launches nothing; KVQ_ERR_SCHEME_MISMATCH
 * unless cache->scheme is KVQ_INT8_KCHAN; KVQ_ERR_INVALID_ARG if the cache
 * has no residual pool or n < 0. */
kvq_status kvq_seal_pages(const kvq_cache* cache, const int32_t* pages, const int32_t* resid_slots, int32_t n,
                          kvq_stream_t stream);

/* Device scratch needed by kvq_decode_attn / kvq_decode_partial /
 * kvq_decode_merge for this cache geometry and query-head count on the
 * current device (split-K partials: at most two per persistent CTA).  The
 * size does not depend on the sequence lengths. */
kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_pages_per_seq,
                                      size_t* bytes);

/* Fused-dequantization paged GQA decode attention ([P2] "Fused
 * Dequantization Attention Kernel"; [P1] "Recap of KV Caching": the new
 * token attends to every cached token, itself included).
 *   q             device, bf16 [num_seqs][num_q_heads][head_dim].
 *   block_table   device, int32 [num_seqs][max_pages_per_seq]: logical page
 *                 i of sequence b is physical page block_table[b][i].
 *   seq_lens      device, int32 [num_seqs]: cached tokens per sequence (0 is
 *                 allowed and gives a zero output row).
 *   out           device, fp32 [num_seqs][num_q_heads][head_dim].
 *   softmax_scale <= 0 selects 1/sqrt(head_dim).
 *   workspace     device, >= kvq_decode_workspace_bytes bytes; contents need
 *                 no initialization and are clobbered.
 * Query head g reads KV head g / (num_q_heads / num_kv_heads); the ratio must
 * be 1, 2, 4 or 8.  num_seqs <= 4096.  The work is split over a persistent
 * grid along logical token positions only, so the output does not depend on
 * which physical pages hold the tokens.  One launch: a (sequence, KV head)
 * whose tokens are split across CTAs is merged by the CTA that delivers its
 * last partial (arrivals are counted in workspace words tagged with a per-call
 * generation, so the workspace needs no zeroing; the last arrival clears its
 * word, so a recorded call can be replayed, e.g. from a CUDA graph, as long
 * as no two calls sharing a workspace run at the same time).  The kernel is
 * launched with programmatic stream serialization: its CTAs may become
 * resident while the kernel ahead of it on the stream (e.g. kvq_append) is
 * still running and set up what needs no input (barriers, tensor memory),
 * but read or write no array argument, cache or workspace byte before that
 * kernel has completed and its writes are visible.
 * kvq_decode_partial followed by kvq_decode_merge is the equivalent
 * two-launch form and gives bitwise the same output. */
kvq_status kvq_decode_attn(const kvq_cache* cache, const void* q, const int32_t* block_table,
                           const int32_t* seq_lens, float* out, int32_t num_seqs,
                           int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                           void* workspace, size_t workspace_bytes, kvq_stream_t stream);

/* Output element types of kvq_decode_attn_out. */
typedef enum kvq_out_dtype {
    KVQ_OUT_F32 = 0,  /* fp32, as kvq_decode_attn */
    KVQ_OUT_BF16 = 1  /* bf16: the fp32 result rounded to nearest even */
} kvq_out_dtype;

/* kvq_decode_attn with the output element type chosen by out_dtype:
 *   out  device, [num_seqs][num_q_heads][head_dim] of fp32 (KVQ_OUT_F32) or
 *        bf16 (KVQ_OUT_BF16); 16-byte aligned.
 * Every output element is the value kvq_decode_attn computes, rounded to
 * nearest even when bf16 (the split partials stay fp32).  Other arguments,
 * rules and errors as kvq_decode_attn; an unknown out_dtype gives
 * KVQ_ERR_INVALID_ARG. */
kvq_status kvq_decode_attn_out(const kvq_cache* cache, const void* q, const int32_t* block_table,
                               const int32_t* seq_lens, void* out, int32_t out_dtype, int32_t num_seqs,
                               int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                               void* workspace, size_t workspace_bytes, kvq_stream_t stream);

/* One decode step that appends its own token ([P1] section "Recap of KV
 * Caching": each step stores the new token's key and value, then attends
 * over the whole cache; [P2] "Technical Architecture": capture, quantize,
 * store, fused dequantized attention).  Equivalent to kvq_append of one new
 * token per sequence followed by kvq_decode_attn_out, and bit-identical to
 * that pair (pools and output):
 *   k_new, v_new  device, bf16 [num_seqs][num_kv_heads][head_dim], 16-byte
 *                 aligned: each sequence's new key and value projections;
 *   seq_lens      counts that INCLUDE the new token, which is stored at
 *                 position seq_lens[b] - 1 of sequence b: the slot its
 *                 block-table row names for that position (a sequence of
 *                 length 0 appends nothing).
 * Other arguments, rules and errors as kvq_decode_attn_out.  Where the
 * CUDA-core kernel serves the GQA ratio (up to 4 for INT8, FP8 and
 * asymmetric INT4) this is ONE launch: the warp that reads a sequence's last
 * position quantizes the new token by the append's rule (the same device
 * code) into its staged copy of the page and into the cache.  Elsewhere it
 * is the append kernel followed by the decode, on the stream.
 * KVQ_ERR_UNSUPPORTED for KVQ_INT8_KCHAN, whose append needs residual slots
 * (kvq_append_kchan, then the decode). */
kvq_status kvq_decode_attn_append(const kvq_cache* cache, const void* k_new, const void* v_new, const void* q,
                                  const int32_t* block_table, const int32_t* seq_lens, void* out,
                                  int32_t out_dtype, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_pages_per_seq, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, kvq_stream_t stream);

/* The first launch of the two-launch form of kvq_decode_attn: every
 * (sequence, KV head) whose tokens one CTA covers entirely gets its final
 * output row; the rest leave split partials (max, sum, unnormalized output)
 * in the workspace.  Same arguments and rules as kvq_decode_attn. */
kvq_status kvq_decode_partial(const kvq_cache* cache, const void* q, const int32_t* block_table,
                              const int32_t* seq_lens, float* out, int32_t num_seqs,
                              int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                              void* workspace, size_t workspace_bytes, kvq_stream_t stream);

/* The second launch: log-sum-exp merge of the split partials into out, and
 * zero rows for empty sequences.  Must follow kvq_decode_partial on the same
 * stream with the same arguments. */
kvq_status kvq_decode_merge(const kvq_cache* cache, const void* q, const int32_t* block_table,
                            const int32_t* seq_lens, float* out, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_pages_per_seq, float softmax_scale,
                            void* workspace, size_t workspace_bytes, kvq_stream_t stream);

/* Table check: flags KVQ_ERR_BAD_TABLE if a sequence is longer than
 * max_pages_per_seq * page_size, or a page it uses is outside the pool. */
kvq_status kvq_validate_tables(const kvq_cache* cache, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t num_seqs,
                               int32_t max_pages_per_seq, kvq_stream_t stream);

/* Synchronizes `stream`, then returns and clears the current device's error
 * flags: KVQ_OK, KVQ_ERR_BAD_TABLE or KVQ_ERR_DEVICE_TIMEOUT (the latter wins
 * when both are set), or KVQ_ERR_CUDA if the synchronization failed. */
kvq_status kvq_last_device_error(kvq_stream_t stream);

/* ---- decode without a caller-provided workspace -----------------------------
 * The pages have no counterpart to this call; it is a convenience of this
 * library.  It is kvq_decode_attn for callers that cannot allocate device
 * memory: code running inside another framework's memory pool (a direct
 * cudaMalloc would bypass the pool's accounting and fail once the pool holds
 * the device memory) and latency-critical paths that cannot accept the
 * device synchronization an allocation may bring.
 *
 * Instead of a workspace it uses a scratch array of KVQ_STATIC_SCRATCH_BYTES
 * bytes compiled into the library: every GPU that loads the library holds
 * that memory until the process exits.  The call allocates nothing.  Its
 * first call on a device looks up the array's device address (set-up, once
 * per device, with that device current); make that first call before any
 * stream capture: a first call made while `stream` is capturing returns
 * KVQ_ERR_INVALID_ARG and enqueues nothing.  Every call shares the array and
 * leaves its contents behind; the words that must start cleared (the split
 * merge's arrival counters) are zeroed on `stream` by each call, with one
 * memset node ahead of the decode launch.  Calls whose kernels overlap on the
 * GPU (other streams, other host threads) race on the array: keep them
 * ordered.  Returns KVQ_ERR_WORKSPACE, enqueuing nothing, if this problem
 * would need more scratch than the array holds (kvq_decode_workspace_bytes
 * reports the need).  The cached address (like the library's per-device
 * error word) is not refreshed after cudaDeviceReset: do not use the library
 * in a process after resetting the device.  Other arguments, rules and
 * errors are those of kvq_decode_attn. */
#define KVQ_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const void* q, const int32_t* block_table,
                                   const int32_t* seq_lens, float* out, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t max_pages_per_seq,
                                   float softmax_scale, kvq_stream_t stream);

/* ---- host page allocator ([P3] "How vLLM Implements KV Cache
 * Optimization": pages are handed out on demand, only used pages cost
 * memory).  The free list starts as the page ids 0..num_pages-1 shuffled by
 * Fisher-Yates driven by SplitMix64(seed), so that physical pages are
 * scattered; allocation pops pages from the end of the list, freeing pushes
 * them back (last freed, first reused).  Pages are reference counted so
 * that sequences can share the pages of a common prefix ([P3] "How vLLM
 * Implements KV Cache Optimization": a prefix that many requests share is
 * cached once and reused; [P1] "Integrating ... PagedAttention": memory
 * sharing across the sequences of a batch): a page is allocated with one
 * reference, kvq_share_pages adds references, kvq_free_pages drops them, and
 * a page returns to the free list when its last reference is dropped.  Host
 * only, not thread-safe. */
typedef struct kvq_allocator kvq_allocator;

/* NULL if num_pages < 1 or the host allocation fails. */
kvq_allocator* kvq_allocator_create(int32_t num_pages, uint64_t seed);
void kvq_allocator_destroy(kvq_allocator* alloc);
/* Pops n page ids into out[0..n).  KVQ_ERR_OUT_OF_PAGES (nothing taken) if
 * fewer than n are free. */
kvq_status kvq_alloc_pages(kvq_allocator* alloc, int32_t n, int32_t* out);
/* Drops one reference to each of the n page ids (an id may repeat, once
 * per reference dropped); pages whose last reference goes are pushed back on
 * the free list in the order given.  KVQ_ERR_INVALID_ARG (nothing changed) if
 * an id is outside the pool, free, or repeated more often than it has
 * references. */
kvq_status kvq_free_pages(kvq_allocator* alloc, int32_t n, const int32_t* pages);
/* Adds one reference to each of the n page ids (an id may repeat, once per
 * reference added), for a sequence that reuses another's prefix pages in its
 * own block table.  KVQ_ERR_INVALID_ARG (nothing changed) if an id is outside
 * the pool or free, or a count would pass 2^31 - 1. */
kvq_status kvq_share_pages(kvq_allocator* alloc, int32_t n, const int32_t* pages);
/* *refs = the references page holds (0: free).  KVQ_ERR_INVALID_ARG if the
 * id is outside the pool or refs is NULL. */
kvq_status kvq_page_refcount(const kvq_allocator* alloc, int32_t page, int32_t* refs);
int32_t kvq_allocator_free_count(const kvq_allocator* alloc);

/* Copies every pool's contents of page src (codes, scales, INT4 zero-points,
 * channel factors: all of its KV heads and slots) to page dst on the stream.  Two uses:
 * copy-on-write, so that a sequence whose shared prefix ends inside a page
 * can take its own copy of that page before appending past the prefix; and
 * moving a page between the device and host tiers (offload of a cold page,
 * fetch of a page needed again).  Either way the caller then updates the
 * block-table entry and drops its reference to src.  One asynchronous copy
 * per pool (device-to-device, device-to-host, host-to-device or host-to-
 * host); no kernel.  KVQ_ERR_INVALID_ARG if src or dst is outside both
 * tiers or src == dst; KVQ_ERR_CUDA if a copy cannot be enqueued. */
kvq_status kvq_copy_page(const kvq_cache* cache, int32_t src, int32_t dst, kvq_stream_t stream);

/* kvq_copy_page for many pages in one launch: for each i < n, every pool's
 * contents of page src[i] are copied to page dst[i] (either tier: a batch of
 * offloads, fetches or copy-on-write copies; [P3] "KV Cache Offloading":
 * pages moved back when needed).  One kernel, 16-byte loads and stores; a
 * host-tier page is read or written in place over NVLink-C2C.
 *   src, dst  device, int32 [n].  The pairs must not overlap (no page is both
 *             a source and a destination, no destination twice); their
 *             order is unspecified.  A pair with an id outside both tiers,
 *             or src[i] == dst[i], is skipped and flagged KVQ_ERR_BAD_TABLE.
 * n == 0 launches nothing; KVQ_ERR_INVALID_ARG if n < 0 or an array is NULL
 * or not 4-byte aligned. */
kvq_status kvq_copy_pages(const kvq_cache* cache, const int32_t* src, const int32_t* dst, int32_t n,
                          kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
