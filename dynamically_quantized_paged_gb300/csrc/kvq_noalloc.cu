// kvq_noalloc.cu -- kvq_decode_attn_noalloc: decode attention for callers
// that cannot allocate device memory.
//
// Some callers must not call cudaMalloc: code that runs inside another
// framework's memory pool (a direct allocation bypasses the pool's accounting
// and fails once the pool holds the device memory), and latency-critical
// paths that cannot accept the implicit device synchronization an allocation
// may bring.  kvq_decode_attn asks them for a workspace; this entry point
// instead uses a fixed scratch array that lives in the library itself.
//
// The array is a file-scope __device__ object of KVQ_STATIC_SCRATCH_BYTES
// bytes: every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, so the device address
// is fetched with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on that device (refused while the stream is
// being captured, since the lookup may load the module).  Every call shares
// the array and finds the previous call's contents in it: the only words
// that must start in a known state, the per-segment arrival counters of the
// split merge, are cleared on the stream before each launch (no other byte is
// read before the same launch writes it).  Two calls whose kernels overlap on
// the GPU race on the array.
#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

constexpr int MAX_DEVICES = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[MAX_DEVICES];

// Device address of the scratch array on the current device: looked up on
// the first call per device (not while `s` is capturing: the lookup may load
// the module, which a capture forbids).  Returns KVQ_OK with *out set, or the
// status to return.
kvq_status scratch_on_current_device(cudaStream_t s, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return KVQ_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return KVQ_ERR_INVALID_ARG;  // first call inside a capture
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KVQ_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const void* q,
                                              const int32_t* block_table, const int32_t* seq_lens,
                                              float* out, int32_t num_seqs, int32_t num_q_heads,
                                              int32_t max_pages_per_seq, float softmax_scale,
                                              kvq_stream_t stream) {
    size_t need = 0;
    kvq_status st = kvq_decode_workspace_bytes(cache, num_seqs, num_q_heads, max_pages_per_seq, &need);
    if (st != KVQ_OK) return st;
    if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;  // beyond the fixed array
    if (num_seqs == 0) return KVQ_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    st = scratch_on_current_device(s, &scratch);
    if (st != KVQ_OK) return st;
    size_t ctr_off = 0, ctr_bytes = 0;
    st = kvq::decode_counter_region(cache, num_seqs, num_q_heads, &ctr_off, &ctr_bytes);
    if (st != KVQ_OK) return st;
    if (ctr_off + ctr_bytes > need) return KVQ_ERR_CUDA;  // layout disagreement: launch nothing
    if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + ctr_off, 0, ctr_bytes, s) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return kvq_decode_attn(cache, q, block_table, seq_lens, out, num_seqs, num_q_heads, max_pages_per_seq,
                           softmax_scale, scratch, (size_t)KVQ_STATIC_SCRATCH_BYTES, stream);
}
