// kvq_decode_int8kc.cu -- instantiations of the tensor-core decode kernel for
// the INT8 scheme with per-channel K scales (separate translation unit so the
// schemes compile in parallel).
#include "kvq_tc.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int8kc(const DecodeParams& p, int G, cudaStream_t s) {
    return tc::launch_scheme<KVQ_INT8_KCHAN>(p, G, s);
}

int decode_ctas_per_sm_int8kc(int head_dim, int G, int /*B*/) {
    return tc::ctas_per_sm_scheme<KVQ_INT8_KCHAN>(head_dim, G);
}

}  // namespace kvq
