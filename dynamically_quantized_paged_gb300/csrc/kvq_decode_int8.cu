// kvq_decode_int8.cu -- instantiations of the tensor-core decode kernel for the
// int8 scheme (separate translation unit so the schemes compile in parallel).
#include "kvq_tc.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int8(const DecodeParams& p, int G, cudaStream_t s) {
    return tc::launch_scheme<KVQ_INT8_SYM_TOKEN>(p, G, s);
}

int decode_ctas_per_sm_int8(int head_dim, int G, int /*B*/) {
    return tc::ctas_per_sm_scheme<KVQ_INT8_SYM_TOKEN>(head_dim, G);
}

}  // namespace kvq
