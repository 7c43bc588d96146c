// kvq_decode_int4sym.cu -- instantiations of the tensor-core decode kernel for
// the symmetric int4 scheme (separate translation unit so the schemes compile
// in parallel).
#include "kvq_tc.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int4sym(const DecodeParams& p, int G, cudaStream_t s) {
    return tc::launch_scheme<KVQ_INT4_SYM_G32>(p, G, s);
}

int decode_ctas_per_sm_int4sym(int head_dim, int G, int /*B*/) {
    return tc::ctas_per_sm_scheme<KVQ_INT4_SYM_G32>(head_dim, G);
}

}  // namespace kvq
