// kvq_decode_int8.cu -- instantiations of the split-K decode kernel for the
// int8 scheme (separate translation unit so the schemes compile in parallel).
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int8(const DecodeParams& p, int G, cudaStream_t s) {
    return launch_decode_partial_scheme<KVQ_INT8_SYM_TOKEN>(p, G, s);
}

}  // namespace kvq
