// kvq_decode_int4.cu -- instantiations of the split-K decode kernel for the
// int4 scheme (separate translation unit so the schemes compile in parallel).
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int4(const DecodeParams& p, int G, cudaStream_t s) {
    return launch_decode_partial_scheme<KVQ_INT4_ASYM_G32>(p, G, s);
}

}  // namespace kvq
