// kvq_decode_fp8.cu -- instantiations of the split-K decode kernel for the
// fp8 scheme (separate translation unit so the schemes compile in parallel).
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_partial_fp8(const DecodeParams& p, int G, cudaStream_t s) {
    return launch_decode_partial_scheme<KVQ_FP8E4M3_TOKEN>(p, G, s);
}

}  // namespace kvq
