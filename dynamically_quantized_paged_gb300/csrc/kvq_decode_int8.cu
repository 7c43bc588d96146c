// kvq_decode_int8.cu -- decode instantiations for the int8 scheme (separate
// translation unit so the schemes compile in parallel): the CUDA-core kernel
// for GQA ratios up to 4, the tensor-core kernel for GQA 8.
#include "kvq_alu.cuh"
#include "kvq_tc.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int8(const DecodeParams& p, int G, cudaStream_t s) {
    if (decode_alu_warps(KVQ_INT8_SYM_TOKEN, G) > 0) return alu::launch_scheme<KVQ_INT8_SYM_TOKEN>(p, G, s);
    return tc::launch_scheme<KVQ_INT8_SYM_TOKEN>(p, G, s);
}

int decode_ctas_per_sm_int8(int head_dim, int G, int B) {
    if (decode_alu_warps(KVQ_INT8_SYM_TOKEN, G) > 0) return alu::ctas_per_sm_scheme<KVQ_INT8_SYM_TOKEN>(head_dim, G, B);
    return tc::ctas_per_sm_scheme<KVQ_INT8_SYM_TOKEN>(head_dim, G);
}

}  // namespace kvq
