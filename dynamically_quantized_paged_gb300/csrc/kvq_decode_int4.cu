// kvq_decode_int4.cu -- decode instantiations for the int4 scheme (separate
// translation unit so the schemes compile in parallel): the CUDA-core kernel
// for GQA ratios up to 4, the tensor-core kernel for GQA 8.
#include "kvq_alu.cuh"
#include "kvq_tc.cuh"

namespace kvq {

cudaError_t launch_decode_partial_int4(const DecodeParams& p, int G, cudaStream_t s) {
    if (decode_alu_warps(KVQ_INT4_ASYM_G32, G) > 0) return alu::launch_scheme<KVQ_INT4_ASYM_G32>(p, G, s);
    return tc::launch_scheme<KVQ_INT4_ASYM_G32>(p, G, s);
}

int decode_ctas_per_sm_int4(int head_dim, int G, int B) {
    if (decode_alu_warps(KVQ_INT4_ASYM_G32, G) > 0) return alu::ctas_per_sm_scheme<KVQ_INT4_ASYM_G32>(head_dim, G, B);
    return tc::ctas_per_sm_scheme<KVQ_INT4_ASYM_G32>(head_dim, G);
}

}  // namespace kvq
