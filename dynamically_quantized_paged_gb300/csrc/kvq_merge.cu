// kvq_merge.cu -- the split merge (K3) instantiations and the scheme dispatch
// of the decode launch.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_partial(const DecodeParams& p, int G, cudaStream_t s) {
    switch (p.c.scheme) {
        case KVQ_INT8_SYM_TOKEN: return launch_decode_partial_int8(p, G, s);
        case KVQ_FP8E4M3_TOKEN: return launch_decode_partial_fp8(p, G, s);
        case KVQ_INT4_SYM_G32: return launch_decode_partial_int4sym(p, G, s);
        case KVQ_INT8_KCHAN: return launch_decode_partial_int8kc(p, G, s);
        default: return launch_decode_partial_int4(p, G, s);
    }
}

int decode_ctas_per_sm(int scheme, int head_dim, int G, int B) {
    switch (scheme) {
        case KVQ_INT8_SYM_TOKEN: return decode_ctas_per_sm_int8(head_dim, G, B);
        case KVQ_FP8E4M3_TOKEN: return decode_ctas_per_sm_fp8(head_dim, G, B);
        case KVQ_INT4_SYM_G32: return decode_ctas_per_sm_int4sym(head_dim, G, B);
        case KVQ_INT8_KCHAN: return decode_ctas_per_sm_int8kc(head_dim, G, B);
        default: return decode_ctas_per_sm_int4(head_dim, G, B);
    }
}

cudaError_t launch_decode_merge(const DecodeParams& p, int G, cudaStream_t s) {
    if (p.c.head_dim == 128) {
        switch (G) {
            case 1: return launch_decode_merge_t<128, 1>(p, s);
            case 2: return launch_decode_merge_t<128, 2>(p, s);
            case 4: return launch_decode_merge_t<128, 4>(p, s);
            default: return launch_decode_merge_t<128, 8>(p, s);
        }
    }
    switch (G) {
        case 1: return launch_decode_merge_t<64, 1>(p, s);
        case 2: return launch_decode_merge_t<64, 2>(p, s);
        case 4: return launch_decode_merge_t<64, 4>(p, s);
        default: return launch_decode_merge_t<64, 8>(p, s);
    }
}

}  // namespace kvq
