// kvq_decode_tc_q8v.cu -- the tensor-core decode kernel (kvq_decode_tc.cuh) for
// V in q8_0.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_q8v(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    return launch_for_v<KVQ_CODEC_Q8_0>(a, q_dtype, st);
}

int decode_tc_q8v_ctas_per_sm(int k_codec, int head_dim, int nt)
{
    return per_sm_for_v<KVQ_CODEC_Q8_0>(k_codec, head_dim, nt);
}

}  // namespace kvq
