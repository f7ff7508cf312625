// kvq_decode_tc_fp4v.cu -- the tensor-core decode kernel (kvq_decode_tc.cuh) for
// V in NVFP4.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_fp4v(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    return launch_for_v<KVQ_CODEC_NVFP4>(a, q_dtype, st);
}

int decode_tc_fp4v_ctas_per_sm(int k_codec, int head_dim, int nt)
{
    return per_sm_for_v<KVQ_CODEC_NVFP4>(k_codec, head_dim, nt);
}

}  // namespace kvq
