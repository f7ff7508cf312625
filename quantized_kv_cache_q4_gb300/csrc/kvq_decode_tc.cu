// kvq_decode_tc.cu -- the tensor-core decode kernel (kvq_decode_tc.cuh) for V
// in Q4_G64, and the dispatch of the decode kernels: prompt chunks to the
// tcgen05 kernel, up to 8 rows per kv head over Q4_G64 V to the single-warp-
// block kernel, everything else to kvq_decode_tc.cuh's four V-codec instances.
#include "kvq_decode_tc.cuh"

namespace kvq {

bool decode_tc_supported(const DecodeArgs &a)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    return R >= 1 &&
           (a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256) && rows < (1LL << 31) &&
           tensor_maps_available();
}

int decode_ctas_per_sm(int k_codec, int v_codec, int head_dim, int rows_per_kv_head)
{
    if (rows_per_kv_head < 1) return 0;
    if (decode_warp_shape(k_codec, v_codec, head_dim, rows_per_kv_head)) return decode_warp_ctas_per_sm(k_codec, v_codec, head_dim);
    const int nt = (min(rows_per_kv_head, kTcRowsPerCta) + 7) / 8;
    if (v_codec == KVQ_CODEC_Q4_G64) return per_sm_for_v<KVQ_CODEC_Q4_G64>(k_codec, head_dim, nt);
    if (v_codec == KVQ_CODEC_Q4_G32) return decode_tc_g32_ctas_per_sm(k_codec, head_dim, nt);
    if (v_codec == KVQ_CODEC_Q8_0) return decode_tc_q8v_ctas_per_sm(k_codec, head_dim, nt);
    if (v_codec == KVQ_CODEC_NVFP4) return decode_tc_fp4v_ctas_per_sm(k_codec, head_dim, nt);
    return 0;
}

cudaError_t launch_decode_tc(const DecodeArgs &args, int q_dtype, cudaStream_t st)
{
    if (prefill_umma_takes(args, q_dtype)) return launch_prefill_umma(args, st);
    if (decode_warp_takes(args)) return launch_decode_warp(args, q_dtype, st);
    DecodeArgs a = args;
    a.n_row_blocks = tc_row_blocks(a.n_q * (a.n_heads / a.n_kv_heads));
    if (a.v.codec == KVQ_CODEC_Q4_G64) return launch_for_v<KVQ_CODEC_Q4_G64>(a, q_dtype, st);
    if (a.v.codec == KVQ_CODEC_Q4_G32) return launch_decode_tc_g32(a, q_dtype, st);
    if (a.v.codec == KVQ_CODEC_Q8_0) return launch_decode_tc_q8v(a, q_dtype, st);
    if (a.v.codec == KVQ_CODEC_NVFP4) return launch_decode_tc_fp4v(a, q_dtype, st);
    return cudaErrorInvalidValue;
}

}  // namespace kvq
