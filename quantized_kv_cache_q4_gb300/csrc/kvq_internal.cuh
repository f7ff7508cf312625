// kvq_internal.cuh -- declarations shared by the CUDA translation units of
// libkvq.so (kernel launchers and the small device helpers they share).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvq.h"

namespace kvq {

constexpr int kWarp = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 4-bit codecs (Q4_G64, Q4_G32) share the code layout; q8_0 has one byte per value.
__host__ __device__ constexpr bool is_q4(int codec) { return codec == KVQ_CODEC_Q4_G64 || codec == KVQ_CODEC_Q4_G32; }
__host__ __device__ constexpr int group_size(int codec) { return codec == KVQ_CODEC_Q4_G64 ? 64 : 32; }
__host__ __device__ constexpr int row_bytes(int codec, int d) { return is_q4(codec) ? d / 2 : d; }
__host__ __device__ constexpr int scales_per_row(int codec, int d) { return d / group_size(codec); }
__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch: a kernel launched with launch_pdl() may start
// while the previous kernel in the stream is finishing; pdl_wait() blocks until
// that kernel's writes are visible and must come before the first global read
// or write.  pdl_trigger() lets the next kernel start launching.  Both are
// no-ops when the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// A cache plane as the kernels see it.
struct Plane {
    int codec;
    uint8_t *qs;
    __half *sc;
};

struct AppendArgs {
    Plane plane[2];             // K then V (n_planes of them are used)
    const void *src[2];
    int n_planes;
    int n_seq, n_new, n_kv_heads, head_dim, capacity;
    const int32_t *pos0;
    int32_t *err;
};

struct DecodeArgs {
    Plane k, v;
    const void *q;
    int n_seq, n_kv_heads, n_heads, n_q, head_dim, capacity;
    float scale_log2;           // softmax_scale * log2(e)
    const int32_t *kv_len;
    int max_kv_len;
    int n_splits;
    float *out, *out_lse;       // final results (used when n_splits == 1)
    float *part_o, *part_lse;   // [n_splits][rows][D], [n_splits][rows] (n_splits > 1)
    int32_t *err;
};

// Token range [lo, hi) of split `split` for a sequence whose last query row
// sees `len` keys: chunks of ceil(len / n_splits) rounded up to 64 tokens.
__host__ __device__ inline void split_range(int len, int n_splits, int split, int &lo, int &hi)
{
    int chunk = (int)ceil_div(ceil_div(len, n_splits), 64) * 64;
    long long l = (long long)split * chunk;
    lo = (int)(l < len ? l : len);
    long long h = l + chunk;
    hi = (int)(h < len ? h : len);
}

// Set the message kvq_last_error() returns on the calling thread.
void set_last_error(const char *msg);

cudaError_t launch_append(const AppendArgs &a, bool src_f16, cudaStream_t st);
cudaError_t launch_decode_simt(const DecodeArgs &a, int q_dtype, cudaStream_t st);
// Tensor-core path: 1..32 query rows per kv head, head_dim 64/128/256, any K and V codec.
bool decode_tc_supported(const DecodeArgs &a);
cudaError_t launch_decode_tc(const DecodeArgs &a, int q_dtype, cudaStream_t st);
// CTAs of the tensor-core decode kernel that fit on one SM for these caches and
// query rows per kv head; 0 if that kernel does not take them or no device answers.
int decode_ctas_per_sm(int k_codec, int v_codec, int head_dim, int rows_per_kv_head);
// The same kernel for V in Q4_G32 and in q8_0 (translation units of their own).
cudaError_t launch_decode_tc_g32(const DecodeArgs &a, int q_dtype, cudaStream_t st);
int decode_tc_g32_ctas_per_sm(int k_codec, int head_dim, int n_tiles);
cudaError_t launch_decode_tc_q8v(const DecodeArgs &a, int q_dtype, cudaStream_t st);
int decode_tc_q8v_ctas_per_sm(int k_codec, int head_dim, int n_tiles);
cudaError_t launch_merge(const float *po, const float *pl, int n_splits, int rows, int head_dim,
                         float *out, float *out_lse, cudaStream_t st);
cudaError_t launch_dequant(const Plane &p, int64_t n_rows, int head_dim, float *out, cudaStream_t st);

}  // namespace kvq
