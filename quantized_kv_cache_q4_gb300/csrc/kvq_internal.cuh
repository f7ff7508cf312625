// kvq_internal.cuh -- declarations shared by the CUDA translation units of
// libkvq.so (kernel launchers and the small device helpers they share).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "kvq.h"

namespace kvq {

constexpr int kWarp = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The 4-bit integer codecs (Q4_G64, Q4_G32) and NVFP4 (E2M1 codes) store two
// codes per byte (value 2j in the low nibble); q8_0 one per byte.  Scales are
// fp16, except NVFP4's one E4M3 byte per 16 values.
__host__ __device__ constexpr bool is_q4(int codec) { return codec == KVQ_CODEC_Q4_G64 || codec == KVQ_CODEC_Q4_G32; }
__host__ __device__ constexpr bool is_fp4(int codec) { return codec == KVQ_CODEC_NVFP4; }
__host__ __device__ constexpr bool two_per_byte(int codec) { return is_q4(codec) || is_fp4(codec); }
__host__ __device__ constexpr int group_size(int codec)
{
    return codec == KVQ_CODEC_Q4_G64 ? 64 : codec == KVQ_CODEC_NVFP4 ? 16 : 32;
}
__host__ __device__ constexpr int row_bytes(int codec, int d) { return two_per_byte(codec) ? d / 2 : d; }
__host__ __device__ constexpr int scales_per_row(int codec, int d) { return d / group_size(codec); }
__host__ __device__ constexpr int scale_bytes(int codec) { return is_fp4(codec) ? 1 : 2; }
__host__ __device__ constexpr int scale_row_bytes(int codec, int d) { return scales_per_row(codec, d) * scale_bytes(codec); }
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

// Hardware conversions (exact): an E4M3 byte to fp32; a byte of two E2M1
// codes to fp16x2 bits (low nibble -> low half).
__device__ __forceinline__ float e4m3_to_float(uint32_t b)
{
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(b & 0xFFu));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte)
{
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte & 0xFFu));
    return h2;
}

// One scale of a plane row as fp32.
template <int CODEC>
__device__ __forceinline__ float load_scale(const uint8_t *row_scales, int g)
{
    if constexpr (is_fp4(CODEC)) return e4m3_to_float(row_scales[g]);
    else return __half2float(reinterpret_cast<const __half *>(row_scales)[g]);
}

// A cache plane as the kernels see it (sc: the scale plane as bytes).
struct Plane {
    int codec;
    uint8_t *qs;
    uint8_t *sc;
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
    int n_row_blocks = 1;       // tensor-core kernel: CTAs per (split, kv head), 32 query rows each
    // Key ranges that are one part of a longer context (host-tier streaming):
    // fixed_len >= 0 replaces kv_len[s] (one sequence, length known on the
    // host), and query token i sees len + causal_extra - n_q + i + 1 keys of
    // the range (capped by len): causal_extra counts the context's keys after
    // the range.
    int fixed_len = -1;
    int causal_extra = 0;
};

// Query rows per kv head the tensor-core kernel gives one CTA, and the blocks
// of them a kv head with R rows takes.
constexpr int kTcRowsPerCta = 32;
inline int tc_row_blocks(int rows_per_kv_head)
{
    return rows_per_kv_head > kTcRowsPerCta ? (int)ceil_div(rows_per_kv_head, kTcRowsPerCta) : 1;
}

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

// A positive per-device value (kernel occupancy, SM count), computed once per
// device by `compute` (which returns a value > 0, or <= 0 on failure and is
// then tried again on the next call).  Safe when several host threads make
// their first call at the same time: the first computes under a lock, the
// others wait for it, later calls read one atomic.
struct PerDevice {
    static constexpr int kMaxDevices = 64;
    std::atomic<int> value[kMaxDevices];
    std::mutex mu;
};

template <typename F>
inline int per_device(PerDevice &pd, int dev, F compute)
{
    if (dev < 0 || dev >= PerDevice::kMaxDevices) return compute();
    int v = pd.value[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    std::lock_guard<std::mutex> lock(pd.mu);
    v = pd.value[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    v = compute();
    if (v > 0) pd.value[dev].store(v, std::memory_order_release);
    return v;
}

// Set the message kvq_last_error() returns on the calling thread.
void set_last_error(const char *msg);
// Set it printf-style and return st.
kvq_status fail_msg(kvq_status st, const char *fmt, ...);
// The argument checks every cache goes through (KVQ_OK or the failure, with
// the message set).
kvq_status check_cache_args(const kvq_cache *c, const char *name);
// The split count kvq_decode_attention uses (n_splits = 0: its default).
int resolve_decode_splits(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q, int32_t max_kv_len,
                          int32_t n_splits);
// Decode attention with validated arguments and a resolved split count:
// launches the decode kernel and, with n_splits > 1, the merge into out/out_lse
// (the partials in workspace).  fixed_len >= 0 gives one sequence's key count
// on the host instead of d_kv_len; causal_extra is DecodeArgs::causal_extra.
kvq_status decode_checked(const kvq_cache *k, const kvq_cache *v, const void *q, int q_dtype, int n_q, int n_heads,
                          float softmax_scale, const int32_t *d_kv_len, int fixed_len, int causal_extra,
                          int max_kv_len, int n_splits, float *out, float *out_lse, void *workspace, int32_t *d_err,
                          cudaStream_t cs);

cudaError_t launch_append(const AppendArgs &a, bool src_f16, cudaStream_t st);
cudaError_t launch_decode_simt(const DecodeArgs &a, int q_dtype, cudaStream_t st);
// Tensor-core path: head_dim 64/128/256, any K and V codec, any number of query
// rows per kv head (blocks of up to 32 rows, one CTA each).
bool decode_tc_supported(const DecodeArgs &a);
cudaError_t launch_decode_tc(const DecodeArgs &a, int q_dtype, cudaStream_t st);
// CTAs of the tensor-core decode kernel that fit on one SM for these caches and
// query rows per kv head; 0 if that kernel does not take them or no device answers.
int decode_ctas_per_sm(int k_codec, int v_codec, int head_dim, int rows_per_kv_head);
// The same kernel for V in Q4_G32, q8_0 and NVFP4 (translation units of their own).
cudaError_t launch_decode_tc_g32(const DecodeArgs &a, int q_dtype, cudaStream_t st);
int decode_tc_g32_ctas_per_sm(int k_codec, int head_dim, int n_tiles);
cudaError_t launch_decode_tc_q8v(const DecodeArgs &a, int q_dtype, cudaStream_t st);
int decode_tc_q8v_ctas_per_sm(int k_codec, int head_dim, int n_tiles);
cudaError_t launch_decode_tc_fp4v(const DecodeArgs &a, int q_dtype, cudaStream_t st);
int decode_tc_fp4v_ctas_per_sm(int k_codec, int head_dim, int n_tiles);
// Up to 8 query rows per kv head over Q4_G64 or q8_0 K and Q4_G64 V (head_dim 64/128/256):
// CTAs of warps that each own whole 16-token blocks (kvq_decode_warp.cu).
// decode_warp_shape: the shapes it takes (also for the split policy);
// decode_warp_takes: it runs these arguments.
bool decode_warp_shape(int k_codec, int v_codec, int head_dim, int rows_per_kv_head);
bool decode_warp_takes(const DecodeArgs &a);
int decode_warp_ctas_per_sm(int k_codec, int v_codec, int head_dim);
cudaError_t launch_decode_warp(const DecodeArgs &a, int q_dtype, cudaStream_t st);
// Prompt-chunk path on the fifth-generation tensor cores (tcgen05): blocks of
// 128 query rows per CTA, Q4_G64 K and V, head_dim 64/128/256,
// fp16 queries.  prefill_umma_shape: the shapes it is meant for (rows per kv
// head at least kUmmaMinRows); prefill_umma_takes: it runs these arguments.
constexpr int kUmmaMinRows = 64;
constexpr int kUmmaRowsPerCta = 128;
bool prefill_umma_shape(int k_codec, int v_codec, int head_dim, int rows_per_kv_head);
bool prefill_umma_takes(const DecodeArgs &a, int q_dtype);
int prefill_umma_ctas_per_sm(int k_codec, int v_codec, int head_dim);
cudaError_t launch_prefill_umma(const DecodeArgs &a, cudaStream_t st);
cudaError_t launch_merge(const float *po, const float *pl, int n_splits, int rows, int head_dim,
                         float *out, float *out_lse, cudaStream_t st);
cudaError_t launch_dequant(const Plane &p, int64_t n_rows, int head_dim, float *out, cudaStream_t st);

}  // namespace kvq
