// kvq_static.cu -- kvq_decode_attention_static: decode attention whose split
// scratch lives in a fixed device array owned by this library, for callers
// that cannot allocate device memory at the point where they decode.
//
// Who cannot allocate: code that enqueues work while a CUDA graph is being
// captured (cudaMalloc is not a stream operation and breaks or is refused by
// the capture), engines that hand all device memory to their own pool and
// forbid raw allocations, and latency-critical paths where an allocation's
// implicit device synchronisation is not acceptable.  Such callers still pass
// their inputs and outputs; only the scratch comes from here.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds KVQ_STATIC_SCRATCH_BYTES of it until the process exits.  Host
// code only sees a host-side stand-in for its name, so the device address is
// looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first call made there.
#include <cstdio>
#include <cstring>

#include "kvq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[KVQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

size_t kvq_static_scratch_bytes(void) { return (size_t)KVQ_STATIC_SCRATCH_BYTES; }

kvq_status kvq_decode_attention_static(const kvq_cache *k, const kvq_cache *v, const void *q, int32_t q_dtype,
                                       int32_t n_q, int32_t n_heads, float softmax_scale, const int32_t *d_kv_len,
                                       int32_t max_kv_len, int32_t n_splits, float *out, float *out_lse,
                                       int32_t *d_err, void *stream)
{
    // the scratch this call needs must fit the array; checked before any CUDA call
    if (k && v && n_heads > 0 && n_q > 0 && max_kv_len > 0 && n_splits >= 0) {
        const size_t need = kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, n_splits);
        if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "decode_static: this call needs %zu bytes of split scratch, the static array holds %zu; "
                     "use fewer splits or kvq_decode_attention with a caller-owned workspace",
                     need, (size_t)KVQ_STATIC_SCRATCH_BYTES);
            kvq::set_last_error(msg);
            return KVQ_EWORKSPACE;
        }
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        char msg[256];
        snprintf(msg, sizeof msg, "decode_static: no usable current device (%s)", cudaGetErrorString(e));
        kvq::set_last_error(msg);
        return KVQ_ECUDA;
    }
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "decode_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            kvq::set_last_error(msg);
            return KVQ_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    return kvq_decode_attention(k, v, q, q_dtype, n_q, n_heads, softmax_scale, d_kv_len, max_kv_len, n_splits, out,
                                out_lse, g_scratch_ptr[dev], (size_t)KVQ_STATIC_SCRATCH_BYTES, d_err, stream);
}

}  // extern "C"
