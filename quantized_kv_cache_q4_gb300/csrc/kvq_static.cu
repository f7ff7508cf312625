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
// looked up with cudaGetSymbolAddress, with the device current.  The address
// belongs to the CUDA context that loaded the module: it is kept per context
// (keyed by the driver's context ID, so a context torn down and created again
// -- e.g. after cudaDeviceReset -- is looked up afresh); where the context ID
// cannot be read, it is looked up on every call (a host-side query that
// allocates nothing).
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "kvq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[KVQ_STATIC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct CtxFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const CtxFns &ctx_fns()
{
    static const CtxFns fns = [] {
        CtxFns f;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
        return f;
    }();
    return fns;
}

// ID of the current context, 0 if it cannot be read.
unsigned long long current_ctx_id()
{
    const CtxFns &f = ctx_fns();
    if (!f.get_current || !f.get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (f.get_current(&c) != CUDA_SUCCESS || !c || f.get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

constexpr int kSlots = 64;
std::mutex g_mu;
unsigned long long g_ctx[kSlots] = {};
void *g_ptr[kSlots] = {};
int g_used = 0, g_next = 0;

// Device address of the scratch array in the current context.
cudaError_t scratch_address(void **out)
{
    const unsigned long long id = current_ctx_id();
    if (id != 0) {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < g_used; ++i)
            if (g_ctx[i] == id) {
                *out = g_ptr[i];
                return cudaSuccess;
            }
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    if (id != 0) {
        std::lock_guard<std::mutex> lock(g_mu);
        const int slot = g_used < kSlots ? g_used++ : (g_next++ % kSlots);
        g_ctx[slot] = id;
        g_ptr[slot] = p;
    }
    *out = p;
    return cudaSuccess;
}

kvq_status fail(kvq_status st, const char *msg)
{
    kvq::set_last_error(msg);
    return st;
}

}  // namespace

extern "C" {

size_t kvq_static_scratch_bytes(void) { return (size_t)KVQ_STATIC_SCRATCH_BYTES; }

kvq_status kvq_decode_attention_static(const kvq_cache *k, const kvq_cache *v, const void *q, int32_t q_dtype,
                                       int32_t n_q, int32_t n_heads, float softmax_scale, const int32_t *d_kv_len,
                                       int32_t max_kv_len, int32_t n_splits, float *out, float *out_lse,
                                       int32_t *d_err, void *stream)
{
    char msg[320];
    if (n_splits < 0 || n_splits > 4096) {
        snprintf(msg, sizeof msg, "decode_static: n_splits=%d outside [0, 4096]", n_splits);
        return fail(KVQ_EINVAL, msg);
    }
    // the scratch this call needs must fit the array; checked before anything
    // is launched.  With the default split count (0), the count is lowered to
    // the largest one whose scratch fits.
    if (k && v && n_heads > 0 && n_q > 0 && max_kv_len > 0) {
        int32_t s = n_splits;
        size_t need = kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, s);
        if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES && n_splits == 0) {
            s = kvq_decode_default_splits(k, v, n_heads, n_q, max_kv_len);
            while (s > 1 && kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, s) > (size_t)KVQ_STATIC_SCRATCH_BYTES)
                s = s * 7 / 8 < s - 1 ? s * 7 / 8 : s - 1;
            need = kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, s);
            n_splits = s;
        }
        if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES) {
            snprintf(msg, sizeof msg,
                     "decode_static: this call needs %zu bytes of split scratch, the static array holds %zu; "
                     "use fewer splits or kvq_decode_attention with a caller-owned workspace",
                     need, (size_t)KVQ_STATIC_SCRATCH_BYTES);
            return fail(KVQ_EWORKSPACE, msg);
        }
    }
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "decode_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return fail(KVQ_ECUDA, msg);
    }
    return kvq_decode_attention(k, v, q, q_dtype, n_q, n_heads, softmax_scale, d_kv_len, max_kv_len, n_splits, out,
                                out_lse, scratch, (size_t)KVQ_STATIC_SCRATCH_BYTES, d_err, stream);
}

}  // extern "C"
