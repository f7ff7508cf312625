// kvq_selftest.cu -- kvq_selftest_bounded_wait: the failure path of the
// library's device waits, exercised on purpose.  One CTA waits, with the same
// bounded mbarrier wait the decode kernels use for their tile copies, on a
// barrier that nothing completes; the wait gives up after its cycle limit
// (~1 s), the kernel ORs KVQ_ERR_TIMEOUT into the caller's error word and
// returns.  Nothing traps and the context stays usable.
#include <cstdio>

#include "kvq_ptx.cuh"

namespace kvq {
namespace {

__global__ void bounded_wait_kernel(int32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);                 // one arrival expected; none is made
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait(b, 0) && err) atomicOr(err, KVQ_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_selftest_bounded_wait(int32_t *d_err, void *stream)
{
    if (!d_err) {
        kvq::set_last_error("selftest: d_err is NULL");
        return KVQ_EINVAL;
    }
    kvq::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d_err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "selftest launch: %s", cudaGetErrorString(e));
        kvq::set_last_error(msg);
        return KVQ_ECUDA;
    }
    return KVQ_OK;
}
