// kvq_merge.cu -- log-sum-exp merge of per-split partial attention results.
//
// softmax over a union of key ranges is the exp(lse)-weighted combination of
// the softmaxes over the parts: with M = max_s lse_s and w_s = exp(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s and lse = M + ln sum_s w_s.  Parts with
// lse = -inf (no visible key) carry no weight and their o is never read.
//
// Grid (row, block of 16 float4 columns).  A block first turns the row's
// n_splits lse values into weights in shared memory, then each thread
// accumulates one float4 column over a strided subset of the splits (16
// subsets); the subsets are summed in shared memory.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeCols = 16;                  // float4 columns per block

__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const float *__restrict__ po, const float *__restrict__ pl, int n_splits, int rows, int D,
             float *__restrict__ out, float *__restrict__ out_lse)
{
    extern __shared__ float sh[];               // w[n_splits], then reduction scratch
    float *w = sh;
    float *red = sh + ((n_splits + 3) & ~3);   // [kMergeThreads] float4, 16-byte aligned
    __shared__ float s_stat[2];
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();

    float mx = -INFINITY;
    for (int s = tid; s < n_splits; s += kMergeThreads) mx = fmaxf(mx, pl[(int64_t)s * rows + row]);
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = -INFINITY;
        for (int i = 0; i < kMergeThreads / 32; ++i) m = fmaxf(m, red[i]);
        s_stat[0] = m;
    }
    __syncthreads();
    const float M = s_stat[0];
    float sum = 0.0f;
    for (int s = tid; s < n_splits; s += kMergeThreads) {
        const float l = pl[(int64_t)s * rows + row];
        const float wt = (l == -INFINITY) ? 0.0f : expf(l - M);
        w[s] = wt;
        sum += wt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    if (tid == 0) {
        float t = 0.0f;
        for (int i = 0; i < kMergeThreads / 32; ++i) t += red[i];
        s_stat[1] = t;
    }
    __syncthreads();
    const float W = s_stat[1];
    const int D4 = D / 4;
    const int cb = blockIdx.y * kMergeCols;           // first float4 column of this block
    if (M == -INFINITY) {
        for (int d = cb * 4 + tid; d < min(D, (cb + kMergeCols) * 4); d += kMergeThreads) out[(int64_t)row * D + d] = 0.0f;
        if (tid == 0 && blockIdx.y == 0 && out_lse) out_lse[row] = -INFINITY;
        return;
    }
    const float inv = 1.0f / W;
    {
        const int c0 = cb;
        const int ncol = min(kMergeCols, D4 - c0);
        const int lanes = max(1, kMergeThreads / ncol);      // split-lanes per column
        const int col = tid % ncol, sl = tid / ncol;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (sl < lanes) {
#pragma unroll 4
            for (int s = sl; s < n_splits; s += lanes) {
                const float wt = w[s];
                if (wt == 0.0f) continue;
                const float4 v = reinterpret_cast<const float4 *>(po + ((int64_t)s * rows + row) * D)[c0 + col];
                acc.x = fmaf(wt, v.x, acc.x); acc.y = fmaf(wt, v.y, acc.y);
                acc.z = fmaf(wt, v.z, acc.z); acc.w = fmaf(wt, v.w, acc.w);
            }
        }
        float4 *r4 = reinterpret_cast<float4 *>(red);
        __syncthreads();
        r4[tid] = acc;
        __syncthreads();
        if (tid < ncol) {
            float4 t = r4[tid];
            for (int k = 1; k < lanes; ++k) {
                const float4 u = r4[k * ncol + tid];
                t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
            }
            t.x *= inv; t.y *= inv; t.z *= inv; t.w *= inv;
            reinterpret_cast<float4 *>(out + (int64_t)row * D)[c0 + tid] = t;
        }
    }
    if (tid == 0 && blockIdx.y == 0 && out_lse) out_lse[row] = M + logf(W);
}

}  // namespace

cudaError_t launch_merge(const float *po, const float *pl, int n_splits, int rows, int head_dim,
                         float *out, float *out_lse, cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    const size_t smem = (size_t)((n_splits + 3) & ~3) * sizeof(float) + (size_t)kMergeThreads * sizeof(float4);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((unsigned)rows, (unsigned)ceil_div(head_dim / 4, kMergeCols));
    return launch_pdl(merge_kernel, grid, dim3(kMergeThreads), smem, st, po, pl, n_splits, rows, head_dim, out,
                      out_lse);
}

}  // namespace kvq
