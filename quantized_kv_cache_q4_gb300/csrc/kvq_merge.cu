// kvq_merge.cu -- log-sum-exp merge of per-split partial attention results.
//
// softmax over a union of key ranges is the exp(lse)-weighted combination of
// the softmaxes over the parts: with M = max_s lse_s and w_s = exp(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s and lse = M + ln sum_s w_s.  Parts with
// lse = -inf (no visible key) carry no weight and their o is never used.
//
// The merge is latency-bound (a few KB per row, straight after the decode
// kernel wrote them), so it is laid out for one round of loads: a block of
// 256 threads covers 16 float4 columns of one row, 16 threads per column, and
// thread j of a column reads the lse and the float4 of splits j, j+16, ...
// together, keeping a running maximum.  The 16 lanes of a column then combine
// their (maximum, weight sum, weighted sum) with shuffles; there is no block
// barrier.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kLanesPerCol = 16;                          // split lanes per float4 column
constexpr int kMergeCols = kMergeThreads / kLanesPerCol;  // float4 columns per block
constexpr int kUnroll = 4;

__device__ __forceinline__ float group_max(float x)
{
#pragma unroll
    for (int o = 1; o < kLanesPerCol; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float group_sum(float x)
{
#pragma unroll
    for (int o = 1; o < kLanesPerCol; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const float *__restrict__ po, const float *__restrict__ pl, int n_splits, int rows, int D,
             float *__restrict__ out, float *__restrict__ out_lse)
{
    const int row = blockIdx.x;
    const int sl = threadIdx.x % kLanesPerCol;
    const int col = blockIdx.y * kMergeCols + threadIdx.x / kLanesPerCol;   // float4 column
    const int D4 = D / 4;
    const bool has_col = col < D4;
    pdl_wait();
    pdl_trigger();

    // one pass over this lane's splits, loading lse and values together and
    // keeping a running maximum (weights relative to it, rescaled when it grows)
    float M = -INFINITY, W = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = sl; s0 < n_splits; s0 += kLanesPerCol * kUnroll) {
        float l[kUnroll];
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int s = s0 + u * kLanesPerCol;
            l[u] = (s < n_splits) ? pl[(int64_t)s * rows + row] : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int s = s0 + u * kLanesPerCol;
            // loaded whether or not the part is empty (independent of the lse load);
            // an empty part's values are never used below
            v[u] = (s < n_splits && has_col)
                       ? reinterpret_cast<const float4 *>(po + ((int64_t)s * rows + row) * D)[col]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mu = M;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) mu = fmaxf(mu, l[u]);
        if (mu == -INFINITY) continue;                 // nothing but empty parts so far
        const float r = expf(M - mu);                  // 0 when M is still -inf
        W *= r;
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        M = mu;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (l[u] == -INFINITY) continue;          // empty part: no weight, value never used
            const float w = expf(l[u] - M);
            W += w;
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
    }
    // combine the 16 lanes of the column: common maximum, rescaled sums
    const float Mg = group_max(M);
    const float r = (M == -INFINITY) ? 0.0f : expf(M - Mg);
    W = group_sum(W * r);
    acc.x = group_sum(acc.x * r);
    acc.y = group_sum(acc.y * r);
    acc.z = group_sum(acc.z * r);
    acc.w = group_sum(acc.w * r);
    M = Mg;
    if (sl == 0 && has_col) {
        float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            const float inv = 1.0f / W;
            res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        reinterpret_cast<float4 *>(out + (int64_t)row * D)[col] = res;
        if (col == 0 && out_lse) out_lse[row] = (M == -INFINITY) ? -INFINITY : M + logf(W);
    }
}

}  // namespace

cudaError_t launch_merge(const float *po, const float *pl, int n_splits, int rows, int head_dim,
                         float *out, float *out_lse, cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)rows, (unsigned)ceil_div(head_dim / 4, kMergeCols));
    // programmatic launch: the decode kernel releases it only after its main
    // loop, so its CTAs are placed on SMs that finishing decode CTAs free, and
    // the launch latency hides behind the decode's tail
    return launch_pdl(merge_kernel, grid, dim3(kMergeThreads), 0, st, po, pl, n_splits, rows, head_dim, out, out_lse);
}

}  // namespace kvq
