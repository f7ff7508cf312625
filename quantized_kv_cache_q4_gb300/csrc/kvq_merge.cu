// kvq_merge.cu -- log-sum-exp merge of per-split partial attention results.
//
// softmax over a union of key ranges is the exp(lse)-weighted combination of
// the softmaxes over the parts: with M = max_s lse_s and w_s = exp(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s and lse = M + ln sum_s w_s.  Parts with
// lse = -inf (no visible key) carry no weight and their o is never used.
//
// The merge is latency-bound (the partials were just written, so they sit in
// L2): it is laid out for at most a round or two of loads per thread.  LPC
// consecutive lanes own one float4 column of one row; lane j of the group reads
// the lse and the float4 of splits j, j + LPC, ... four at a time (all issued
// before any is used), keeping a running maximum, and the group combines its
// (maximum, weight sum, weighted sum) with shuffles.  LPC grows with the split
// count (many splits: a warp per column; few splits, many rows: a lane per
// column) so that both shapes need few rounds and few CTAs.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kUnroll = 4;

template <int LPC>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const float *__restrict__ po, const float *__restrict__ pl, int n_splits, int rows, int D,
             float *__restrict__ out, float *__restrict__ out_lse)
{
    const int D4 = D / 4;
    const int sl = threadIdx.x % LPC;
    const int64_t item = (int64_t)blockIdx.x * (kMergeThreads / LPC) + threadIdx.x / LPC;
    const bool active = item < (int64_t)rows * D4;     // idle groups still take part in the shuffles
    const int row = active ? (int)(item / D4) : 0, col = active ? (int)(item % D4) : 0;
    pdl_wait();
    pdl_trigger();

    float M = -INFINITY, W = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = sl; active && s0 < n_splits; s0 += LPC * kUnroll) {
        float l[kUnroll];
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int s = s0 + u * LPC;
            l[u] = (s < n_splits) ? pl[(int64_t)s * rows + row] : -INFINITY;
            // loaded whether or not the part is empty (independent of the lse load);
            // an empty part's values are never used below
            v[u] = (s < n_splits) ? reinterpret_cast<const float4 *>(po + ((int64_t)s * rows + row) * D)[col]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mu = M;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) mu = fmaxf(mu, l[u]);
        if (mu == -INFINITY) continue;         // nothing but empty parts so far
        const float r = expf(M - mu);          // 0 when M is still -inf
        W *= r;
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        M = mu;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (l[u] == -INFINITY) continue;  // empty part: no weight, value never used
            const float w = expf(l[u] - M);
            W += w;
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
    }
    // combine the LPC lanes of the column: common maximum, rescaled sums
    float Mg = M;
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) Mg = fmaxf(Mg, __shfl_xor_sync(0xffffffffu, Mg, o));
    const float r = (M == -INFINITY) ? 0.0f : expf(M - Mg);
    W *= r;
    acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) {
        W += __shfl_xor_sync(0xffffffffu, W, o);
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (active && sl == 0) {
        float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mg != -INFINITY) {
            const float inv = 1.0f / W;
            res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        reinterpret_cast<float4 *>(out + (int64_t)row * D)[col] = res;
        if (col == 0 && out_lse) out_lse[row] = (Mg == -INFINITY) ? -INFINITY : Mg + logf(W);
    }
}

template <int LPC>
cudaError_t launch_lpc(const float *po, const float *pl, int n_splits, int rows, int D, float *out, float *out_lse,
                       cudaStream_t st)
{
    const int64_t items = (int64_t)rows * (D / 4);
    const dim3 grid((unsigned)ceil_div(items, kMergeThreads / LPC));
    // programmatic launch: the decode kernel releases it only after its main
    // loop, so its CTAs are placed on SMs that finishing decode CTAs free, and
    // the launch latency hides behind the decode's tail
    return launch_pdl(merge_kernel<LPC>, grid, dim3(kMergeThreads), 0, st, po, pl, n_splits, rows, D, out, out_lse);
}

}  // namespace

cudaError_t launch_merge(const float *po, const float *pl, int n_splits, int rows, int head_dim,
                         float *out, float *out_lse, cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    // lanes per column: enough that a lane loads at most half a round of
    // kUnroll splits (the merge is a chain of dependent L2 round trips: measured
    // on GB300, 37 splits x 24 rows take 15.2 us of the attention call with 32
    // lanes, 15.8 with 16, 17.7 with 8), fewer while that would take more than
    // about a quarter wave of threads
    static PerDevice pd;
    int dev = 0;
    int n_sm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        n_sm = per_device(pd, dev, [dev]() -> int {
            int v = 0;
            return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 0;
        });
    if (n_sm <= 0) n_sm = 152;
    int lpc = 1;
    while (lpc < 32 && lpc * kUnroll < 2 * n_splits) lpc *= 2;
    const int64_t items = (int64_t)rows * (head_dim / 4);
    while (lpc > 1 && items * lpc > (int64_t)n_sm * 512) lpc /= 2;
    switch (lpc) {
    case 1: return launch_lpc<1>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    case 2: return launch_lpc<2>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    case 4: return launch_lpc<4>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    case 8: return launch_lpc<8>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    case 16: return launch_lpc<16>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    default: return launch_lpc<32>(po, pl, n_splits, rows, head_dim, out, out_lse, st);
    }
}

}  // namespace kvq
