// kvq_decode_simt.cu -- generic split-K decode attention over a packed cache on
// the CUDA cores.  It serves every shape the library accepts (any head_dim in
// {64,128,256,512}, any number of query rows per kv head, any codec pair) and
// is the baseline the tensor-core kernel is checked against.
//
// What it computes (den_llama.cpp, "What's in the fork": the fattn-vec
// kernels over the Q4_G64 cache; "Results": 1 + 2 MTP draft tokens): for each
// (sequence s, kv head kh, split) the query rows of that kv head -- query
// token i of query head kh*G + j is row i*G + j -- attend to the split's
// tokens [lo, hi) intersected with the row's visible keys (kv_len - n_q + i +
// 1).  The result per row is either final (one split) or a partial normalised
// over the split plus its log-sum-exp, merged later by kvq_merge_splits.
//
// Layout of the work: grid (split, kv head, sequence), 4 warps.  Rows are
// processed 8 at a time.  A warp takes 32 tokens at a time: for q.k each lane
// owns one token and dequantizes its whole K row against the 8 query rows held
// in shared memory; the online softmax is reduced over the warp; for p.V each
// lane owns head_dim/32 consecutive output values and walks the 32 tokens.
// Scores are kept in log2 units (q pre-multiplied by softmax_scale*log2 e).
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kSimtWarps = 4;
constexpr int kRowsPerPass = 8;

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// The values of N consecutive codes starting at value index v0 of a row (v0 a
// multiple of N): the integer codes, or NVFP4's E2M1 values.
template <int CODEC, int N>
__device__ __forceinline__ void load_codes(const uint8_t *row, int v0, float (&c)[N])
{
    if constexpr (is_fp4(CODEC)) {
        const uint8_t *p = row + v0 / 2;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const uint32_t h2 = e2m1x2_to_h2(p[j]);
            c[2 * j] = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
            c[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
        }
    } else if constexpr (is_q4(CODEC)) {
        const uint8_t *p = row + v0 / 2;
        uint64_t w;
        if constexpr (N == 2) w = *p;
        else if constexpr (N == 4) w = *reinterpret_cast<const uint16_t *>(p);
        else if constexpr (N == 8) w = *reinterpret_cast<const uint32_t *>(p);
        else {
            uint2 u = *reinterpret_cast<const uint2 *>(p);
            w = (uint64_t)u.x | ((uint64_t)u.y << 32);
        }
#pragma unroll
        for (int j = 0; j < N; ++j) {
            int nib = (int)((w >> (4 * j)) & 0xF);
            c[j] = (float)(nib >= 8 ? nib - 16 : nib);
        }
    } else {
        const uint8_t *p = row + v0;
#pragma unroll
        for (int j = 0; j < N; ++j) c[j] = (float)(int8_t)p[j];
    }
}

template <typename QT>
__device__ __forceinline__ float load_q(const QT *p) { return (float)*p; }
template <>
__device__ __forceinline__ float load_q<__half>(const __half *p) { return __half2float(*p); }

template <int KC, int VC, int VPL, typename QT>
__global__ void __launch_bounds__(kSimtWarps * 32) decode_simt_kernel(DecodeArgs a)
{
    constexpr int D = VPL * 32;
    constexpr int KG = group_size(KC), VG = group_size(VC);
    constexpr int KRB = row_bytes(KC, D), VRB = row_bytes(VC, D);
    constexpr int RB = kRowsPerPass;

    __shared__ float qf[RB][D];
    __shared__ float pbuf[kSimtWarps][32][RB];
    __shared__ float cm[kSimtWarps][RB], cl[kSimtWarps][RB];
    __shared__ float obuf[RB][D];

    const int split = blockIdx.x, kh = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.n_heads / a.n_kv_heads;
    const int R = a.n_q * G;
    // no early trigger: a dependent merge launch starts once this grid ends
    pdl_wait();

    int len = a.fixed_len >= 0 ? a.fixed_len : a.kv_len[s];
    if (len < 0 || len > a.max_kv_len) {
        if (threadIdx.x == 0 && split == 0 && kh == 0 && a.err) atomicOr(a.err, KVQ_ERR_KV_LEN);
        len = len < 0 ? 0 : a.max_kv_len;
    }
    int lo, hi;
    split_range(len, a.n_splits, split, lo, hi);

    const int64_t plane_row = ((int64_t)s * a.n_kv_heads + kh) * a.capacity;
    const uint8_t *kqs = a.k.qs + plane_row * KRB;
    constexpr int KSR = scale_row_bytes(KC, D), VSR = scale_row_bytes(VC, D);
    const uint8_t *ksc = a.k.sc + plane_row * KSR;
    const uint8_t *vqs = a.v.qs + plane_row * VRB;
    const uint8_t *vsc = a.v.sc + plane_row * VSR;
    const QT *q = static_cast<const QT *>(a.q);
    const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;

    for (int rb0 = 0; rb0 < R; rb0 += RB) {
        const int nr = min(RB, R - rb0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < RB * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            float val = 0.0f;
            if (r < nr) {
                const int row = rb0 + r, i = row / G, j = row % G;
                val = load_q(q + (((int64_t)s * a.n_q + i) * a.n_heads + kh * G + j) * D + d) * a.scale_log2;
            }
            qf[r][d] = val;
        }
        __syncthreads();

        int nvis[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int i = (rb0 + r) / G;
            nvis[r] = (r < nr) ? len + a.causal_extra - a.n_q + i + 1 : 0;
        }
        float m[RB], l[RB], o[RB][VPL];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.0f;
#pragma unroll
            for (int v = 0; v < VPL; ++v) o[r][v] = 0.0f;
        }

        for (int tb = lo + warp * 32; tb < hi; tb += kSimtWarps * 32) {
            const int t = tb + lane;
            const bool valid = t < hi;
            float acc[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) acc[r] = 0.0f;
            if (valid) {
                const uint8_t *krow = kqs + (int64_t)t * KRB;
#pragma unroll 1
                for (int g = 0; g < D / KG; ++g) {
                    const float dsc = load_scale<KC>(ksc + (int64_t)t * KSR, g);
                    float part[RB];
#pragma unroll
                    for (int r = 0; r < RB; ++r) part[r] = 0.0f;
#pragma unroll 1
                    for (int v0 = g * KG; v0 < (g + 1) * KG; v0 += 8) {
                        float c[8];
                        load_codes<KC, 8>(krow, v0, c);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const float cf = c[jj];
#pragma unroll
                            for (int r = 0; r < RB; ++r) part[r] = fmaf(qf[r][v0 + jj], cf, part[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < RB; ++r) acc[r] = fmaf(dsc, part[r], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float z = (valid && t < nvis[r]) ? acc[r] : -INFINITY;
                const float mn = fmaxf(m[r], warp_max(z));
                const float corr = (mn == -INFINITY) ? 1.0f : exp2f(m[r] - mn);
                const float p = (z == -INFINITY) ? 0.0f : exp2f(z - mn);
                l[r] = l[r] * corr + warp_sum(p);
#pragma unroll
                for (int v = 0; v < VPL; ++v) o[r][v] *= corr;
                m[r] = mn;
                pbuf[warp][lane][r] = p;
            }
            __syncwarp();
            const int nt = min(32, hi - tb);
#pragma unroll 1
            for (int j = 0; j < nt; ++j) {
                const int tj = tb + j;
                float c[VPL];
                load_codes<VC, VPL>(vqs + (int64_t)tj * VRB, lane * VPL, c);
                const float dsc = load_scale<VC>(vsc + (int64_t)tj * VSR, (lane * VPL) / VG);
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float p = pbuf[warp][j][r];
#pragma unroll
                    for (int v = 0; v < VPL; ++v) o[r][v] = fmaf(p, dsc * c[v], o[r][v]);
                }
            }
            __syncwarp();
        }

        // combine the four warps' (m, l, o) of each row
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < RB; ++r) { cm[warp][r] = m[r]; cl[warp][r] = l[r]; }
        }
        for (int idx = threadIdx.x; idx < RB * D; idx += blockDim.x) obuf[idx / D][idx % D] = 0.0f;
        __syncthreads();
        float f[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float M = -INFINITY;
            for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, cm[w][r]);
            float L = 0.0f;
            for (int w = 0; w < kSimtWarps; ++w)
                if (cm[w][r] != -INFINITY) L += cl[w][r] * exp2f(cm[w][r] - M);
            f[r] = (m[r] == -INFINITY || L == 0.0f) ? 0.0f : exp2f(m[r] - M) / L;
        }
        for (int w = 0; w < kSimtWarps; ++w) {
            if (warp == w) {
#pragma unroll
                for (int r = 0; r < RB; ++r)
#pragma unroll
                    for (int v = 0; v < VPL; ++v) obuf[r][lane * VPL + v] += f[r] * o[r][v];
            }
            __syncthreads();
        }
        for (int idx = threadIdx.x; idx < nr * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            const int row = rb0 + r, i = row / G, j = row % G;
            const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + j;
            if (a.n_splits == 1) a.out[orow * D + d] = obuf[r][d];
            else a.part_o[((int64_t)split * rows_total + orow) * D + d] = obuf[r][d];
        }
        if (threadIdx.x < nr) {
            const int r = threadIdx.x;
            float M = -INFINITY, L = 0.0f;
            for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, cm[w][r]);
            for (int w = 0; w < kSimtWarps; ++w)
                if (cm[w][r] != -INFINITY) L += cl[w][r] * exp2f(cm[w][r] - M);
            const float lse = (L > 0.0f) ? (M + log2f(L)) * kLn2 : -INFINITY;
            const int row = rb0 + r, i = row / G, j = row % G;
            const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + j;
            if (a.n_splits == 1) { if (a.out_lse) a.out_lse[orow] = lse; }
            else a.part_lse[(int64_t)split * rows_total + orow] = lse;
        }
    }
}

template <int KC, int VC, int VPL>
cudaError_t launch3(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    dim3 grid(a.n_splits, a.n_kv_heads, a.n_seq);
    if (q_dtype == KVQ_F16) return launch_pdl(decode_simt_kernel<KC, VC, VPL, __half>, grid, dim3(kSimtWarps * 32), 0, st, a);
    return launch_pdl(decode_simt_kernel<KC, VC, VPL, float>, grid, dim3(kSimtWarps * 32), 0, st, a);
}

template <int KC, int VC>
cudaError_t launch2(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    switch (a.head_dim) {
    case 64: return launch3<KC, VC, 2>(a, q_dtype, st);
    case 128: return launch3<KC, VC, 4>(a, q_dtype, st);
    case 256: return launch3<KC, VC, 8>(a, q_dtype, st);
    case 512: return launch3<KC, VC, 16>(a, q_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int KC>
cudaError_t launch_v(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    switch (a.v.codec) {
    case KVQ_CODEC_Q4_G64: return launch2<KC, KVQ_CODEC_Q4_G64>(a, q_dtype, st);
    case KVQ_CODEC_Q8_0: return launch2<KC, KVQ_CODEC_Q8_0>(a, q_dtype, st);
    case KVQ_CODEC_Q4_G32: return launch2<KC, KVQ_CODEC_Q4_G32>(a, q_dtype, st);
    case KVQ_CODEC_NVFP4: return launch2<KC, KVQ_CODEC_NVFP4>(a, q_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    switch (a.k.codec) {
    case KVQ_CODEC_Q4_G64: return launch_v<KVQ_CODEC_Q4_G64>(a, q_dtype, st);
    case KVQ_CODEC_Q8_0: return launch_v<KVQ_CODEC_Q8_0>(a, q_dtype, st);
    case KVQ_CODEC_Q4_G32: return launch_v<KVQ_CODEC_Q4_G32>(a, q_dtype, st);
    case KVQ_CODEC_NVFP4: return launch_v<KVQ_CODEC_NVFP4>(a, q_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq
