// kvq_append.cu -- quantize-on-append: new K/V rows are quantized to Q4_G64,
// Q4_G32, q8_0 or NVFP4 and written at their cache positions (den_llama.cpp,
// "What's in the fork": the set-rows / cpy-utils quantize path of the Q4_G64
// codec; the codec itself in "What this fork is": 4-bit signed codes sharing
// an fp16 scale per 64-value group; the NVFP4 KV type of the same section, read as
// NVIDIA's published NVFP4).
//
// One warp quantizes one (plane, sequence, new token, kv head) row.  Lane l
// owns the VPL = head_dim/32 consecutive values [l*VPL, (l+1)*VPL); a group of
// 64 (Q4_G64), 32 (Q4_G32, q8_0) or 16 (NVFP4) values is then group/VPL
// aligned lanes whose absmax is combined with xor-shuffles.  The arithmetic is
// the codec rule itself: scale = fp16_rne(absmax / qmax) via IEEE division
// (__fdiv_rn), saturated to 65504; code = clamp(rne(x / (float)scale)) via
// IEEE division and round-to-nearest-even conversion.  NVFP4: scale =
// E4M3(absmax / 6), code = E2M1(x / scale), the hardware's round-to-nearest-
// even saturating conversions, the code's sign bit set from the value's.  This
// TU must not be built with fast-math.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

template <int N>
__device__ __forceinline__ void load_vals(const float *p, float (&x)[N])
{
    static_assert(N % 2 == 0, "");
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            float4 f = *reinterpret_cast<const float4 *>(p + i);
            x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
        }
    } else {
        float2 f = *reinterpret_cast<const float2 *>(p);
        x[0] = f.x; x[1] = f.y;
    }
}

template <int N>
__device__ __forceinline__ void load_vals(const __half *p, float (&x)[N])
{
    if constexpr (N % 8 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 8) {
            uint4 u = *reinterpret_cast<const uint4 *>(p + i);
            const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __half22float2(h[j]);
                x[i + 2 * j] = f.x; x[i + 2 * j + 1] = f.y;
            }
        }
    } else if constexpr (N == 4) {
        uint2 u = *reinterpret_cast<const uint2 *>(p);
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
        float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
        __half2 h = *reinterpret_cast<const __half2 *>(p);
        float2 a = __half22float2(h);
        x[0] = a.x; x[1] = a.y;
    }
}

// Store N bytes held little-endian in `lo` (and `hi` for N == 16).
template <int N>
__device__ __forceinline__ void store_bytes(uint8_t *p, uint64_t lo, uint64_t hi)
{
    if constexpr (N == 16) {
        uint4 u;
        u.x = (uint32_t)lo; u.y = (uint32_t)(lo >> 32); u.z = (uint32_t)hi; u.w = (uint32_t)(hi >> 32);
        *reinterpret_cast<uint4 *>(p) = u;
    } else if constexpr (N == 8) {
        *reinterpret_cast<uint2 *>(p) = make_uint2((uint32_t)lo, (uint32_t)(lo >> 32));
    } else if constexpr (N == 4) {
        *reinterpret_cast<uint32_t *>(p) = (uint32_t)lo;
    } else if constexpr (N == 2) {
        *reinterpret_cast<uint16_t *>(p) = (uint16_t)lo;
    } else {
        *p = (uint8_t)lo;
    }
}

// Scale of a group from the lane-local absmax: combined over the LPG aligned
// lanes of the group, divided by qmax, rounded once to fp16, saturated.
template <int LPG>
__device__ __forceinline__ __half group_scale(float amax, float qmax)
{
#pragma unroll
    for (int off = 1; off < LPG; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __half h = __float2half_rn(__fdiv_rn(amax, qmax));
    if (__hisinf(h)) h = __ushort_as_half((unsigned short)0x7BFF);
    return h;
}

__device__ __forceinline__ int code_of(float x, float d, int qmin, int qmax)
{
    if (d == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(x, d));
    return q < qmin ? qmin : (q > qmax ? qmax : q);
}

// One row's share of a lane (VPL consecutive values) as 4-bit codes: the group
// scale from the absmax over the GS / VPL lanes of the group, then the codes
// packed two per byte (even value low nibble).
template <int VPL, int GS>
__device__ __forceinline__ void store_q4(const Plane &P, int64_t crow, int lane, const float (&x)[VPL], float amax)
{
    constexpr int D = VPL * 32;
    constexpr int LPG = GS / VPL;                      // lanes per group
    const __half hs = group_scale<LPG>(amax, 7.0f);
    const float d = __half2float(hs);
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        const uint64_t nib = (uint64_t)(code_of(x[v], d, -8, 7) & 0xF);
        if (v < 16) lo |= nib << (4 * v);
        else hi |= nib << (4 * (v - 16));
    }
    store_bytes<VPL / 2>(P.qs + crow * (D / 2) + lane * (VPL / 2), lo, hi);
    if (lane % LPG == 0) reinterpret_cast<__half *>(P.sc)[crow * (D / GS) + lane / LPG] = hs;
}

// NVFP4: blocks of 16 values (16 / VPL aligned lanes).  The block's absmax / 6
// (IEEE division) to E4M3 (cvt.rn.satfinite), then each value divided by the
// decoded scale (IEEE) to E2M1 (cvt.rn.satfinite), two codes per byte, the
// sign bits taken from the values so that a negative value rounding to 0 is
// -0 whatever the converter does with it; all codes 0 when the scale is 0.
template <int VPL>
__device__ __forceinline__ void store_fp4(const Plane &P, int64_t crow, int lane, const float (&x)[VPL], float amax)
{
    constexpr int D = VPL * 32;
    constexpr int LPG = 16 / VPL;
#pragma unroll
    for (int off = 1; off < LPG; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    unsigned short e16;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e16) : "f"(0.0f), "f"(__fdiv_rn(amax, 6.0f)));
    const uint32_t sb = e16 & 0xFFu;
    const float d = e4m3_to_float(sb);
    uint64_t lo = 0, hi = 0;
    if (d != 0.0f) {
#pragma unroll
        for (int v = 0; v < VPL; v += 2) {
            uint32_t b;
            asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
                : "=r"(b) : "f"(__fdiv_rn(x[v + 1], d)), "f"(__fdiv_rn(x[v], d)));
            b = (b & 0x77u) | (signbit(x[v]) ? 0x08u : 0u) | (signbit(x[v + 1]) ? 0x80u : 0u);
            if (v < 16) lo |= (uint64_t)b << (4 * v);
            else hi |= (uint64_t)b << (4 * (v - 16));
        }
    }
    store_bytes<VPL / 2>(P.qs + crow * (D / 2) + lane * (VPL / 2), lo, hi);
    if (lane % LPG == 0) P.sc[crow * (D / 16) + lane / LPG] = (uint8_t)sb;
}

template <int VPL, typename SrcT>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a)
{
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t per_plane = (int64_t)a.n_seq * a.n_new * a.n_kv_heads;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= per_plane * a.n_planes) return;
    const int pl = (int)(row / per_plane);
    const int64_t src_row = row - pl * per_plane;        // (s * n_new + i) * n_kv_heads + h
    const int h = (int)(src_row % a.n_kv_heads);
    const int64_t si = src_row / a.n_kv_heads;
    const int i = (int)(si % a.n_new);
    const int s = (int)(si / a.n_new);

    // the source row does not depend on the position: both loads in flight at once
    constexpr int D = VPL * 32;
    const SrcT *src = static_cast<const SrcT *>(pl ? a.src[1] : a.src[0]) + src_row * D + lane * VPL;
    float x[VPL];
    load_vals<VPL>(src, x);
    const int p0 = a.pos0[s];
    if (p0 < 0 || (int64_t)p0 + a.n_new > a.capacity) {
        if (lane == 0 && i == 0 && h == 0 && pl == 0 && a.err) atomicOr(a.err, KVQ_ERR_APPEND_POS);
        return;
    }
    float amax = 0.0f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) amax = fmaxf(amax, fabsf(x[v]));

    const Plane P = pl ? a.plane[1] : a.plane[0];   // no dynamic index into the parameter block
    const int64_t crow = ((int64_t)s * a.n_kv_heads + h) * a.capacity + p0 + i;
    if (P.codec == KVQ_CODEC_Q4_G64) {
        store_q4<VPL, 64>(P, crow, lane, x, amax);
    } else if (P.codec == KVQ_CODEC_Q4_G32) {
        store_q4<VPL, 32>(P, crow, lane, x, amax);
    } else if (P.codec == KVQ_CODEC_NVFP4) {
        store_fp4<VPL>(P, crow, lane, x, amax);
    } else {
        constexpr int LPG = 32 / VPL;
        const __half hs = group_scale<LPG>(amax, 127.0f);
        const float d = __half2float(hs);
        uint64_t lo = 0, hi = 0;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const uint64_t b = (uint64_t)(uint8_t)(int8_t)code_of(x[v], d, -127, 127);
            if (v < 8) lo |= b << (8 * v);
            else hi |= b << (8 * (v - 8));
        }
        store_bytes<VPL>(P.qs + crow * D + lane * VPL, lo, hi);
        if (lane % LPG == 0) reinterpret_cast<__half *>(P.sc)[crow * (D / 32) + lane / LPG] = hs;
    }
}

template <int VPL>
cudaError_t launch_append_vpl(const AppendArgs &a, bool f16, cudaStream_t st)
{
    const int64_t rows = (int64_t)a.n_planes * a.n_seq * a.n_new * a.n_kv_heads;
    const int warps = 8;
    const int64_t blocks = ceil_div(rows, warps);
    if (blocks == 0) return cudaSuccess;
    if (f16) return launch_pdl(append_kernel<VPL, __half>, dim3((unsigned)blocks), dim3(warps * 32), 0, st, a);
    return launch_pdl(append_kernel<VPL, float>, dim3((unsigned)blocks), dim3(warps * 32), 0, st, a);
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, bool src_f16, cudaStream_t st)
{
    switch (a.head_dim) {
    case 64: return launch_append_vpl<2>(a, src_f16, st);
    case 128: return launch_append_vpl<4>(a, src_f16, st);
    case 256: return launch_append_vpl<8>(a, src_f16, st);
    case 512: return launch_append_vpl<16>(a, src_f16, st);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Dequantization of whole rows to fp32 (scale * code), for inspection/tests.
// One thread per 8 consecutive values of a row.
// ---------------------------------------------------------------------------
namespace {
__global__ void dequant_kernel(Plane p, int64_t n_rows, int head_dim, float *out)
{
    const int per_row = head_dim / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_rows * per_row) return;
    const int64_t r = idx / per_row;
    const int v0 = (int)(idx % per_row) * 8;
    const int gs = group_size(p.codec);
    float *o = out + r * head_dim + v0;
    if (is_fp4(p.codec)) {
        const float d = e4m3_to_float(p.sc[r * (head_dim / 16) + v0 / 16]);
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p.qs + r * (head_dim / 2) + v0 / 2);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t h2 = e2m1x2_to_h2(w >> (8 * j));
            o[2 * j] = d * __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
            o[2 * j + 1] = d * __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
        }
        return;
    }
    const float d = __half2float(reinterpret_cast<const __half *>(p.sc)[r * (head_dim / gs) + v0 / gs]);
    if (is_q4(p.codec)) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p.qs + r * (head_dim / 2) + v0 / 2);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int c = (int)((w >> (4 * j)) & 0xF);
            o[j] = d * (float)(c >= 8 ? c - 16 : c);
        }
    } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(p.qs + r * head_dim + v0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int8_t c = (int8_t)(((j < 4 ? w.x : w.y) >> (8 * (j & 3))) & 0xFF);
            o[j] = d * (float)c;
        }
    }
}
}  // namespace

cudaError_t launch_dequant(const Plane &p, int64_t n_rows, int head_dim, float *out, cudaStream_t st)
{
    const int64_t n = n_rows * (head_dim / 8);
    if (n == 0) return cudaSuccess;
    dequant_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, st>>>(p, n_rows, head_dim, out);
    return cudaGetLastError();
}

}  // namespace kvq
