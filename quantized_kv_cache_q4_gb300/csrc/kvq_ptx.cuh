// kvq_ptx.cuh -- inline-PTX building blocks of the tensor-core decode kernels:
// mbarriers with bounded waits, TMA (2D tiled and 1D bulk) loads, ldmatrix /
// mma.sync, the signed-nibble and int8 unpack to exact fp16
// integers, the swizzled tile geometry and the tensor-map encoder.
#pragma once

#include <cuda.h>

#include "kvq_internal.cuh"

namespace kvq {
namespace ptx {

constexpr int kTile = 64;          // tokens per pipeline stage
constexpr long long kWaitCycles = 1LL << 31;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}


__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// L2 policy for data read once per call (the packed cache): evicted first, so
// the stream does not push out what the next kernels need (their code, the
// split partials, the query).
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}


__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = a * b + c with a separate accumulator input c
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d = (a & M) ^ X | 0x6400 per 16-bit half, with the mask/xor pattern folded into
// the two constant operands b, c (truth table 0xAC: b&c -> 1, b&~c -> ~a, ~b&c -> a).
__device__ __forceinline__ uint32_t lop3_ac(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xAC;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Eight signed 4-bit codes of a 32-bit word (nibble p = bits 4p..4p+3) as four
// fp16x2 integers with their bias left in, for operands whose bias is removed
// after the MMA: h[0] = (p0, p4), h[2] = (p2, p6) as 1032 + q (the even
// head_dim indices), h[1] = (p1, p5), h[3] = (p3, p7) as 1152 + 16 q (the odd
// ones).  One LOP3 per two values.
__device__ __forceinline__ void unpack_q4_biased(uint32_t w, uint32_t (&h)[4])
{
    const uint32_t w8 = w >> 8;
    h[0] = lop3_ac(w, 0x64086408u, 0x64076407u);
    h[1] = lop3_ac(w, 0x64806480u, 0x64706470u);
    h[2] = lop3_ac(w8, 0x64086408u, 0x64076407u);
    h[3] = lop3_ac(w8, 0x64806480u, 0x64706470u);
}

// int8 codes as 1152 + q (byte b becomes 0x64 : (b ^ 0x80)), pairs (b0, b1), (b2, b3).
__device__ __forceinline__ void unpack_q8_biased(uint32_t w, uint32_t (&h)[2])
{
    const uint32_t x = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(h[0]) : "r"(x), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7342;" : "=r"(h[1]) : "r"(x), "r"(0x64646464u));
}

// NG consecutive fp16 scales at p (2*NG bytes, naturally aligned) as floats, with
// the widest shared-memory load that fits.
template <int NG>
__device__ __forceinline__ void load_scales(const uint8_t *p, float (&out)[NG])
{
    if constexpr (NG == 1) {
        out[0] = __half2float(*reinterpret_cast<const __half *>(p));
    } else if constexpr (NG == 2) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(p));
        out[0] = f.x; out[1] = f.y;
    } else if constexpr (NG == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const float2 a = __half22float2(u32_as_h2(u.x)), b = __half22float2(u32_as_h2(u.y));
        out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    } else {
        static_assert(NG % 8 == 0, "");
#pragma unroll
        for (int k = 0; k < NG; k += 8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(p + 2 * k);
            const float2 a = __half22float2(u32_as_h2(u.x)), b = __half22float2(u32_as_h2(u.y));
            const float2 c = __half22float2(u32_as_h2(u.z)), d = __half22float2(u32_as_h2(u.w));
            out[k] = a.x; out[k + 1] = a.y; out[k + 2] = b.x; out[k + 3] = b.y;
            out[k + 4] = c.x; out[k + 5] = c.y; out[k + 6] = d.x; out[k + 7] = d.y;
        }
    }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Shared-memory layout of one codes tile: rows of BI bytes (the TMA box width,
// <= 128), NB boxes side by side for rows wider than 128 bytes, each box
// swizzled by TMA with a BI-byte span: the 16-byte chunk index is XORed with
// address bits 7.. (the row index modulo 8, 4 or 2).
template <int ROWB>
struct TileGeom {
    static constexpr int BI = ROWB < 128 ? ROWB : 128;
    static constexpr int NB = ROWB / BI;
    static constexpr int CPB = BI / 16;                  // chunks per box row
    static constexpr int BYTES = kTile * ROWB;
    __device__ static __forceinline__ uint32_t chunk_addr(uint32_t base, int t, int c)
    {
        const int box = c / CPB, cc = c % CPB;
        const uint32_t off = (uint32_t)(t * BI + cc * 16);
        const uint32_t phys = off ^ (((off >> 7) & (CPB - 1)) << 4);
        return base + (uint32_t)(box * kTile * BI) + phys;
    }
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }


// TMA descriptor of a codes plane [rows][row_bytes] with boxes of box_rows
// rows (encoded once per distinct argument set and kept; thread-safe).
bool make_codes_map(CUtensorMap *m, void *base, int row_bytes, int64_t rows, int box_rows);
bool tensor_maps_available();

}  // namespace ptx
}  // namespace kvq
