// kvq_decode_common.cuh -- pieces the two tensor-core decode kernels share:
// the head_dim order in which the packed-code unpack delivers values (and the
// matching permuted, swizzled fp16 copy of the query rows with the K-bias
// terms), and the code-to-fp16 conversions of K and V operands.
#pragma once

#include "kvq_ptx.cuh"

namespace kvq {
using namespace ptx;
namespace {

// head_dim index fed by k-position kp (0..15) of k-step ks, in the order the K
// unpack delivers values (Q4_G64: pairs (d, d + 4) of a 4-byte piece; q8_0 and
// NVFP4: pairs (d, d + 1)).
template <int KC>
__device__ __forceinline__ int kpos_to_d(int ks, int kp)
{
    const int hi = kp >> 3, t = (kp & 7) >> 1, h = kp & 1;
    if constexpr (KC == KVQ_CODEC_Q4_G64) return 64 * (ks >> 2) + 32 * hi + 8 * t + (ks & 3) + 4 * h;
    // Q4_G32: both k-steps of a group come from its one 16-byte chunk (nibble
    // pairs 2 sub / 2 sub + 1 for the two k halves)
    else if constexpr (KC == KVQ_CODEC_Q4_G32) return 32 * (ks >> 1) + 8 * t + 2 * (ks & 1) + hi + 4 * h;
    // NVFP4: byte e of a 4-byte piece converts to the pair (2e, 2e + 1)
    else if constexpr (KC == KVQ_CODEC_NVFP4) return 64 * (ks >> 2) + 32 * hi + 8 * t + 2 * (ks & 3) + h;
    else return 32 * (ks >> 1) + 16 * hi + 4 * t + 2 * (ks & 1) + h;
}


// byte offset of 16-byte chunk c of row n of the permuted query copy (D halves a row)
template <int D>
__device__ __forceinline__ uint32_t qp_chunk_off(int n, int c)
{
    return (uint32_t)(n * D * 2 + ((c ^ (n & 7)) << 4));
}

// Nibble pair e (0..3) of a code word as fp16x2 with its bias left in: pair e
// holds nibbles e and e + 4 (the order the ldmatrix.trans fragment pairs two
// tokens in), as 1032 + q for even e and 1152 + 16 q for odd e.
__device__ __forceinline__ uint32_t q4_pair_biased(uint32_t w, int e)
{
    const uint32_t x = (e & 2) ? (w >> 8) : w;
    return (e & 1) ? lop3_ac(x, 0x64806480u, 0x64706470u) : lop3_ac(x, 0x64086408u, 0x64076407u);
}

// The same pair as fp16 subnormals: (q + 8) * 2^-24 for even e, 16 (q + 8) *
// 2^-24 for odd e (the nibble with its sign bit flipped is the significand;
// one LOP3, no exponent bits).
__device__ __forceinline__ uint32_t q4_pair_sub(uint32_t w, int e)
{
    const uint32_t x = (e & 2) ? (w >> 8) : w;
    return (e & 1) ? lop3_ac(x, 0x00800080u, 0x00700070u) : lop3_ac(x, 0x00080008u, 0x00070007u);
}

// q8_0 V after ldmatrix.trans: a word holds head_dim bytes (d, d + 1) of two
// tokens, [t0 d, t0 d+1, t1 d, t1 d+1]; the A fragment wants (t0, t1) at one d.
// As fp16 subnormals (q + 128) 2^-24: even d = (w ^ 0x80 per byte) & 0x00FF00FF
// (one LOP3, 0x28 = (a ^ b) & c), odd d the same on bytes 1, 3 moved down.
__device__ __forceinline__ void q8_pairs_sub(uint32_t w, uint32_t &ev, uint32_t &od)
{
    uint32_t hi;
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(ev) : "r"(w), "r"(0x00800080u), "r"(0x00FF00FFu));
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(hi) : "r"(w), "r"(0x80008000u), "r"(0xFF00FF00u));
    od = hi >> 8;
}

// The same pairs without offset: q exactly (1152 + q from the exponent byte
// 0x64, then an exact fp16 subtraction of 1152 = 0x6480).
__device__ __forceinline__ void q8_pairs(uint32_t w, uint32_t &ev, uint32_t &od)
{
    const uint32_t x = w ^ 0x80808080u;
    uint32_t e, o;
    asm("prmt.b32 %0, %1, %2, 0x4240;" : "=r"(e) : "r"(x), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4341;" : "=r"(o) : "r"(x), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(ev) : "r"(e), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(od) : "r"(o), "r"(0x64806480u));
}

// NVFP4 K after ldmatrix: the 4 bytes of a word hold head_dim values
// (2e, 2e + 1) of one token in byte e; each becomes an fp16x2 by the hardware
// E2M1 conversion, multiplied (exactly) by the block's scale pair.
__device__ __forceinline__ uint32_t fp4_byte_h2(uint32_t w, int e, uint32_t s2)
{
    const uint32_t h = e2m1x2_to_h2(w >> (8 * e));
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(s2));
    return r;
}

// An E4M3 byte (bits 0-7 of b) as the fp16x2 pair (s, s).
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t b)
{
    uint32_t d, h2;
    asm("prmt.b32 %0, %1, 0, 0x0000;" : "=r"(d) : "r"(b));
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(d));
    return h2;
}

// NVFP4 V after ldmatrix.trans: a word holds nibbles e = 0..3 (head_dim
// values 4 gid + e) of token t0 in bits 0-15 and of t1 in bits 16-31; pair e
// gathers nibble e of both into one byte (0xE4 = (a & c) | (b & ~c)), the
// hardware E2M1 conversion makes it (t0, t1) as fp16x2, times the tokens'
// scales s2.
__device__ __forceinline__ uint32_t fp4_pair(uint32_t w, int e, uint32_t s2)
{
    const uint32_t lo = w >> (4 * e), hi = w >> (12 + 4 * e);
    uint32_t b, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(b) : "r"(lo), "r"(hi), "r"(0x0000000Fu));
    const uint32_t h = e2m1x2_to_h2(b);
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(s2));
    return r;
}

// The pair without any offset: q for even e, 16 q for odd e (an exact fp16
// subtraction of 1032 = 0x6408 or 1152 = 0x6480 from the biased form).
__device__ __forceinline__ uint32_t q4_pair(uint32_t w, int e)
{
    const uint32_t b = q4_pair_biased(w, e);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(b), "r"((e & 1) ? 0x64806480u : 0x64086408u));
    return r;
}

// The query rows as fp16, head_dim permuted to the K-unpack order and swizzled
// for ldmatrix ([ROWS][D], rows >= R zero); with Q4_G64 K the odd head_dim
// indices are divided by 16 (exact for normal values) because their codes
// arrive as 1152 + 16 q.  Each thread builds whole 16-byte chunks (8
// k-positions of one k-step, so of one K group); the CPG chunks of a group sit
// in consecutive lanes, whose shuffle sum gives minus the group's bias term
// sum_d bias(d) q(d) (bias 1032 at even, 1152 at odd d for Q4_G64; 1152 for
// q8_0) in kb_s[group][row].  An fp32 query is split into fp16 parts,
// value = hi + lo: hi goes to qp, lo (the fp32 remainder rounded to fp16) to
// qp_lo in the same layout, and the bias terms cover hi + lo; the K product
// then takes one MMA per part, so the query keeps about 22 bits instead of 11.
template <int KC, int D, int ROWS, int NTH, typename QT>
__device__ __forceinline__ void prep_query(const QT *qst, uint8_t *qp, uint8_t *qp_lo, float *kb_s, int R, bool ok)
{
    constexpr bool SPLIT = sizeof(QT) == 4;
    constexpr int CPR = D / 8;                     // chunks per row
    constexpr int CPG = (is_fp4(KC) ? 64 : group_size(KC)) / 8;   // chunks per K accumulation group
    for (int ci = threadIdx.x; ci < ROWS * CPR; ci += NTH) {   // whole warps per step
        const int n = ci / CPR, c = ci % CPR;
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int kg = 8 * c + j;
            const int d = kpos_to_d<KC>(kg >> 4, kg & 15);
            x[j] = 0.0f;
            if (n < R && ok) {
                if constexpr (sizeof(QT) == 2) x[j] = __half2float(qst[n * D + d]);
                else x[j] = qst[n * D + d];
            }
            if constexpr (is_q4(KC))
                if (d & 1) x[j] *= 0.0625f;
        }
        uint32_t hw[4], lw[4];
        float b = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hw[j] = pack_f16x2(x[2 * j], x[2 * j + 1]);
            float2 hf = __half22float2(u32_as_h2(hw[j]));
            if constexpr (SPLIT) {
                lw[j] = pack_f16x2(x[2 * j] - hf.x, x[2 * j + 1] - hf.y);   // exact fp32 remainders, rounded
                const float2 lf = __half22float2(u32_as_h2(lw[j]));
                hf.x += lf.x;
                hf.y += lf.y;
            }
            // Q4_G64: j-th pair is (d, d + 4) with d's parity that of the k-step
            const int kg = 8 * c + 2 * j;
            const bool even = is_q4(KC) && ((kpos_to_d<KC>(kg >> 4, kg & 15) & 1) == 0);
            if constexpr (!is_fp4(KC)) b = fmaf(even ? 1032.0f : 1152.0f, hf.x + hf.y, b);
        }
        *reinterpret_cast<uint4 *>(qp + qp_chunk_off<D>(n, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if constexpr (SPLIT)
            *reinterpret_cast<uint4 *>(qp_lo + qp_chunk_off<D>(n, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
#pragma unroll
        for (int off = 1; off < CPG; off <<= 1) b += __shfl_xor_sync(0xffffffffu, b, off);
        if (c % CPG == 0) kb_s[(c / CPG) * ROWS + n] = -b;
    }
}

}  // namespace
}  // namespace kvq
