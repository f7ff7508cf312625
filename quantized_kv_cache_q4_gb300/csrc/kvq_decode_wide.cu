// kvq_decode_wide.cu -- split-K decode attention on the tensor cores for 9..32
// query rows per kv head: the MTP verify shape, where 1 + 2 draft tokens of a
// sequence meet a GQA group of 6 (18 rows; den_llama.cpp, "Results": MTP
// n-max 2).  Same result as the other decode kernels.
//
// With 24-32 rows an accumulator of the whole head_dim per warp would not fit
// in registers, so a 64-token tile is worked in two phases by the four
// consumer warps of a CTA:
//   A. warp w computes S^T = K Q^T for tokens [16w, 16w+16) of the tile and
//      all NT = ceil(rows/8) n-tiles (K unpacked once, Q B-fragments loaded
//      with ldmatrix from a swizzled, head_dim-permuted copy in shared
//      memory).  The per-row tile maximum is reduced over the CTA through
//      shared memory behind a named barrier, so every warp holds the same
//      running maximum; p = 2^(s - m) is written to shared memory.
//   B. warp w owns a quarter of head_dim (one 64-value V group at D = 256)
//      and accumulates O^T for all rows over the tile's 64 tokens, folding the
//      V scale of each token into p (P' rounded once to fp16).
// Because the four warps share the running maximum, their outputs need no
// rescaling at the end: each warp writes its slice of head_dim divided by the
// row sum.
//
// The producer warp, the TMA ring, the unpack and the bounded waits are those
// of the narrow kernel (kvq_ptx.cuh).
#include "kvq_ptx.cuh"

namespace kvq {
using namespace ptx;
namespace {

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

template <int KC, int D, int NT>
struct WideCfg {
    static constexpr int KRB = row_bytes(KC, D), VRB = D / 2;
    static constexpr int KSB = 2 * scales_per_row(KC, D), VSB = 2 * (D / 64);
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = align_up(kTile * KRB, 1024);
    static constexpr int KS_OFF = V_OFF + align_up(kTile * VRB, 1024);
    static constexpr int VS_OFF = KS_OFF + align_up(kTile * KSB, 128);
    static constexpr int STAGE = align_up(VS_OFF + kTile * VSB, 1024);
    static constexpr int ROWS = 32;                               // Q rows kept (zero past R)
    static constexpr int PS = NT * 8 + 4;                         // p row stride (floats), bank spread
    static constexpr int Q_OFF = kStages * STAGE;                 // fp16 [32][D], swizzled
    static constexpr int P_OFF = Q_OFF + ROWS * D * 2;            // fp32 [64][PS]
    static constexpr int RED_OFF = P_OFF + align_up(kTile * PS * 4, 16);   // fp32 [4][32] max, [4][32] sum
    static constexpr int BAR_OFF = RED_OFF + 2 * kConsumerWarps * 32 * 4;
    static constexpr int SMEM = BAR_OFF + 2 * kStages * 8 + 1024;
    static constexpr int MT_PER_WARP = 4 * (D / 64) / kConsumerWarps;   // 16-wide d tiles per warp
};

// head_dim index that k-position kp (0..15) of k-step ks feeds, matching the
// order in which the K unpack delivers values (see the narrow kernel).
template <int KC>
__device__ __forceinline__ int kpos_to_d(int ks, int kp)
{
    const int hi = kp >> 3, t = (kp & 7) >> 1, h = kp & 1;
    if constexpr (KC == KVQ_CODEC_Q4_G64) {
        const int g = ks >> 2, st = ks & 3;
        return 64 * g + 32 * hi + 8 * t + st + 4 * h;
    } else {
        const int g = ks >> 1, st = ks & 1;
        return 32 * g + 16 * hi + 4 * t + 2 * st + h;
    }
}

// byte offset of 16-byte chunk c of row n in the swizzled Q copy (row = D halves)
template <int D>
__device__ __forceinline__ uint32_t q_chunk_off(int n, int c)
{
    return (uint32_t)(n * D * 2 + ((c ^ (n & 7)) << 4));
}

template <int KC, int D, int NT, typename QT>
__global__ void __launch_bounds__(kThreads, 2)
decode_wide_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv)
{
    using C = WideCfg<KC, D, NT>;
    using KG = TileGeom<C::KRB>;
    using VG = TileGeom<C::VRB>;
    constexpr int NGK = D / group_size(KC);
    constexpr int KSTEP_PER_G = group_size(KC) / 16;
    constexpr int MTW = C::MT_PER_WARP;                  // 4 at D=256, 2 at D=128

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = smem + C::Q_OFF;
    float *p_s = reinterpret_cast<float *>(smem + C::P_OFF);
    float *red_m = reinterpret_cast<float *>(smem + C::RED_OFF);      // [warps][32]
    float *red_l = red_m + kConsumerWarps * 32;                        // [warps][32]
    const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);
    const uint32_t bar_empty = bar_full + kStages * 8;
    __shared__ volatile int s_timeout;

    const int split = blockIdx.x, kh = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int G = a.n_heads / a.n_kv_heads;
    const int R = a.n_q * G;                             // 9..32 on this path
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    pdl_wait();
    pdl_trigger();

    int len = a.kv_len[s];
    if (len < 0 || len > a.max_kv_len) {
        if (threadIdx.x == 0 && split == 0 && kh == 0 && a.err) atomicOr(a.err, KVQ_ERR_KV_LEN);
        len = len < 0 ? 0 : a.max_kv_len;
    }
    int lo, hi;
    split_range(len, a.n_splits, split, lo, hi);
    const int n_tiles = (int)ceil_div(hi - lo, kTile);
    const int64_t plane_row = ((int64_t)s * a.n_kv_heads + kh) * a.capacity;

    if (threadIdx.x == 0) {
        s_timeout = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Q rows of this kv head, fp16, head_dim permuted to the K-unpack order and
    // swizzled in 16-byte chunks; rows >= R are zero.
    {
        const QT *q = static_cast<const QT *>(a.q);
        for (int idx = threadIdx.x; idx < C::ROWS * D; idx += kThreads) {
            const int n = idx / D, kg = idx % D;                 // kg = 16 * ks + kp
            __half v = __float2half_rn(0.0f);
            if (n < R) {
                const int d = kpos_to_d<KC>(kg >> 4, kg & 15);
                const int i = n / G, jj = n % G;
                const QT x = q[(((int64_t)s * a.n_q + i) * a.n_heads + kh * G + jj) * D + d];
                if constexpr (sizeof(QT) == 2) v = x;
                else v = __float2half_rn(x);
            }
            *reinterpret_cast<__half *>(q_s + q_chunk_off<D>(n, kg >> 3) + (kg & 7) * 2) = v;
        }
    }
    __syncthreads();

    // consumer state: O^T for this warp's MTW 16-wide d tiles x NT n-tiles
    float o[MTW][NT][4];
#pragma unroll
    for (int t = 0; t < MTW; ++t)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[t][nt][c] = 0.0f;
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) m[nt][0] = m[nt][1] = -INFINITY, l[nt][0] = l[nt][1] = 0.0f;
    // this warp's d tiles: global tile index mt = warp * MTW + t, group g = mt / 4, e = mt % 4
    const int g_w = (warp * MTW) / 4, e0 = (warp * MTW) % 4;

    if (warp == kConsumerWarps) {
        // ---------------- producer (as in the narrow kernel) ----------------
        if (lane == 0) {
            const uint8_t *ksc = reinterpret_cast<const uint8_t *>(a.k.sc);
            const uint8_t *vsc = reinterpret_cast<const uint8_t *>(a.v.sc);
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages;
                if (j >= kStages && !mbar_wait(bar_empty + 8 * st, ((j / kStages) & 1) ^ 1)) {
                    s_timeout = 1;
                    break;
                }
                if (s_timeout) break;
                const int t0 = lo + j * kTile;
                const uint32_t base = smem_u32(smem + st * C::STAGE);
                const uint32_t full = bar_full + 8 * st;
                mbar_expect_tx(full, (uint32_t)(KG::BYTES + VG::BYTES + kTile * (C::KSB + C::VSB)));
                const int y = (int)(plane_row + t0);
#pragma unroll
                for (int b = 0; b < KG::NB; ++b)
                    tma_load_2d(base + C::K_OFF + b * kTile * KG::BI, &tmk, b * KG::BI, y, full);
#pragma unroll
                for (int b = 0; b < VG::NB; ++b)
                    tma_load_2d(base + C::V_OFF + b * kTile * VG::BI, &tmv, b * VG::BI, y, full);
                bulk_load(base + C::KS_OFF, ksc + (plane_row + t0) * C::KSB, kTile * C::KSB, full);
                bulk_load(base + C::VS_OFF, vsc + (plane_row + t0) * C::VSB, kTile * C::VSB, full);
                issued = j + 1;
            }
            // never leave while a copy into this CTA's shared memory is in flight
            // (normally a no-op: the consumers have already seen every tile land)
            for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j)
                if (!mbar_wait(bar_full + 8 * (j % kStages), (j / kStages) & 1)) s_timeout = 1;
        }
    } else {
        // ---------------- consumers ----------------
        int nv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = nt * 8 + 2 * tig + c;
                nv[nt][c] = r < R ? len - a.n_q + r / G + 1 : 0x7FFFFFFF;
            }
        int nv_min = 0x7FFFFFFF;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) nv_min = min(nv_min, min(nv[nt][0], nv[nt][1]));
        const float sl2 = a.scale_log2;
        const int tl = warp * 16;
        const uint32_t q_base = smem_u32(q_s);

        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % kStages;
            if (s_timeout || !mbar_wait(bar_full + 8 * st, (j / kStages) & 1)) {
                s_timeout = 1;
            }
            // the named barriers below need all four warps every tile, so a
            // timed-out warp keeps going with masked data instead of leaving
            const bool dead = s_timeout != 0;
            const int t_tile = lo + j * kTile;
            const int tb = t_tile + tl;
            const uint32_t base = smem_u32(smem + st * C::STAGE);
            const uint32_t kt = base + C::K_OFF, vt = base + C::V_OFF;
            const uint8_t *ksp = smem + st * C::STAGE + C::KS_OFF;
            const uint8_t *vsp = smem + st * C::STAGE + C::VS_OFF;

            // ---- phase A: S^T for this warp's 16 tokens ----
            float sc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[nt][c] = 0.0f;
            if (tb < hi && !dead) {
                const __half *sk0 = reinterpret_cast<const __half *>(ksp + (tl + gid) * C::KSB);
                const __half *sk1 = reinterpret_cast<const __half *>(ksp + (tl + gid + 8) * C::KSB);
                const int ltok = tl + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int lch = lane >> 4;
#pragma unroll
                for (int g = 0; g < NGK; ++g) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(KG::chunk_addr(kt, ltok, 2 * g + lch), r0, r1, r2, r3);
                    float cg[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) cg[nt][c] = 0.0f;
                    uint32_t h0[4], h1[4], h2[4], h3[4];
                    if constexpr (KC == KVQ_CODEC_Q4_G64) {
                        unpack_q4(r0, h0);
                        unpack_q4(r1, h1);
                        unpack_q4(r2, h2);
                        unpack_q4(r3, h3);
                    } else {
                        uint32_t t2[2];
                        unpack_q8(r0, t2); h0[0] = t2[0]; h0[1] = t2[1];
                        unpack_q8(r1, t2); h1[0] = t2[0]; h1[1] = t2[1];
                        unpack_q8(r2, t2); h2[0] = t2[0]; h2[1] = t2[1];
                        unpack_q8(r3, t2); h3[0] = t2[0]; h3[1] = t2[1];
                    }
#pragma unroll
                    for (int k = 0; k < KSTEP_PER_G; ++k) {
                        const int ks = g * KSTEP_PER_G + k;
#pragma unroll
                        for (int np = 0; np < (NT + 1) / 2; ++np) {
                            // n-tiles 2np and 2np+1 (row 31 exists, so the pair is always readable)
                            const int qrow = (2 * np + (lane >> 4)) * 8 + (lane & 7);
                            uint32_t b00, b01, b10, b11;
                            ldsm_x4(q_base + q_chunk_off<D>(qrow, 2 * ks + ((lane >> 3) & 1)), b00, b01, b10, b11);
                            mma16816(cg[2 * np], h0[k], h1[k], h2[k], h3[k], b00, b01);
                            if (2 * np + 1 < NT) mma16816(cg[2 * np + 1], h0[k], h1[k], h2[k], h3[k], b10, b11);
                        }
                    }
                    const float d0 = __half2float(sk0[g]) * sl2, d1 = __half2float(sk1[g]) * sl2;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        sc[nt][0] = fmaf(cg[nt][0], d0, sc[nt][0]);
                        sc[nt][1] = fmaf(cg[nt][1], d0, sc[nt][1]);
                        sc[nt][2] = fmaf(cg[nt][2], d1, sc[nt][2]);
                        sc[nt][3] = fmaf(cg[nt][3], d1, sc[nt][3]);
                    }
                }
            }
            {
                const int ta = tb + gid, tc = ta + 8;
                const bool tail = dead || tb + 16 > hi || tb + 16 > nv_min;
                if (tail) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (dead || !(ta < hi && ta < nv[nt][0])) sc[nt][0] = -INFINITY;
                        if (dead || !(ta < hi && ta < nv[nt][1])) sc[nt][1] = -INFINITY;
                        if (dead || !(tc < hi && tc < nv[nt][0])) sc[nt][2] = -INFINITY;
                        if (dead || !(tc < hi && tc < nv[nt][1])) sc[nt][3] = -INFINITY;
                    }
                }
            }
            // ---- CTA-wide running max per row ----
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx0 = fmaxf(sc[nt][0], sc[nt][2]), mx1 = fmaxf(sc[nt][1], sc[nt][3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                if (gid == 0) {
                    red_m[warp * 32 + nt * 8 + 2 * tig] = mx0;
                    red_m[warp * 32 + nt * 8 + 2 * tig + 1] = mx1;
                }
            }
            consumer_bar();
            float corr[NT][2];
            bool grow = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col = nt * 8 + 2 * tig + c;
                    float tmax = red_m[col];
#pragma unroll
                    for (int w = 1; w < kConsumerWarps; ++w) tmax = fmaxf(tmax, red_m[w * 32 + col]);
                    const float mn = fmaxf(m[nt][c], tmax);
                    corr[nt][c] = (mn == -INFINITY) ? 1.0f : ex2(m[nt][c] - mn);
                    grow |= mn > m[nt][c];
                    m[nt][c] = mn;
                }
            // p for this warp's tokens, written for phase B
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float ms0 = (m[nt][0] == -INFINITY) ? 0.0f : m[nt][0];
                const float ms1 = (m[nt][1] == -INFINITY) ? 0.0f : m[nt][1];
                const float p0 = ex2(sc[nt][0] - ms0), p1 = ex2(sc[nt][1] - ms1);
                const float p2 = ex2(sc[nt][2] - ms0), p3 = ex2(sc[nt][3] - ms1);
                l[nt][0] = l[nt][0] * corr[nt][0] + p0 + p2;
                l[nt][1] = l[nt][1] * corr[nt][1] + p1 + p3;
                *reinterpret_cast<float2 *>(p_s + (tl + gid) * C::PS + nt * 8 + 2 * tig) = make_float2(p0, p1);
                *reinterpret_cast<float2 *>(p_s + (tl + gid + 8) * C::PS + nt * 8 + 2 * tig) = make_float2(p2, p3);
            }
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int t = 0; t < MTW; ++t)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        o[t][nt][0] *= corr[nt][0];
                        o[t][nt][1] *= corr[nt][1];
                        o[t][nt][2] *= corr[nt][0];
                        o[t][nt][3] *= corr[nt][1];
                    }
            }
            consumer_bar();

            // ---- phase B: O^T += V^T P'^T over the tile, this warp's d slice ----
            if (!dead) {
                const int ltok0 = (lane & 7) + 8 * (lane >> 4);
                const int lch = (lane >> 3) & 1;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    if (t_tile + 16 * kk >= hi) break;
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(VG::chunk_addr(vt, 16 * kk + ltok0, 2 * g_w + lch), r0, r1, r2, r3);
                    uint32_t u0[4], u1[4], u2[4], u3[4];
                    unpack_q4(r0, u0);
                    unpack_q4(r1, u1);
                    unpack_q4(r2, u2);
                    unpack_q4(r3, u3);
                    // V scales of the four tokens this lane's B fragment covers (0 past the split end)
                    float sv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tk = 16 * kk + 2 * tig + (q & 1) + 8 * (q >> 1);
                        sv[q] = (t_tile + tk < hi)
                                    ? __half2float(reinterpret_cast<const __half *>(vsp + tk * C::VSB)[g_w])
                                    : 0.0f;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int col = nt * 8 + gid;
                        const float *pr = p_s + (16 * kk + 2 * tig) * C::PS + col;
                        const uint32_t b0 = pack_f16x2(pr[0] * sv[0], pr[C::PS] * sv[1]);
                        const uint32_t b1 = pack_f16x2(pr[8 * C::PS] * sv[2], pr[9 * C::PS] * sv[3]);
#pragma unroll
                        for (int t = 0; t < MTW; ++t) {
                            // e = e0 + t with e0 in {0, 4 - MTW}: compile-time register indices
                            const bool up = (MTW < 4) && e0 != 0;
                            const int el = t, eh = (t + 4 - MTW) & 3;
                            mma16816(o[t][nt], up ? u0[eh] : u0[el], up ? u1[eh] : u1[el], up ? u2[eh] : u2[el],
                                     up ? u3[eh] : u3[el], b0, b1);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        }
        // row sums: over the 8 lanes of a column, then over the warps
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
                l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
            }
        if (gid == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                red_l[warp * 32 + nt * 8 + 2 * tig] = l[nt][0];
                red_l[warp * 32 + nt * 8 + 2 * tig + 1] = l[nt][1];
            }
        }
        consumer_bar();
        // every warp holds the same m, so its slice only needs 1 / L
        const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n = nt * 8 + 2 * tig + (c & 1);
                if (n >= R) continue;
                float L = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) L += red_l[w * 32 + n];
                const float M = m[nt][c & 1];
                const bool empty = (M == -INFINITY || L <= 0.0f);
                const float inv = empty ? 0.0f : 1.0f / L;
                const int i = n / G, jj = n % G;
                const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + jj;
                float *dst = (a.n_splits == 1) ? a.out + orow * D : a.part_o + ((int64_t)split * rows_total + orow) * D;
                const int d = 64 * g_w + 32 * (c >> 1) + 4 * gid + e0;
                if constexpr (MTW == 4) {
                    *reinterpret_cast<float4 *>(dst + d) =
                        make_float4(o[0][nt][c] * inv, o[1][nt][c] * inv, o[2][nt][c] * inv, o[3][nt][c] * inv);
                } else {
#pragma unroll
                    for (int t = 0; t < MTW; ++t) dst[d + t] = o[t][nt][c] * inv;
                }
                if (warp == 0 && gid == 0 && (c >> 1) == 0) {
                    const float lse = empty ? -INFINITY : (M + log2f(L)) * kLn2;
                    if (a.n_splits == 1) {
                        if (a.out_lse) a.out_lse[orow] = lse;
                    } else {
                        a.part_lse[(int64_t)split * rows_total + orow] = lse;
                    }
                }
            }
        if (threadIdx.x == 0 && s_timeout && a.err) atomicOr(a.err, KVQ_ERR_TIMEOUT);
    }
}

template <int KC, int D, int NT, typename QT>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t st)
{
    using C = WideCfg<KC, D, NT>;
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    CUtensorMap tk, tv;
    if (!make_codes_map(&tk, a.k.qs, C::KRB, rows) || !make_codes_map(&tv, a.v.qs, C::VRB, rows))
        return cudaErrorInvalidValue;
    auto kern = decode_wide_kernel<KC, D, NT, QT>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        // two CTAs per SM need the largest shared-memory carveout
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    dim3 grid(a.n_splits, a.n_kv_heads, a.n_seq);
    return launch_pdl(kern, grid, dim3(kThreads), C::SMEM, st, a, tk, tv);
}

template <int KC, int D, typename QT>
cudaError_t launch_nt(const DecodeArgs &a, cudaStream_t st)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    switch ((R + 7) / 8) {
    case 2: return launch_t<KC, D, 2, QT>(a, st);
    case 3: return launch_t<KC, D, 3, QT>(a, st);
    case 4: return launch_t<KC, D, 4, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int KC, typename QT>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st)
{
    switch (a.head_dim) {
    case 128: return launch_nt<KC, 128, QT>(a, st);
    case 256: return launch_nt<KC, 256, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_wide_supported(const DecodeArgs &a)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    return R > 8 && R <= 32 && a.v.codec == KVQ_CODEC_Q4_G64 && (a.head_dim == 128 || a.head_dim == 256) &&
           rows < (1LL << 31) && tensor_maps_available();
}

cudaError_t launch_decode_wide(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    const bool k4 = a.k.codec == KVQ_CODEC_Q4_G64;
    if (q_dtype == KVQ_F16)
        return k4 ? launch_d<KVQ_CODEC_Q4_G64, __half>(a, st) : launch_d<KVQ_CODEC_Q8_0, __half>(a, st);
    return k4 ? launch_d<KVQ_CODEC_Q4_G64, float>(a, st) : launch_d<KVQ_CODEC_Q8_0, float>(a, st);
}

}  // namespace kvq
