// kvq_decode_mma.cu -- split-K decode attention over a packed Q4_G64 (or q8_0-K)
// cache on the tensor cores, for up to 8 query rows per kv head (GQA group x
// query tokens <= 8) and head_dim 64/128/256.
//
// What it computes is the same as the generic kernel (den_llama.cpp, "What's
// in the fork": the fattn-vec Q4_G64 instances; "What this fork is": signed
// INT4 + one FP16 scale per 64 values): per (sequence, kv head, split) the
// softmax attention of that kv head's query rows over the split's tokens,
// emitted as a final result (one split) or as a partial normalised over the
// split with its log-sum-exp.
//
// Design (sm_103a):
//  * One producer warp streams each 64-token tile of packed K and V codes with
//    2D TMA (128/64/32-byte swizzle, so ldmatrix below is bank-conflict free)
//    and the fp16 scales with 1D bulk copies into a 4-stage shared-memory ring
//    guarded by mbarriers.  Four consumer warps each take 16 tokens of a tile.
//  * S^T = K Q^T on mma.sync.m16n8k16 (tokens are the M=16 side, the <= 8
//    query rows the N=8 side).  ldmatrix.x4 hands each lane 4-byte pieces of
//    two token rows; the nibbles are turned into fp16 integers in registers
//    with one LOP3 + one HADD2/HFMA2 per two values (1024 + code trick), so the
//    codes enter the MMA exactly.  Each 64-value group accumulates separately
//    and is scaled by its fp16 scale in fp32.  The head_dim order inside a
//    k-step is permuted consistently in K and Q (a dot product does not care).
//  * Online softmax in log2 units on the S^T fragment; the running max per
//    query row is reduced across the 8 lanes that share it.
//  * O^T += V^T P'^T on mma.sync with V^T from ldmatrix.x4.trans (which pairs
//    two tokens at the same head_dim index, exactly the A-fragment pairing) and
//    P' = p * v_scale(token, group) converted to fp16 and moved from the
//    accumulator layout to the B-operand layout with movmatrix.trans.
//  * At the end the four warps' (max, sum, O) are combined through shared
//    memory and written as fp32.
//
// Every wait on an mbarrier is bounded: after ~1 s the kernel sets
// KVQ_ERR_TIMEOUT in the caller's error word and finishes without further
// waits; nothing traps.
#include "kvq_ptx.cuh"

namespace kvq {
using namespace ptx;
namespace {

template <int KC, int D>
struct MmaCfg {
    static constexpr int KRB = row_bytes(KC, D), VRB = D / 2;
    static constexpr int KSB = 2 * scales_per_row(KC, D), VSB = 2 * (D / 64);
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = align_up(kTile * KRB, 1024);
    static constexpr int KS_OFF = V_OFF + align_up(kTile * VRB, 1024);
    static constexpr int VS_OFF = KS_OFF + align_up(kTile * KSB, 128);
    static constexpr int STAGE = align_up(VS_OFF + kTile * VSB, 1024);
    static constexpr int Q_OFF = kStages * STAGE;                  // fp16 [8][D]
    static constexpr int BAR_OFF = Q_OFF + 8 * D * 2;
    static constexpr int SMEM = BAR_OFF + 2 * kStages * 8 + 1024;  // + slack for 1024-byte alignment
    static constexpr int COMB = kConsumerWarps * 8 * (D + 2) * 4;  // combine scratch (reuses the stages)
    static_assert(COMB <= kStages * STAGE, "combine scratch must fit in the ring");
};

template <int KC, int D, typename QT>
__global__ void __launch_bounds__(kThreads, 2)
decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv)
{
    using C = MmaCfg<KC, D>;
    using KG = TileGeom<C::KRB>;
    using VG = TileGeom<C::VRB>;
    constexpr int NGK = D / group_size(KC);      // K scale groups per row
    constexpr int NGV = D / 64;                  // V scale groups per row
    constexpr int KSTEP_PER_G = group_size(KC) / 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __half *q_s = reinterpret_cast<__half *>(smem + C::Q_OFF);
    const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);
    const uint32_t bar_empty = bar_full + kStages * 8;
    __shared__ volatile int s_timeout;

    const int split = blockIdx.x, kh = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.n_heads / a.n_kv_heads;
    const int R = a.n_q * G;                     // <= 8 on this path
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
    // query rows of this kv head as fp16 (rows >= R are zero)
    {
        const QT *q = static_cast<const QT *>(a.q);
        for (int idx = threadIdx.x; idx < 8 * D; idx += kThreads) {
            const int r = idx / D, d = idx % D;
            __half v = __float2half_rn(0.0f);
            if (r < R) {
                const int i = r / G, j = r % G;
                const QT x = q[(((int64_t)s * a.n_q + i) * a.n_heads + kh * G + j) * D + d];
                if constexpr (sizeof(QT) == 2) v = x;
                else v = __float2half_rn(x);
            }
            q_s[idx] = v;
        }
    }
    __syncthreads();

    const int gid = lane >> 2, tig = lane & 3;
    float o[NGV][4][4];
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
#pragma unroll
    for (int g = 0; g < NGV; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[g][e][c] = 0.0f;

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
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
        // Q as the B operand of S^T = K Q^T, head_dim order matching the K unpack
        uint32_t qb[NGK][KSTEP_PER_G][2];
#pragma unroll
        for (int g = 0; g < NGK; ++g)
#pragma unroll
            for (int st = 0; st < KSTEP_PER_G; ++st) {
                int da, db;
                if constexpr (KC == KVQ_CODEC_Q4_G64) {
                    da = 64 * g + 8 * tig + st;             // pair (da, da + 4)
                    db = da + 32;
                    qb[g][st][0] = h2_as_u32(__halves2half2(q_s[gid * D + da], q_s[gid * D + da + 4]));
                    qb[g][st][1] = h2_as_u32(__halves2half2(q_s[gid * D + db], q_s[gid * D + db + 4]));
                } else {
                    da = 32 * g + 4 * tig + 2 * st;         // pair (da, da + 1)
                    db = da + 16;
                    qb[g][st][0] = h2_as_u32(__halves2half2(q_s[gid * D + da], q_s[gid * D + da + 1]));
                    qb[g][st][1] = h2_as_u32(__halves2half2(q_s[gid * D + db], q_s[gid * D + db + 1]));
                }
            }
        // visible keys of this lane's two query-row columns (padding rows: no mask)
        int nv[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int r = 2 * tig + c;
            nv[c] = r < R ? len - a.n_q + r / G + 1 : 0x7FFFFFFF;
        }
        const int nv_min = min(nv[0], nv[1]);
        const float sl2 = a.scale_log2;
        const int tl = warp * 16;                               // this warp's first token in a tile

        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % kStages;
            if (s_timeout || !mbar_wait(bar_full + 8 * st, (j / kStages) & 1)) {
                s_timeout = 1;
                break;
            }
            const int tb = lo + j * kTile + tl;
            if (tb < hi) {
                const uint32_t base = smem_u32(smem + st * C::STAGE);
                const uint32_t kt = base + C::K_OFF, vt = base + C::V_OFF;
                const uint8_t *ksp = smem + st * C::STAGE + C::KS_OFF;
                const uint8_t *vsp = smem + st * C::STAGE + C::VS_OFF;

                // ---- S^T = K Q^T ----
                float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                {
                    const __half *sk0 = reinterpret_cast<const __half *>(ksp + (tl + gid) * C::KSB);
                    const __half *sk1 = reinterpret_cast<const __half *>(ksp + (tl + gid + 8) * C::KSB);
                    const int ltok = tl + (lane & 7) + 8 * ((lane >> 3) & 1);
                    const int lch = lane >> 4;
#pragma unroll
                    for (int g = 0; g < NGK; ++g) {
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(KG::chunk_addr(kt, ltok, 2 * g + lch), r0, r1, r2, r3);
                        float cg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        if constexpr (KC == KVQ_CODEC_Q4_G64) {
                            uint32_t h0[4], h1[4], h2[4], h3[4];
                            unpack_q4(r0, h0);
                            unpack_q4(r1, h1);
                            unpack_q4(r2, h2);
                            unpack_q4(r3, h3);
#pragma unroll
                            for (int k = 0; k < 4; ++k) mma16816(cg, h0[k], h1[k], h2[k], h3[k], qb[g][k][0], qb[g][k][1]);
                        } else {
                            uint32_t h0[2], h1[2], h2[2], h3[2];
                            unpack_q8(r0, h0);
                            unpack_q8(r1, h1);
                            unpack_q8(r2, h2);
                            unpack_q8(r3, h3);
#pragma unroll
                            for (int k = 0; k < 2; ++k) mma16816(cg, h0[k], h1[k], h2[k], h3[k], qb[g][k][0], qb[g][k][1]);
                        }
                        const float d0 = __half2float(sk0[g]) * sl2, d1 = __half2float(sk1[g]) * sl2;
                        sc[0] = fmaf(cg[0], d0, sc[0]);
                        sc[1] = fmaf(cg[1], d0, sc[1]);
                        sc[2] = fmaf(cg[2], d1, sc[2]);
                        sc[3] = fmaf(cg[3], d1, sc[3]);
                    }
                }
                // ---- mask the tail / causal rows ----
                // (tokens past the split end may hold any bytes: their scores
                // are selected away and their V scale replaced by 0 below)
                const bool okA = tb + gid < hi, okC = tb + gid + 8 < hi;
                if (tb + 16 > hi || tb + 16 > nv_min) {
                    const int ta = tb + gid, tc = ta + 8;
                    if (!(ta < hi && ta < nv[0])) sc[0] = -INFINITY;
                    if (!(ta < hi && ta < nv[1])) sc[1] = -INFINITY;
                    if (!(tc < hi && tc < nv[0])) sc[2] = -INFINITY;
                    if (!(tc < hi && tc < nv[1])) sc[3] = -INFINITY;
                }
                // ---- online softmax (log2 units) ----
                float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const bool grow = mx0 > m[0] || mx1 > m[1];
                if (__any_sync(0xffffffffu, grow)) {
                    const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
                    const float c0 = (n0 == -INFINITY) ? 1.0f : ex2(m[0] - n0);
                    const float c1 = (n1 == -INFINITY) ? 1.0f : ex2(m[1] - n1);
                    m[0] = n0;
                    m[1] = n1;
                    l[0] *= c0;
                    l[1] *= c1;
#pragma unroll
                    for (int g = 0; g < NGV; ++g)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            o[g][e][0] *= c0;
                            o[g][e][1] *= c1;
                            o[g][e][2] *= c0;
                            o[g][e][3] *= c1;
                        }
                }
                const float ms0 = (m[0] == -INFINITY) ? 0.0f : m[0];
                const float ms1 = (m[1] == -INFINITY) ? 0.0f : m[1];
                float p[4];
                p[0] = ex2(sc[0] - ms0);
                p[1] = ex2(sc[1] - ms1);
                p[2] = ex2(sc[2] - ms0);
                p[3] = ex2(sc[3] - ms1);
                l[0] += p[0] + p[2];
                l[1] += p[1] + p[3];

                // ---- O^T += V^T P'^T ----
                {
                    const __half *sv0 = reinterpret_cast<const __half *>(vsp + (tl + gid) * C::VSB);
                    const __half *sv1 = reinterpret_cast<const __half *>(vsp + (tl + gid + 8) * C::VSB);
                    const int ltok = tl + (lane & 7) + 8 * (lane >> 4);
                    const int lch = (lane >> 3) & 1;
#pragma unroll
                    for (int g = 0; g < NGV; ++g) {
                        const float v0 = okA ? __half2float(sv0[g]) : 0.0f;
                        const float v1 = okC ? __half2float(sv1[g]) : 0.0f;
                        const uint32_t b0 = movm_t(pack_f16x2(p[0] * v0, p[1] * v0));
                        const uint32_t b1 = movm_t(pack_f16x2(p[2] * v1, p[3] * v1));
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_t(VG::chunk_addr(vt, ltok, 2 * g + lch), r0, r1, r2, r3);
                        uint32_t u0[4], u1[4], u2[4], u3[4];
                        unpack_q4(r0, u0);
                        unpack_q4(r1, u1);
                        unpack_q4(r2, u2);
                        unpack_q4(r3, u3);
#pragma unroll
                        for (int e = 0; e < 4; ++e) mma16816(o[g][e], u0[e], u1[e], u2[e], u3[e], b0, b1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        }
        // per-column sums over the 8 lanes that share a column
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
    }
    // every consumer is past its last tile, so every issued copy has landed and
    // the ring can be reused as combine scratch
    __syncthreads();
    if (warp < kConsumerWarps) {
        float *cm = reinterpret_cast<float *>(smem);        // [warps][8]
        float *cl = cm + kConsumerWarps * 8;                // [warps][8]
        float *co = cl + kConsumerWarps * 8;                // [warps][8][D]
        if (gid == 0) {
            cm[warp * 8 + 2 * tig] = m[0];
            cm[warp * 8 + 2 * tig + 1] = m[1];
            cl[warp * 8 + 2 * tig] = l[0];
            cl[warp * 8 + 2 * tig + 1] = l[1];
        }
#pragma unroll
        for (int g = 0; g < NGV; ++g)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n = 2 * tig + (c & 1);
                const int d = 64 * g + 32 * (c >> 1) + 4 * gid;
                *reinterpret_cast<float4 *>(co + ((size_t)warp * 8 + n) * D + d) =
                    make_float4(o[g][0][c], o[g][1][c], o[g][2][c], o[g][3][c]);
            }
    }
    __syncthreads();

    // ---------------- combine the consumer warps and write ----------------
    {
        const float *cm = reinterpret_cast<const float *>(smem);
        const float *cl = cm + kConsumerWarps * 8;
        const float *co = cl + kConsumerWarps * 8;
        const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;
        for (int idx = threadIdx.x; idx < R * (D / 4); idx += kThreads) {
            const int n = idx / (D / 4), d4 = idx % (D / 4);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * 8 + n]);
            float L = 0.0f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = cm[w * 8 + n];
                    if (mw == -INFINITY) continue;
                    const float f = ex2(mw - M);
                    L = fmaf(f, cl[w * 8 + n], L);
                    const float4 v = *reinterpret_cast<const float4 *>(co + ((size_t)w * 8 + n) * D + 4 * d4);
                    acc.x = fmaf(f, v.x, acc.x);
                    acc.y = fmaf(f, v.y, acc.y);
                    acc.z = fmaf(f, v.z, acc.z);
                    acc.w = fmaf(f, v.w, acc.w);
                }
                const float inv = 1.0f / L;
                acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
            }
            const int i = n / G, jj = n % G;
            const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + jj;
            float *dst = (a.n_splits == 1) ? a.out + orow * D : a.part_o + ((int64_t)split * rows_total + orow) * D;
            reinterpret_cast<float4 *>(dst)[d4] = acc;
            if (d4 == 0) {
                const float lse = (M == -INFINITY || L <= 0.0f) ? -INFINITY : (M + log2f(L)) * kLn2;
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int KC, int D, typename QT>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t st)
{
    using C = MmaCfg<KC, D>;
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    CUtensorMap tk, tv;
    if (!make_codes_map(&tk, a.k.qs, C::KRB, rows) || !make_codes_map(&tv, a.v.qs, C::VRB, rows))
        return cudaErrorInvalidValue;
    auto kern = decode_mma_kernel<KC, D, QT>;
    static bool attr_set[64] = {};           // the attribute is per device
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

template <int KC, typename QT>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st)
{
    switch (a.head_dim) {
    case 64: return launch_t<KC, 64, QT>(a, st);
    case 128: return launch_t<KC, 128, QT>(a, st);
    case 256: return launch_t<KC, 256, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

namespace ptx {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Codes plane [rows][row_bytes] as a 2D uint8 tensor, box = (min(row_bytes,128), kTile).
bool make_codes_map(CUtensorMap *m, void *base, int row_bytes, int64_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int bi = row_bytes < 128 ? row_bytes : 128;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)bi, (cuuint32_t)kTile};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = bi == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : bi == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tensor_maps_available() { return encode_fn() != nullptr; }

}  // namespace ptx

bool decode_mma_supported(const DecodeArgs &a)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    return R <= 8 && a.v.codec == KVQ_CODEC_Q4_G64 &&
           (a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256) && rows < (1LL << 31) &&
           tensor_maps_available();
}

cudaError_t launch_decode_mma(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    const bool k4 = a.k.codec == KVQ_CODEC_Q4_G64;
    if (q_dtype == KVQ_F16)
        return k4 ? launch_d<KVQ_CODEC_Q4_G64, __half>(a, st) : launch_d<KVQ_CODEC_Q8_0, __half>(a, st);
    return k4 ? launch_d<KVQ_CODEC_Q4_G64, float>(a, st) : launch_d<KVQ_CODEC_Q8_0, float>(a, st);
}

}  // namespace kvq
