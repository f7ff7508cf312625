// kvq_decode_tc.cuh -- split-K decode / MTP-verify attention over a packed cache
// on the tensor cores, for any number of query rows per kv head (GQA group x
// query tokens; up to 32 in one CTA, more -- a prompt chunk -- in blocks of
// 32, one CTA each), head_dim 64/128/256, K and V each in Q4_G64, Q4_G32, q8_0 or
// NVFP4 (the kernel template; kvq_decode_tc.cu, kvq_decode_tc_g32.cu,
// kvq_decode_tc_q8v.cu and kvq_decode_tc_fp4v.cu hold its instances for the
// four V codecs, so that they compile in parallel).  NVFP4 codes enter the
// MMAs as exact fp16 values already multiplied by their E4M3 scales (an E2M1
// value times an E4M3 scale has at most 6 significant bits), so they need no
// bias, offset or per-group scaling of the accumulators.
// (den_llama.cpp, "What's in the fork": the fattn-vec Q4_G64 instances; "What
// this fork is": the 4-bit code with an fp16 scale per 64-value group; "Results": MTP
// n-max 2, i.e. 1 + 2 query tokens per sequence).
//
// Per (sequence, kv head, split) the query rows of the kv head attend to the
// split's tokens intersected with each row's visible keys; the result is final
// (one split) or a partial normalised over the split with its log-sum-exp.
// Shapes of up to 8 rows per kv head over Q4_G64 V with Q4_G64 or q8_0 K go to
// the single-warp-block kernel of kvq_decode_warp.cu instead; this kernel takes
// the rest (MTP verify with more rows, the other V codecs, NVFP4 or Q4_G32 K).
//
// Work of one CTA (four warps, no dedicated producer), one CTA barrier per tile:
//  * Thread 0 fetches the query rows with 1D bulk copies and the first tiles of
//    64 tokens (K and V codes by swizzled 2D TMA, their scales by bulk
//    copies) into a 3-stage (2 for q8_0 K and V) shared-memory ring.  After the barrier of tile j it
//    refills the stage of tile j - 1, which every warp has finished with.
//  * Phase A: warp w computes S^T = K Q^T for tokens [16w, 16w+16) of the tile
//    and all n-tiles of 8 rows on mma.sync.m16n8k16.  The K codes enter as
//    exact fp16 integers with their bias (1032 + q or 1152 + 16 q, one LOP3 per
//    two values); each 64-value group starts its accumulator at minus the
//    group's bias term and is scaled by the group's fp16 scale in fp32.  The
//    scores (log2 units) and the warp's per-row maximum go to shared memory
//    (double-buffered by tile parity, so one barrier per tile suffices).
//  * Phase B: every warp forms the same new running maximum from the four
//    warps' maxima, turns the scores of its operand fragments into
//    p = 2^(s - m) (keeping the row sums itself) and accumulates
//    O^T += V^T P'^T for its quarter of head_dim over the tile's 64 tokens:
//    V^T fragments from ldmatrix.trans (it pairs two tokens at one head_dim
//    index, the A-fragment pairing); P' = p * v_scale(token) is rounded once
//    to fp16.  With one n-tile and one V group per warp the V codes enter as
//    exact fp16 subnormals (q + 8) 2^-24 (16 (q + 8) 2^-24 at odd head_dim
//    indices), one LOP3 per two values, and their offset 8 is removed once per
//    tile from the tile's sum of P' (one MMA against a ones operand per 16
//    tokens); otherwise, where that sum would take one MMA per n-tile and V
//    group, an exact fp16 subtraction turns the biased form into q (16 q).
//    The V offset is kept small, unlike the K bias: the MMA aligns its
//    addends to the largest one and drops the bits below about 25, so
//    1032 * P' terms would cost the output about ten bits.
//  * Because the warps share the maximum and each owns its own columns, the
//    end of the CTA is a division by the row sum: no cross-warp combine.
//
// Every mbarrier wait is bounded: after ~1 s the kernel sets KVQ_ERR_TIMEOUT in
// the caller's error word and finishes without further waits; nothing traps.
#pragma once

#include "kvq_decode_common.cuh"

namespace kvq {
using namespace ptx;
namespace {

constexpr int kW = 4;                        // warps
constexpr int kT = kW * 32;                  // threads

__device__ __forceinline__ void warps_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kT) : "memory"); }

template <int KC, int VC, int D, int NT, typename QT>
struct TcCfg {
    static constexpr int KRB = row_bytes(KC, D), VRB = row_bytes(VC, D);
    static constexpr int KSB = scale_row_bytes(KC, D), VSB = scale_row_bytes(VC, D);
    // K accumulation groups: the codec's scale groups, or for NVFP4 (scales
    // applied to the operands) the 64 values of one ldmatrix unit
    static constexpr int KGS = is_fp4(KC) ? 64 : group_size(KC);
    static constexpr int NGK = D / KGS;
    static constexpr int ROWS = NT * 8;                           // query rows kept (zero past R)
    static constexpr int PS = ROWS + 4;                           // score row stride in floats (bank spread)
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = align_up(kTile * KRB, 1024);
    static constexpr int KS_OFF = V_OFF + align_up(kTile * VRB, 1024);
    static constexpr int VS_OFF = KS_OFF + align_up(kTile * KSB, 128);
    static constexpr int STAGE = align_up(VS_OFF + kTile * VSB, 1024);
    // ring stages: 3, or 2 where 3 would leave room for one CTA per SM only
    // (q8_0 K and V: 34 KB a stage)
    static constexpr int NS = STAGE <= 27 * 1024 ? 3 : 2;
    static constexpr int QP_OFF = NS * STAGE;                     // fp16 [ROWS][D], permuted, swizzled
    // an fp32 query also keeps its low fp16 part (same layout)
    static constexpr bool QLO = sizeof(QT) == 4;
    static constexpr int QPL_OFF = QP_OFF + ROWS * D * 2;
    static constexpr int KB_OFF = QPL_OFF + (QLO ? ROWS * D * 2 : 0);   // fp32 [NGK][ROWS]: minus the K bias terms
    // the query rows as given are only read before the first tile, the score
    // tiles and the maxima only after it: they share one region
    static constexpr int U_OFF = KB_OFF + align_up(ROWS * NGK * 4, 16);
    static constexpr int QST_OFF = U_OFF;
    static constexpr int S_OFF = U_OFF;                                   // fp32 [2][64][PS] scores
    static constexpr int RED_OFF = S_OFF + align_up(2 * kTile * PS * 4, 16);  // fp32 [2][kW][32] maxima
    // V scales of the tile transposed to [group][token] (0 past the split end), by tile parity
    static constexpr int NGV = D / group_size(VC);
    static constexpr int VT_OFF = RED_OFF + 2 * kW * 32 * 4;                  // fp16 [2][NGV][64]
    static constexpr int QST_BYTES = ROWS * D * (int)sizeof(QT);
    static constexpr int PR_BYTES = (VT_OFF - U_OFF) + 2 * NGV * kTile * 2;
    static constexpr int BAR_OFF = align_up(U_OFF + (QST_BYTES > PR_BYTES ? QST_BYTES : PR_BYTES), 16);
    static constexpr int SMEM = BAR_OFF + (NS + 1) * 8 + 1024;            // + alignment slack
    static constexpr int MTW = (D / 64 * 4) / kW;                 // 16-row head_dim tiles per warp in phase B
    // CTAs per SM the kernel is built for (shared memory allows 3 up to 16 rows)
    static constexpr int MIN_BLOCKS = NT <= 2 ? 3 : 2;
};

template <typename C, typename KG, typename VG>
__device__ __forceinline__ void issue_tile(uint32_t base, uint32_t full, const CUtensorMap *tmk,
                                           const CUtensorMap *tmv, const uint8_t *ksc, const uint8_t *vsc,
                                           int64_t row0)
{
    // the cache is read once per call: evict-first in L2
    const uint64_t pol = evict_first_policy();
    mbar_expect_tx(full, (uint32_t)(KG::BYTES + VG::BYTES + kTile * (C::KSB + C::VSB)));
    const int y = (int)row0;
#pragma unroll
    for (int b = 0; b < KG::NB; ++b)
        tma_load_2d(base + C::K_OFF + b * kTile * KG::BI, tmk, b * KG::BI, y, full, pol);
#pragma unroll
    for (int b = 0; b < VG::NB; ++b)
        tma_load_2d(base + C::V_OFF + b * kTile * VG::BI, tmv, b * VG::BI, y, full, pol);
    bulk_load_hint(base + C::KS_OFF, ksc + row0 * C::KSB, kTile * C::KSB, full, pol);
    bulk_load_hint(base + C::VS_OFF, vsc + row0 * C::VSB, kTile * C::VSB, full, pol);
}

template <int KC, int VC, int D, int NT, typename QT>
__global__ void __launch_bounds__(kT, (TcCfg<KC, VC, D, NT, QT>::MIN_BLOCKS))
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv)
{
    using C = TcCfg<KC, VC, D, NT, QT>;
    constexpr int kS = C::NS;
    using KG = TileGeom<C::KRB>;
    using VG = TileGeom<C::VRB>;
    constexpr int NGK = C::NGK;
    constexpr int KSTEP_PER_G = C::KGS / 16;
    constexpr int MTW = C::MTW;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qp = smem + C::QP_OFF;
    float *kb_s = reinterpret_cast<float *>(smem + C::KB_OFF);
    float *s_s0 = reinterpret_cast<float *>(smem + C::S_OFF);        // [2][64][PS]
    float *red_m0 = reinterpret_cast<float *>(smem + C::RED_OFF);    // [2][kW][32]
    __half *vt0 = reinterpret_cast<__half *>(smem + C::VT_OFF);      // [2][NGV][64]
    const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);
    const uint32_t bar_q = bar_full + kS * 8;
    __shared__ volatile int s_timeout;
    __shared__ int s_issued;

    // grid y: kv head x block of up to 8 NT query rows (one block unless a kv
    // head has more than 32 rows, as a prompt chunk does)
    const int split = blockIdx.x, kh = blockIdx.y / a.n_row_blocks, rblk = blockIdx.y % a.n_row_blocks;
    __shared__ int s_seq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int G = a.n_heads / a.n_kv_heads;
    const int r0 = rblk * 8 * NT;                         // this CTA's first row of the kv head
    const int R = min(8 * NT, a.n_q * G - r0);           // its rows
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        s_timeout = 0;
        s_issued = 0;
        for (int i = 0; i < kS; ++i) mbar_init(bar_full + 8 * i, 1);
        mbar_init(bar_q, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait();
    // The grid's z index is a rank: sequences in order of decreasing length, so
    // the CTAs of the longest sequences of a ragged batch are dispatched first
    // (a longest-first schedule).  Ties go by index; identity beyond kT sequences.
    int s = blockIdx.z;
    if (a.n_seq > 1 && a.n_seq <= kT) {
        if ((int)threadIdx.x < a.n_seq) {
            const int t = threadIdx.x, lt = a.kv_len[t];
            int rank = 0;
            for (int u = 0; u < a.n_seq; ++u) {
                const int lu = a.kv_len[u];
                rank += (lu > lt) || (lu == lt && u < t);
            }
            if (rank == (int)blockIdx.z) s_seq = t;
        }
        __syncthreads();
        s = s_seq;
    }
    // query rows r0 .. r0 + R - 1 (row r is head r % G of query token r / G;
    // a token's heads of this kv head are one contiguous run) by bulk copy, in
    // parallel with what follows
    if (threadIdx.x == 0) {
        const uint32_t row = (uint32_t)(D * sizeof(QT));
        mbar_expect_tx(bar_q, row * (uint32_t)R);
        const QT *q = static_cast<const QT *>(a.q);
        if (a.n_row_blocks == 1) {           // all n_q tokens, G heads each (no division on this path)
            for (int i = 0; i < a.n_q; ++i)
                bulk_load(smem_u32(smem + C::QST_OFF) + (uint32_t)(i * G) * row,
                          q + (((int64_t)s * a.n_q + i) * a.n_heads + kh * G) * D, (uint32_t)G * row, bar_q);
        } else {
            for (int i = r0 / G; i <= (r0 + R - 1) / G; ++i) {
                const int j0 = max(0, r0 - i * G), j1 = min(G, r0 + R - i * G);
                bulk_load(smem_u32(smem + C::QST_OFF) + (uint32_t)(i * G + j0 - r0) * row,
                          q + (((int64_t)s * a.n_q + i) * a.n_heads + kh * G + j0) * D, (uint32_t)(j1 - j0) * row,
                          bar_q);
            }
        }
    }

    int len = a.fixed_len >= 0 ? a.fixed_len : a.kv_len[s];
    if (len < 0 || len > a.max_kv_len) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0 && a.err) atomicOr(a.err, KVQ_ERR_KV_LEN);
        len = len < 0 ? 0 : a.max_kv_len;
    }
    int lo, hi;
    split_range(len, a.n_splits, split, lo, hi);
    // no row of this CTA sees past its last query token's keys (with one row
    // block the last row is the last query token, which sees them all)
    if (a.n_row_blocks > 1) hi = max(lo, min(hi, len + a.causal_extra - a.n_q + (r0 + R - 1) / G + 1));
    const int n_tiles = (int)ceil_div(hi - lo, kTile);
    const int64_t plane_row = ((int64_t)s * a.n_kv_heads + kh) * a.capacity;
    const uint8_t *ksc = reinterpret_cast<const uint8_t *>(a.k.sc);
    const uint8_t *vsc = reinterpret_cast<const uint8_t *>(a.v.sc);
    if (threadIdx.x == 0) {
        const int first = min(kS, n_tiles);
        for (int j = 0; j < first; ++j)
            issue_tile<C, KG, VG>(smem_u32(smem + j * C::STAGE), bar_full + 8 * j, &tmk, &tmv, ksc, vsc,
                                  plane_row + lo + j * kTile);
        s_issued = first;
    }

    // the query rows, permuted and swizzled, and the K bias terms
    if (!mbar_wait(bar_q, 0)) s_timeout = 1;
    prep_query<KC, D, C::ROWS, kT>(reinterpret_cast<const QT *>(smem + C::QST_OFF), qp, smem + C::QPL_OFF, kb_s, R,
                                   !s_timeout);
    __syncthreads();

    int nv[NT][2];
    int nv_min = 0x7FFFFFFF;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int r = nt * 8 + 2 * tig + c;
            nv[nt][c] = r < R ? len + a.causal_extra - a.n_q + (r0 + r) / G + 1 : 0x7FFFFFFF;   // padding rows: no mask
            nv_min = min(nv_min, nv[nt][c]);
        }
    const float sl2 = a.scale_log2;
    const int tl = warp * 16;                                           // phase A tokens
    // K fragments: one ldmatrix.x4 per 32 bytes of a token row (two 16-byte
    // chunks: one group of Q4_G64 or q8_0, two groups of Q4_G32, four NVFP4 blocks)
    constexpr int NLU = C::KRB / 32;
    constexpr int GPU = (KC == KVQ_CODEC_Q4_G32) ? 2 : 1;          // K groups per ldmatrix
    uint32_t koff[NLU];
    {
        const int ktok = tl + (lane & 7) + 8 * ((lane >> 3) & 1), kch = lane >> 4;
#pragma unroll
        for (int u = 0; u < NLU; ++u) koff[u] = KG::chunk_addr(C::K_OFF, ktok, 2 * u + kch);
    }
    // Phase B head_dim slice: 16-row tiles mt = warp * MTW + t; tile mt covers
    // the 16-byte V chunk mt / 2 (32 head_dim values), its rows 0-7 the nibble
    // pair 2 (mt % 2) (even head_dim index), rows 8-15 the pair 2 (mt % 2) + 1
    // (odd index), so a tile never spans two V groups.  The warp's tiles lie in
    // chunks cw and cw1 (= cw when it has at most two tiles).
    // q8_0 V instead: tile t is the 16-byte chunk MTW * warp + t (16 head_dim
    // values), rows 0-7 its even, rows 8-15 its odd head_dim indices; one
    // ldmatrix.x4.trans covers two chunks.
    constexpr bool V8 = (VC == KVQ_CODEC_Q8_0);
    constexpr bool F4V = is_fp4(VC);        // NVFP4 V: Q4's tile layout, exact scaled values
    const int cw = (warp * MTW) >> 1, cw1 = (MTW == 4) ? cw + 1 : cw;
    constexpr int NGW = (MTW == 4 && VC != KVQ_CODEC_Q4_G64 && !F4V) ? 2 : 1;  // V groups a warp's tiles touch
    // V codes as fp16 subnormals with their offset removed per tile (one n-tile)
    constexpr bool kSubV = (NT == 1 && (NGW == 1 || V8)) && !F4V;
    const int gv0 = V8 ? (MTW * warp) / 2 : (32 * cw) / group_size(VC);  // the first of them
    constexpr int NLV = V8 ? (MTW + 1) / 2 : 1;                          // ldmatrix per 16 tokens
    uint32_t voff[NLV];
#pragma unroll
    for (int u = 0; u < NLV; ++u) {
        const int ca = V8 ? MTW * warp + 2 * u : cw, cb = V8 ? (MTW >= 2 ? ca + 1 : ca) : cw1;
        voff[u] = VG::chunk_addr(C::V_OFF, (lane & 7) + 8 * (lane >> 4), ((lane >> 3) & 1) ? cb : ca);
    }
    const uint32_t qp_base = smem_u32(qp), qpl_base = smem_u32(smem + C::QPL_OFF);
    // with one n-tile the query's B fragments fit in registers for the whole CTA
    // (an fp16 query; the two parts of an fp32 one are read from shared memory)
    constexpr bool QLO = C::QLO;
    constexpr bool QREG = (NT == 1) && !QLO;
    constexpr int KSTEPS = D / 16;
    uint32_t qf[QREG ? KSTEPS : 1][2];
    if constexpr (QREG) {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
            ldsm_x2(qp_base + qp_chunk_off<D>(lane & 7, 2 * ks + ((lane >> 3) & 1)), qf[ks][0], qf[ks][1]);
    }

    float o[MTW][NT][4];
#pragma unroll
    for (int t = 0; t < MTW; ++t)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[t][nt][c] = 0.0f;
    // running maximum and (partial) sum of row nt * 8 + gid, the row this lane's
    // phase-B operand fragments belong to; every warp holds the same maxima
    float mg[NT], lg[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mg[nt] = -INFINITY, lg[nt] = 0.0f;

    // ---- phase A of tile jj: S^T for this warp's 16 tokens (log2 units, not yet
    // masked) and the tile's V scales transposed for phase B (0 past the split end)
    auto phase_a = [&](int jj, float (&sc)[NT][4]) {
        const int st = jj % kS;
        const int tb = lo + jj * kTile + tl;
        const uint32_t base = smem_u32(smem + st * C::STAGE);
        const uint8_t *ksp = smem + st * C::STAGE + C::KS_OFF;
        const uint8_t *vsp = smem + st * C::STAGE + C::VS_OFF;
        __half *vt = vt0 + (jj & 1) * (C::NGV * kTile);
        for (int i = lane; i < 16 * C::NGV; i += 32) {
            const int t = i & 15, g = i >> 4;
            __half sv = __float2half_rn(0.0f);
            if (tb + t < hi) {
                if constexpr (is_fp4(VC)) sv = __float2half_rn(e4m3_to_float(vsp[(tl + t) * C::VSB + g]));
                else sv = reinterpret_cast<const __half *>(vsp + (tl + t) * C::VSB)[g];
            }
            vt[g * kTile + tl + t] = sv;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[nt][c] = 0.0f;
        float sk0[NGK], sk1[NGK];
        if constexpr (is_fp4(KC)) {
#pragma unroll
            for (int g = 0; g < NGK; ++g) sk0[g] = sk1[g] = 1.0f;     // the scales go into the operands
        } else {
            load_scales<NGK>(ksp + (tl + gid) * C::KSB, sk0);
            load_scales<NGK>(ksp + (tl + gid + 8) * C::KSB, sk1);
        }
#pragma unroll
        for (int u = 0; u < NLU; ++u) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(base + koff[u], r0, r1, r2, r3);
            uint32_t h0[4], h1[4], h2[4], h3[4];
            if constexpr (is_fp4(KC)) {
                // this lane's 8 values of a chunk are one 16-value block: block
                // 4u + tig / 2 (chunk 2u) and 4u + 2 + tig / 2 (chunk 2u + 1)
                const int ba = 4 * u + (tig >> 1), bb = ba + 2;
                const uint32_t s0a = e4m3_pair(ksp[(tl + gid) * C::KSB + ba]);
                const uint32_t s1a = e4m3_pair(ksp[(tl + gid + 8) * C::KSB + ba]);
                const uint32_t s0b = e4m3_pair(ksp[(tl + gid) * C::KSB + bb]);
                const uint32_t s1b = e4m3_pair(ksp[(tl + gid + 8) * C::KSB + bb]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    h0[e] = fp4_byte_h2(r0, e, s0a);
                    h1[e] = fp4_byte_h2(r1, e, s1a);
                    h2[e] = fp4_byte_h2(r2, e, s0b);
                    h3[e] = fp4_byte_h2(r3, e, s1b);
                }
            } else if constexpr (is_q4(KC)) {
                unpack_q4_biased(r0, h0);
                unpack_q4_biased(r1, h1);
                unpack_q4_biased(r2, h2);
                unpack_q4_biased(r3, h3);
            } else {
                uint32_t t2[2];
                unpack_q8_biased(r0, t2); h0[0] = t2[0]; h0[1] = t2[1];
                unpack_q8_biased(r1, t2); h1[0] = t2[0]; h1[1] = t2[1];
                unpack_q8_biased(r2, t2); h2[0] = t2[0]; h2[1] = t2[1];
                unpack_q8_biased(r3, t2); h3[0] = t2[0]; h3[1] = t2[1];
            }
#pragma unroll
            for (int gi = 0; gi < GPU; ++gi) {
                const int g = u * GPU + gi;
                // each group's accumulator starts at minus its bias term (the first
                // k-step's MMA takes it as its accumulator input)
                float cg[NT][4];
                float2 nb2[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    nb2[nt] = *reinterpret_cast<const float2 *>(kb_s + g * C::ROWS + nt * 8 + 2 * tig);
#pragma unroll
                for (int k = 0; k < KSTEP_PER_G; ++k) {
                    const int ks = g * KSTEP_PER_G + k;
                    // A fragment: Q4_G32 takes both k halves from the group's own chunk
                    // (nibble pairs 2k and 2k + 1); the others take k half 0 from the
                    // first chunk and half 1 from the second
                    uint32_t a0, a1, a2, a3;
                    if constexpr (KC == KVQ_CODEC_Q4_G32) {
                        a0 = gi ? h2[2 * k] : h0[2 * k];
                        a1 = gi ? h3[2 * k] : h1[2 * k];
                        a2 = gi ? h2[2 * k + 1] : h0[2 * k + 1];
                        a3 = gi ? h3[2 * k + 1] : h1[2 * k + 1];
                    } else {
                        a0 = h0[k];
                        a1 = h1[k];
                        a2 = h2[k];
                        a3 = h3[k];
                    }
#pragma unroll
                    for (int np = 0; np < (NT + 1) / 2; ++np) {
                        // B fragments of n-tiles 2np and 2np+1 (the second exists only
                        // when 2np + 1 < NT)
                        uint32_t b00, b01, b10, b11;
                        if constexpr (QREG) {
                            b00 = qf[ks][0];
                            b01 = qf[ks][1];
                            b10 = b11 = 0u;
                        } else if (2 * np + 1 < NT) {
                            const int qrow = (2 * np + (lane >> 4)) * 8 + (lane & 7);
                            ldsm_x4(qp_base + qp_chunk_off<D>(qrow, 2 * ks + ((lane >> 3) & 1)), b00, b01, b10, b11);
                        } else {
                            const int qrow = 2 * np * 8 + (lane & 7);
                            ldsm_x2(qp_base + qp_chunk_off<D>(qrow, 2 * ks + ((lane >> 3) & 1)), b00, b01);
                            b10 = b11 = 0u;
                        }
                        if (k == 0) {
                            const float2 c = nb2[2 * np];
                            mma16816_c(cg[2 * np], a0, a1, a2, a3, b00, b01, c.x, c.y, c.x, c.y);
                            if (2 * np + 1 < NT) {
                                const float2 c1 = nb2[2 * np + 1];
                                mma16816_c(cg[2 * np + 1], a0, a1, a2, a3, b10, b11, c1.x, c1.y, c1.x, c1.y);
                            }
                        } else {
                            mma16816(cg[2 * np], a0, a1, a2, a3, b00, b01);
                            if (2 * np + 1 < NT) mma16816(cg[2 * np + 1], a0, a1, a2, a3, b10, b11);
                        }
                        if constexpr (QLO) {
                            // the low part of an fp32 query, into the same accumulators
                            if (2 * np + 1 < NT) {
                                const int qrow = (2 * np + (lane >> 4)) * 8 + (lane & 7);
                                ldsm_x4(qpl_base + qp_chunk_off<D>(qrow, 2 * ks + ((lane >> 3) & 1)), b00, b01, b10,
                                        b11);
                                mma16816(cg[2 * np], a0, a1, a2, a3, b00, b01);
                                mma16816(cg[2 * np + 1], a0, a1, a2, a3, b10, b11);
                            } else {
                                const int qrow = 2 * np * 8 + (lane & 7);
                                ldsm_x2(qpl_base + qp_chunk_off<D>(qrow, 2 * ks + ((lane >> 3) & 1)), b00, b01);
                                mma16816(cg[2 * np], a0, a1, a2, a3, b00, b01);
                            }
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    sc[nt][0] = fmaf(cg[nt][0], sk0[g], sc[nt][0]);
                    sc[nt][1] = fmaf(cg[nt][1], sk0[g], sc[nt][1]);
                    sc[nt][2] = fmaf(cg[nt][2], sk1[g], sc[nt][2]);
                    sc[nt][3] = fmaf(cg[nt][3], sk1[g], sc[nt][3]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[nt][c] *= sl2;
    };

    // ---- end of phase A: mask (split end, causal rows), store the scores and
    // this warp's per-row maximum of the tile for phase B
    auto phase_a_store = [&](int jj, float (&sc)[NT][4]) {
        const int tb = lo + jj * kTile + tl;
        const int ta = tb + gid, tc = ta + 8;
        if (tb + 16 > hi || tb + 16 > nv_min) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (!(ta < hi && ta < nv[nt][0])) sc[nt][0] = -INFINITY;
                if (!(ta < hi && ta < nv[nt][1])) sc[nt][1] = -INFINITY;
                if (!(tc < hi && tc < nv[nt][0])) sc[nt][2] = -INFINITY;
                if (!(tc < hi && tc < nv[nt][1])) sc[nt][3] = -INFINITY;
            }
        }
        float *s_s = s_s0 + (jj & 1) * (kTile * C::PS);
        float *red_m = red_m0 + (jj & 1) * (kW * 32);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            *reinterpret_cast<float2 *>(s_s + (tl + gid) * C::PS + nt * 8 + 2 * tig) = make_float2(sc[nt][0], sc[nt][1]);
            *reinterpret_cast<float2 *>(s_s + (tl + gid + 8) * C::PS + nt * 8 + 2 * tig) =
                make_float2(sc[nt][2], sc[nt][3]);
            float mx0 = fmaxf(sc[nt][0], sc[nt][2]), mx1 = fmaxf(sc[nt][1], sc[nt][3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            if (gid == 0) *reinterpret_cast<float2 *>(red_m + warp * 32 + nt * 8 + 2 * tig) = make_float2(mx0, mx1);
        }
    };

    // ---- phase B of tile jj: softmax of the tile and O^T += V^T P'^T for this
    // warp's head_dim slice
    auto phase_b = [&](int jj) {
        const int st = jj % kS;
        const uint32_t base = smem_u32(smem + st * C::STAGE);
        const float *s_s = s_s0 + (jj & 1) * (kTile * C::PS);
        const float *red_m = red_m0 + (jj & 1) * (kW * 32);
        const __half *vt = vt0 + (jj & 1) * (C::NGV * kTile);
        // new running maximum of row nt * 8 + gid (the same in every warp)
        float cf[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = nt * 8 + gid;
            float tmax = red_m[r];
#pragma unroll
            for (int w = 1; w < kW; ++w) tmax = fmaxf(tmax, red_m[w * 32 + r]);
            const float mn = fmaxf(mg[nt], tmax);
            cf[nt] = (mn == -INFINITY) ? 1.0f : ex2(mg[nt] - mn);
            mg[nt] = mn;
            lg[nt] *= cf[nt];
        }
        // accumulator columns are rows 2 tig and 2 tig + 1: their factors come from
        // the lanes whose fragment row they are (1 unless the maximum grew)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float c0 = __shfl_sync(0xffffffffu, cf[nt], 8 * tig);
            const float c1 = __shfl_sync(0xffffffffu, cf[nt], 8 * tig + 4);
#pragma unroll
            for (int t = 0; t < MTW; ++t) {
                o[t][nt][0] *= c0;
                o[t][nt][1] *= c1;
                o[t][nt][2] *= c0;
                o[t][nt][3] *= c1;
            }
        }
        float msub[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) msub[nt] = (mg[nt] == -INFINITY) ? 0.0f : mg[nt];
        // sum over the tile's tokens of P' per row (the same in all 16 accumulator
        // rows), one per V group the warp touches, for removing the codes' offset
        // (subnormal form only)
        float psum[NGW][NT][4];
#pragma unroll
        for (int q = 0; q < NGW; ++q)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) psum[q][nt][c] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
            // tokens past the split end have score -inf (p = 0) and V scale 0
            // tokens 0-7 of chunks a, b, tokens 8-15 of chunks a, b
            uint32_t rv[NLV][4];
#pragma unroll
            for (int u = 0; u < NLV; ++u)
                ldsm_x4_t(base + voff[u] + (uint32_t)(16 * kk * VG::BI), rv[u][0], rv[u][1], rv[u][2], rv[u][3]);
            float p[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float *sr = s_s + (16 * kk + 2 * tig) * C::PS + nt * 8 + gid;
                p[nt][0] = ex2(sr[0] - msub[nt]);
                p[nt][1] = ex2(sr[C::PS] - msub[nt]);
                p[nt][2] = ex2(sr[8 * C::PS] - msub[nt]);
                p[nt][3] = ex2(sr[9 * C::PS] - msub[nt]);
                lg[nt] += (p[nt][0] + p[nt][1]) + (p[nt][2] + p[nt][3]);
            }
            // P' = p * v_scale(token, group), one B fragment set per V group
            // (NVFP4: P' = p, the scales are in the V operands)
            uint32_t b0[NGW][NT], b1[NGW][NT];
            if constexpr (F4V) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    b0[0][nt] = pack_f16x2(p[nt][0], p[nt][1]);
                    b1[0][nt] = pack_f16x2(p[nt][2], p[nt][3]);
                }
            }
#pragma unroll
            for (int q = 0; q < NGW && !F4V; ++q) {
                const __half *vq = vt + (gv0 + q) * kTile + 16 * kk + 2 * tig;
                const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(vq));
                const float2 s89 = __half22float2(*reinterpret_cast<const __half2 *>(vq + 8));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    b0[q][nt] = pack_f16x2(p[nt][0] * s01.x, p[nt][1] * s01.y);
                    b1[q][nt] = pack_f16x2(p[nt][2] * s89.x, p[nt][3] * s89.y);
                }
            }
#pragma unroll
            for (int t = 0; t < MTW; ++t) {
                const int q = (NGW == 2) ? (t >> 1) : 0;
                uint32_t a0, a1, a2, a3;
                if constexpr (V8) {
                    // tile t: load t / 2, chunk a or b by t's parity
                    const int u = t >> 1;
                    const bool b = (MTW >= 2) && (t & 1);
                    const uint32_t ra = b ? rv[u][1] : rv[u][0], rb = b ? rv[u][3] : rv[u][2];
                    if constexpr (kSubV) {
                        q8_pairs_sub(ra, a0, a1);
                        q8_pairs_sub(rb, a2, a3);
                    } else {
                        q8_pairs(ra, a0, a1);
                        q8_pairs(rb, a2, a3);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816(o[t][nt], a0, a1, a2, a3, b0[q][nt], b1[q][nt]);
                    continue;
                }
                // tile t: chunk cw + lc, nibble pairs 2j (rows 0-7) and 2j + 1 (rows 8-15)
                const int lc = (MTW >= 2) ? (t >> 1) : 0;
                const int j = (MTW >= 2) ? (t & 1) : (warp & 1);
                const uint32_t ra = lc ? rv[0][1] : rv[0][0], rb = lc ? rv[0][3] : rv[0][2];
                if constexpr (F4V) {
                    // the lane's head_dim values 32 c + 4 gid + e lie in block 2 c + gid / 4;
                    // the scales of tokens (2 tig, 2 tig + 1) and (2 tig + 8, 2 tig + 9)
                    const __half *vq = vt + (2 * (cw + lc) + (gid >> 2)) * kTile + 16 * kk + 2 * tig;
                    const uint32_t s01 = *reinterpret_cast<const uint32_t *>(vq);
                    const uint32_t s89 = *reinterpret_cast<const uint32_t *>(vq + 8);
                    a0 = fp4_pair(ra, 2 * j, s01); a1 = fp4_pair(ra, 2 * j + 1, s01);
                    a2 = fp4_pair(rb, 2 * j, s89); a3 = fp4_pair(rb, 2 * j + 1, s89);
                } else if constexpr (kSubV) {
                    a0 = q4_pair_sub(ra, 2 * j); a1 = q4_pair_sub(ra, 2 * j + 1);
                    a2 = q4_pair_sub(rb, 2 * j); a3 = q4_pair_sub(rb, 2 * j + 1);
                } else {
                    a0 = q4_pair(ra, 2 * j); a1 = q4_pair(ra, 2 * j + 1);
                    a2 = q4_pair(rb, 2 * j); a3 = q4_pair(rb, 2 * j + 1);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(o[t][nt], a0, a1, a2, a3, b0[q][nt], b1[q][nt]);
            }
            if constexpr (kSubV) {
                constexpr uint32_t kOnes = 0x3C003C00u;             // fp16x2 (1, 1)
#pragma unroll
                for (int q = 0; q < NGW; ++q)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(psum[q][nt], kOnes, kOnes, kOnes, kOnes, b0[q][nt], b1[q][nt]);
            }
        }
        // remove the offset: Q4 8 * 2^-24 per P' on rows 0-7 (even head_dim
        // index), 128 * 2^-24 on rows 8-15 (odd index); q8_0 128 * 2^-24
#pragma unroll
        for (int t = 0; kSubV && t < MTW; ++t) {
            const int q = (NGW == 2) ? (t >> 1) : 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    o[t][nt][c] = fmaf((c < 2 && !V8) ? -0x1p-21f : -0x1p-17f, psum[q][nt][c], o[t][nt][c]);
        }
    };

    if constexpr (NT == 1) {
        // Software-pipelined tile loop: iteration j runs phase A of tile j + 1 and
        // phase B of tile j, two independent instruction streams in one block (the
        // scores, maxima and transposed V scales are double-buffered by tile
        // parity), then the one CTA barrier, which also orders every warp's reads
        // of tile j before its stage is refilled with tile j + kS.  The last
        // tile's phase B runs alone.  After a timeout the waits are skipped and
        // the warps keep stepping over stale data (the result is flagged as
        // invalid), so every warp reaches every barrier.
        if (n_tiles > 0) {
            if (!s_timeout && !mbar_wait(bar_full, 0)) s_timeout = 1;
            float sc[NT][4];
            phase_a(0, sc);
            phase_a_store(0, sc);
        }
        warps_sync();
        for (int j = 0; j + 1 < n_tiles; ++j) {
            if (!s_timeout && !mbar_wait(bar_full + 8 * ((j + 1) % kS), ((j + 1) / kS) & 1)) s_timeout = 1;
            float sc[NT][4];
            phase_a(j + 1, sc);
            phase_b(j);
            phase_a_store(j + 1, sc);
            warps_sync();
            if (threadIdx.x == 0 && !s_timeout && j + kS < n_tiles) {
                issue_tile<C, KG, VG>(smem_u32(smem + (j % kS) * C::STAGE), bar_full + 8 * (j % kS), &tmk, &tmv, ksc,
                                      vsc, plane_row + lo + (j + kS) * kTile);
                s_issued = j + kS + 1;
            }
        }
        if (n_tiles > 0) phase_b(n_tiles - 1);
    } else {
        // Several n-tiles: registers do not allow both phases at once.  Per tile:
        // phase A, the one CTA barrier (which also orders every warp's reads of
        // tile j - 1 before that stage is refilled with tile j - 1 + kS), phase B.
        for (int j = 0; j < n_tiles; ++j) {
            if (!s_timeout && !mbar_wait(bar_full + 8 * (j % kS), (j / kS) & 1)) s_timeout = 1;
            float sc[NT][4];
            phase_a(j, sc);
            phase_a_store(j, sc);
            warps_sync();
            if (threadIdx.x == 0 && j >= 1 && !s_timeout && j - 1 + kS < n_tiles) {
                issue_tile<C, KG, VG>(smem_u32(smem + ((j - 1) % kS) * C::STAGE), bar_full + 8 * ((j - 1) % kS), &tmk,
                                      &tmv, ksc, vsc, plane_row + lo + (j - 1 + kS) * kTile);
                s_issued = j - 1 + kS + 1;
            }
            phase_b(j);
        }
    }
    // the dependent launch (the merge of the splits) may start now: its CTAs
    // find the SMs that finishing CTAs of this grid leave free
    pdl_trigger();

    // row sums: each lane summed a quarter of the tokens of its fragment row
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        lg[nt] += __shfl_xor_sync(0xffffffffu, lg[nt], 1);
        lg[nt] += __shfl_xor_sync(0xffffffffu, lg[nt], 2);
    }
    // never leave while a copy into this CTA's shared memory could be in flight
    // (only possible after a timeout; otherwise every issued copy was waited on)
    if (threadIdx.x == 0 && s_timeout) {
        const int issued = s_issued;
        for (int j = issued - 1; j >= 0 && j >= issued - kS; --j) mbar_wait(bar_full + 8 * (j % kS), (j / kS) & 1);
        mbar_wait(bar_q, 0);
    }
    const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int cl = 0; cl < 2; ++cl) {
            // accumulator column 2 tig + cl (elements cl and cl + 2 of a tile): its sum
            // and maximum sit in the lanes whose fragment row it is
            const float L = __shfl_sync(0xffffffffu, lg[nt], 8 * tig + 4 * cl);
            const float M = __shfl_sync(0xffffffffu, mg[nt], 8 * tig + 4 * cl);
            const int n = nt * 8 + 2 * tig + cl;
            if (n >= R) continue;
            const bool empty = (M == -INFINITY || L <= 0.0f);
            // the V codes entered as q 2^-24 or q (even head_dim index) and, for the
            // 4-bit codecs, 16 times that (odd)
            const float inv = empty ? 0.0f : (kSubV ? 0x1p24f : 1.0f) / L;
            const float inv16 = (V8 || F4V) ? inv : inv * 0.0625f;
            const int i = (r0 + n) / G, jj = (r0 + n) % G;
            const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + jj;
            float *dst = (a.n_splits == 1) ? a.out + orow * D : a.part_o + ((int64_t)split * rows_total + orow) * D;
            if constexpr (V8) {
                // tile t: head_dim 16 (MTW warp + t) + 2 gid (+ 1)
#pragma unroll
                for (int t = 0; t < MTW; ++t)
                    *reinterpret_cast<float2 *>(dst + 16 * (MTW * warp + t) + 2 * gid) =
                        make_float2(o[t][nt][cl] * inv, o[t][nt][cl + 2] * inv16);
            } else if constexpr (MTW >= 2) {
                // tiles 2 lc and 2 lc + 1 fill head_dim 32 (cw + lc) + 4 gid + 0..3
#pragma unroll
                for (int lc = 0; lc < MTW / 2; ++lc)
                    *reinterpret_cast<float4 *>(dst + 32 * (cw + lc) + 4 * gid) =
                        make_float4(o[2 * lc][nt][cl] * inv, o[2 * lc][nt][cl + 2] * inv16,
                                    o[2 * lc + 1][nt][cl] * inv, o[2 * lc + 1][nt][cl + 2] * inv16);
            } else {
                *reinterpret_cast<float2 *>(dst + 32 * cw + 4 * gid + 2 * (warp & 1)) =
                    make_float2(o[0][nt][cl] * inv, o[0][nt][cl + 2] * inv16);
            }
            if (warp == 0 && gid == 0) {
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Kernel attributes (dynamic shared memory, carveout), set once per device, and
// the CTAs per SM they allow.
template <typename C, typename Kern>
cudaError_t prepare_kernel(Kern kern, int *per_sm)
{
    static PerDevice pd;                     // per device; set once, thread-safe
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int n = per_device(pd, dev, [&]() -> int {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        r = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (r != cudaSuccess) return -(int)r;
        int v = 0;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kT, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        return v > 0 ? v : -(int)cudaErrorInvalidConfiguration;
    });
    if (n <= 0) return (cudaError_t)(-n);
    *per_sm = n;
    return cudaSuccess;
}

template <typename C, typename Kern>
cudaError_t launch_cfg(Kern kern, const DecodeArgs &a, cudaStream_t st)
{
    static_assert(C::SMEM <= 227 * 1024, "shared memory of one CTA");
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    CUtensorMap tk, tv;
    if (!make_codes_map(&tk, a.k.qs, C::KRB, rows, kTile) || !make_codes_map(&tv, a.v.qs, C::VRB, rows, kTile))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaError_t e = prepare_kernel<C>(kern, &per_sm);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_splits, a.n_kv_heads * a.n_row_blocks, a.n_seq);
    return launch_pdl(kern, grid, dim3(kT), C::SMEM, st, a, tk, tv);
}

template <int KC, int VC, int D>
int per_sm_nt(int nt)
{
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (nt) {
    case 1: e = prepare_kernel<TcCfg<KC, VC, D, 1, __half>>(decode_tc_kernel<KC, VC, D, 1, __half>, &n); break;
    case 2: e = prepare_kernel<TcCfg<KC, VC, D, 2, __half>>(decode_tc_kernel<KC, VC, D, 2, __half>, &n); break;
    case 3: e = prepare_kernel<TcCfg<KC, VC, D, 3, __half>>(decode_tc_kernel<KC, VC, D, 3, __half>, &n); break;
    case 4: e = prepare_kernel<TcCfg<KC, VC, D, 4, __half>>(decode_tc_kernel<KC, VC, D, 4, __half>, &n); break;
    default: break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int KC, int VC>
int per_sm_d(int head_dim, int nt)
{
    switch (head_dim) {
    case 64: return per_sm_nt<KC, VC, 64>(nt);
    case 128: return per_sm_nt<KC, VC, 128>(nt);
    case 256: return per_sm_nt<KC, VC, 256>(nt);
    default: return 0;
    }
}

template <int KC, int VC, int D, int NT, typename QT>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t st)
{
    return launch_cfg<TcCfg<KC, VC, D, NT, QT>>(decode_tc_kernel<KC, VC, D, NT, QT>, a, st);
}

template <int KC, int VC, int D, typename QT>
cudaError_t launch_nt(const DecodeArgs &a, cudaStream_t st)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    switch (R > 32 ? 4 : (R + 7) / 8) {
    case 1: return launch_t<KC, VC, D, 1, QT>(a, st);
    case 2: return launch_t<KC, VC, D, 2, QT>(a, st);
    case 3: return launch_t<KC, VC, D, 3, QT>(a, st);
    case 4: return launch_t<KC, VC, D, 4, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int KC, int VC, typename QT>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st)
{
    switch (a.head_dim) {
    case 64: return launch_nt<KC, VC, 64, QT>(a, st);
    case 128: return launch_nt<KC, VC, 128, QT>(a, st);
    case 256: return launch_nt<KC, VC, 256, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int VC, typename QT>
cudaError_t launch_k(const DecodeArgs &a, cudaStream_t st)
{
    switch (a.k.codec) {
    case KVQ_CODEC_Q4_G64: return launch_d<KVQ_CODEC_Q4_G64, VC, QT>(a, st);
    case KVQ_CODEC_Q8_0: return launch_d<KVQ_CODEC_Q8_0, VC, QT>(a, st);
    case KVQ_CODEC_Q4_G32: return launch_d<KVQ_CODEC_Q4_G32, VC, QT>(a, st);
    case KVQ_CODEC_NVFP4: return launch_d<KVQ_CODEC_NVFP4, VC, QT>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

// The kernel for V in codec VC: launch, and CTAs per SM for a K codec.
template <int VC>
cudaError_t launch_for_v(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    return q_dtype == KVQ_F16 ? launch_k<VC, __half>(a, st) : launch_k<VC, float>(a, st);
}

template <int VC>
int per_sm_for_v(int k_codec, int head_dim, int nt)
{
    switch (k_codec) {
    case KVQ_CODEC_Q4_G64: return per_sm_d<KVQ_CODEC_Q4_G64, VC>(head_dim, nt);
    case KVQ_CODEC_Q8_0: return per_sm_d<KVQ_CODEC_Q8_0, VC>(head_dim, nt);
    case KVQ_CODEC_Q4_G32: return per_sm_d<KVQ_CODEC_Q4_G32, VC>(head_dim, nt);
    case KVQ_CODEC_NVFP4: return per_sm_d<KVQ_CODEC_NVFP4, VC>(head_dim, nt);
    default: return 0;
    }
}

}  // namespace
}  // namespace kvq
