// kvq_decode_warp.cu -- split-K decode attention for up to 8 query rows per
// kv head (a GQA group of one token, or 1 + k MTP tokens of a narrow group)
// over a Q4_G64 V plane with a Q4_G64 or q8_0 K plane, or the q8_0 K / Q4_G32 V
// pair: one CTA of 12 warps per SM, each warp owning whole blocks of 16 tokens
// over all of head_dim.  (den_llama.cpp, "What's in the fork": the fattn-vec
// Q4_G64 instances; "What this fork is": 4-bit signed codes sharing one fp16
// scale per 64 values, the q8_0 K / Q4_G64 V pair, and the q8_0 K / q4_0 V
// FlashAttention pair, q4_0 read as 4-bit codes with a scale per 32 values.)
//
// Per (sequence, kv head, split) the split's tokens are cut into blocks of 16
// and each warp takes a contiguous run of them, streamed through its own ring
// of two shared-memory stages (K and V codes by 2D TMA, 32 rows a box for
// 4-bit K after a first stage of 16, 16 for q8_0 K, whose rows take two
// 128-byte boxes; the fp16 scales by bulk copies).  Each warp keeps its own
// online-softmax state, so nothing in the loop waits on another warp.  Per
// block the warp:
//  * computes S^T = K Q^T (tokens on M, query rows on N) on mma.sync.m16n8k16:
//    the K codes enter as exact fp16 integers with their bias (4-bit: 1032 + q,
//    or 1152 + 16 q at odd head_dim indices, one LOP3 per two values; q8_0:
//    1152 + q, one PRMT per two values), each scale group in its own
//    accumulator that starts at minus the group's bias term and is then
//    scaled by the token's fp16 scale in fp32;
//  * takes the block's per-row maximum with three shuffles and forms
//    p = 2^(s - m) against a running reference m that is raised (with O and
//    the sums rescaled) only when a block's maximum passes it by more than 2^8,
//    or by anything while a V scale of the block is 256 or more, so P' below
//    stays a finite fp16 value;
//  * forms P' = p * v_scale(token, group) in fp32, rounds it once to fp16 and
//    transposes the 8x8 fp16 fragments with movmatrix into the B operand of
//    O^T += V^T P'^T (so every exponential is computed once and no score goes
//    through shared memory);
//  * accumulates O^T over all of head_dim: V^T fragments from ldmatrix.trans
//    (two tokens at one head_dim index), the V codes as exact fp16 subnormals
//    (q + 8) 2^-24 (16 (q + 8) 2^-24 at odd indices), one LOP3 per two values;
//    the offset 8 is removed at the end from the sum of P' per group, which
//    one MMA against an all-ones operand accumulates per block.
// At the end each warp leaves its (reference, sum, sums of P', raw O^T) in
// shared memory (O^T over its own K ring), and after one barrier every thread
// forms whole outputs of the CTA: its normalised result (one split) or its
// partial with the log-sum-exp for the merge kernel.
//
// Every mbarrier wait is bounded: after ~1 s the warp stops waiting, the CTA
// sets KVQ_ERR_TIMEOUT in the caller's error word and finishes; nothing traps.
#include "kvq_decode_common.cuh"

namespace kvq {
using namespace ptx;
namespace {

constexpr int kBlk = 16;            // tokens per warp block (one MMA row tile)
constexpr int kWW = 12;             // warps per CTA
constexpr int kWMinBlocks = 1;      // CTAs per SM
constexpr int kWS = 2;              // ring stages per warp
constexpr int kWRows = 8;           // query rows per kv head (one n-tile)

template <int KC, int VC, int D, typename QT>
struct WCfg {
    static constexpr int NGK = D / group_size(KC);    // K scale groups per row
    static constexpr int VGS = group_size(VC);        // V (4-bit) scale group: 64 or 32 values
    static constexpr int NGV = D / VGS;               // V scale groups per row
    static constexpr int NCP = D / 64;                // V chunk pairs per row (one ldmatrix.trans each)
    static constexpr int KRB = row_bytes(KC, D);      // code bytes per row
    static constexpr int VRB = D / 2;
    static constexpr int KBI = KRB < 128 ? KRB : 128; // K box width (bytes); K rows of 256 bytes take two boxes
    static constexpr int KNB = KRB / KBI;
    static constexpr int KSTEPS_G = group_size(KC) / 16;                // MMA k-steps per K group
    // blocks per ring stage: two (one copy of 32 rows) for 4-bit K, one for
    // q8_0 K, whose stages are twice as large
    static constexpr int SBLK = KC == KVQ_CODEC_Q8_0 ? 1 : 2;
    static constexpr int ST = SBLK * kBlk;           // rows per stage
    static constexpr int CBK = ST * KRB, CBV = ST * VRB;               // code bytes of a stage
    static constexpr int SBKB = kBlk * NGK * 2, SBVB = kBlk * NGV * 2;  // scale bytes of a block
    static constexpr int SBK = SBLK * SBKB, SBV = SBLK * SBVB;
    static constexpr int NSLOT = kWW * kWS;
    static constexpr int NTH = kWW * 32;
    static constexpr bool QLO = sizeof(QT) == 4;      // fp32 query: hi + lo fp16 parts
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + NSLOT * CBK;
    static constexpr int KS_OFF = V_OFF + NSLOT * CBV;
    static constexpr int VS_OFF = KS_OFF + NSLOT * SBK;
    static constexpr int QP_OFF = align_up(VS_OFF + NSLOT * SBV, 128);  // fp16 [8][D] permuted, swizzled
    static constexpr int QPL_OFF = QP_OFF + kWRows * D * 2;            // its low part (fp32 query)
    static constexpr int KB_OFF = QPL_OFF + (QLO ? kWRows * D * 2 : 0);  // fp32 [NGK][8] minus the K bias terms
    // the same as accumulator inputs, [NGK][tig][4] = (row 2 tig, 2 tig + 1, 2 tig, 2 tig + 1)
    static constexpr int KBD_OFF = KB_OFF + align_up(NGK * kWRows * 4, 16);
    static constexpr int QST_OFF = KBD_OFF + NGK * 64;                  // the query rows as given
    static constexpr int RED_OFF = QST_OFF + kWRows * D * (int)sizeof(QT);   // fp32 [kWW][16]: m, l per row
    static constexpr int PSR_OFF = RED_OFF + kWW * 16 * 4;                   // fp32 [kWW][NGV][8]: sums of P'
    static constexpr int BAR_OFF = align_up(PSR_OFF + kWW * NGV * 8 * 4, 16);
    static constexpr int SMEM = BAR_OFF + (NSLOT + 1) * 8 + 1024;           // + alignment slack
    // each warp's O for the combine, fp32 [8][D], over its own K ring (which
    // no other warp touches, so it may write while the others still stream)
    static_assert(kWRows * D * 4 == kWS * CBK, "a warp's O fills its K ring");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// NG fp16 scales (NG = 1, 2, 4 or 8) at a shared address as raw words
template <int NG>
__device__ __forceinline__ void lds_scales(uint32_t addr, uint32_t (&w)[(NG + 1) / 2])
{
    if constexpr (NG == 8) {
        const uint4 v = lds128(addr);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else if constexpr (NG == 4) {
        const uint2 v = lds64(addr);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        w[0] = lds32(addr & ~3u);
        if constexpr (NG == 1) w[0] = (addr & 2u) ? (w[0] >> 16) : (w[0] & 0xFFFFu);
    }
}

template <int NG>
__device__ __forceinline__ void scales_to_float(const uint32_t (&w)[(NG + 1) / 2], float (&f)[NG])
{
#pragma unroll
    for (int g = 0; g < NG; ++g)
        f[g] = __half2float(__ushort_as_half((unsigned short)((g & 1) ? (w[g >> 1] >> 16) : (w[g >> 1] & 0xFFFFu))));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <int KC, int VC, int D, typename QT>
__global__ void __launch_bounds__(kWW * 32, kWMinBlocks)
decode_warp_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmk1, const __grid_constant__ CUtensorMap tmv1)
{
    using C = WCfg<KC, VC, D, QT>;
    constexpr int NGK = C::NGK, NGV = C::NGV, NCP = C::NCP;
    constexpr bool G32V = (VC == KVQ_CODEC_Q4_G32);
    constexpr bool K8 = (KC == KVQ_CODEC_Q8_0);
    using KG = TileGeom<C::KBI>;
    using VG = TileGeom<C::VRB>;

    // the base rounded up to 1024 bytes by pointer arithmetic on the shared
    // array, so that every access below stays a shared-memory access
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t bars = smem_u32(smem + C::BAR_OFF);          // [kWW][kWS], then the query's
    const uint32_t bar_q = bars + C::NSLOT * 8;
    float *kb_s = reinterpret_cast<float *>(smem + C::KB_OFF);
    float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
    float *psr = reinterpret_cast<float *>(smem + C::PSR_OFF);
    constexpr int kSBlk = C::SBLK;
    __shared__ int s_seq;
    __shared__ int s_timeout;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int split = blockIdx.x, kh = blockIdx.y;
    const int G = a.n_heads / a.n_kv_heads;
    const int R = a.n_q * G;                                    // <= 8
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        if constexpr (C::SBLK > 1) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk1)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv1)) : "memory");
        }
        s_timeout = 0;
        for (int i = 0; i <= C::NSLOT; ++i) mbar_init(bars + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait();
    // The grid's z index is a rank: sequences in order of decreasing length, so
    // the CTAs of the longest sequences of a ragged batch are dispatched first.
    int s = blockIdx.z;
    if (a.n_seq > 1 && a.n_seq <= C::NTH) {
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
    // the query rows of this kv head (row r: head r % G of token r / G), one
    // bulk copy per token, in parallel with what follows
    if (threadIdx.x == 0) {
        const uint32_t row = (uint32_t)(D * sizeof(QT));
        mbar_expect_tx(bar_q, row * (uint32_t)R);
        const QT *q = static_cast<const QT *>(a.q);
        for (int i = 0; i < a.n_q; ++i)
            bulk_load(smem_u32(smem + C::QST_OFF) + (uint32_t)(i * G) * row,
                      q + (((int64_t)s * a.n_q + i) * a.n_heads + kh * G) * D, (uint32_t)G * row, bar_q);
    }

    int len = a.fixed_len >= 0 ? a.fixed_len : a.kv_len[s];
    if (len < 0 || len > a.max_kv_len) {
        if (threadIdx.x == 0 && split == 0 && kh == 0 && a.err) atomicOr(a.err, KVQ_ERR_KV_LEN);
        len = len < 0 ? 0 : a.max_kv_len;
    }
    int lo, hi;
    split_range(len, a.n_splits, split, lo, hi);
    // this warp's blocks: a contiguous run [wb0, wb0 + my_nb) of the split's
    // 16-token blocks.  The run's first ring stage holds one block, every later
    // one kSBlk (the last the remainder): the whole grid issues its first
    // copies at once, and a smaller first copy lands sooner, so the warps start
    // computing while the rest of that wave is still arriving.
    const int nb = (int)ceil_div(hi - lo, kBlk);
    const int wb0 = (warp * nb) / kWW;
    const int my_nb = ((warp + 1) * nb) / kWW - wb0;
    const int n_st = my_nb > 0 ? 1 + (my_nb + kSBlk - 2) / kSBlk : 0;
    auto stage_blocks = [&](int j) { return j == 0 ? 1 : min(kSBlk, my_nb - 1 - kSBlk * (j - 1)); };
    const int64_t plane_row = ((int64_t)s * a.n_kv_heads + kh) * a.capacity;
    const uint8_t *ksc = reinterpret_cast<const uint8_t *>(a.k.sc);
    const uint8_t *vsc = reinterpret_cast<const uint8_t *>(a.v.sc);
    const uint32_t slot0 = (uint32_t)warp * kWS;
    const uint32_t k_ring = smem_u32(smem + C::K_OFF) + slot0 * C::CBK;    // this warp's stages
    const uint32_t v_ring = smem_u32(smem + C::V_OFF) + slot0 * C::CBV;
    const uint32_t ks_ring = smem_u32(smem + C::KS_OFF) + slot0 * C::SBK;
    const uint32_t vs_ring = smem_u32(smem + C::VS_OFF) + slot0 * C::SBV;
    const uint32_t bar_ring = bars + 8 * slot0;

    // lane 0 fills (and refills) the warp's stages in order; the cache is read
    // once per call, so evict-first in L2.  A stage's codes are one box of
    // kSBlk * 16 rows per plane (two side by side for 256-byte K rows), a box
    // of 16 rows (maps tmk1, tmv1) for a stage of one block; the scales are
    // copied for the blocks the stage holds.
    int n_issued = 0, iss_slot = 0;
    int iss_row = (int)(plane_row + lo) + kBlk * wb0;      // the next stage's first plane row
    const uint64_t pol = evict_first_policy();
    auto issue = [&]() {
        const uint32_t bar = bar_ring + 8 * (uint32_t)iss_slot;
        const uint32_t nbl = (uint32_t)stage_blocks(n_issued);
        const bool full = (nbl == (uint32_t)kSBlk);
        const CUtensorMap *mk = full ? &tmk : &tmk1, *mv = full ? &tmv : &tmv1;
        mbar_expect_tx(bar, nbl * (uint32_t)(kBlk * (C::KRB + C::VRB) + C::SBKB + C::SBVB));
#pragma unroll
        for (int bx = 0; bx < C::KNB; ++bx)
            tma_load_2d(k_ring + (uint32_t)iss_slot * C::CBK + (uint32_t)(bx * C::ST * C::KBI), mk, bx * C::KBI,
                        iss_row, bar, pol);
        tma_load_2d(v_ring + (uint32_t)iss_slot * C::CBV, mv, 0, iss_row, bar, pol);
        bulk_load_hint(ks_ring + (uint32_t)iss_slot * C::SBK, ksc + (int64_t)iss_row * (NGK * 2), nbl * C::SBKB, bar,
                       pol);
        bulk_load_hint(vs_ring + (uint32_t)iss_slot * C::SBV, vsc + (int64_t)iss_row * (NGV * 2), nbl * C::SBVB, bar,
                       pol);
        ++n_issued;
        iss_row += kBlk * (int)nbl;
        iss_slot = (iss_slot + 1 == kWS) ? 0 : iss_slot + 1;
    };
    // each warp's first stage now, its second after the query preparation (an
    // issuing lane waits while the copy engine takes its requests)
    if (lane == 0 && n_st > 0) issue();

    // the query rows, permuted and swizzled, and the K bias terms
    // (the same answer in every thread, so the warps' loops stay uniform)
    const bool q_ok = __syncthreads_and(mbar_wait(bar_q, 0)) != 0;
    if (!q_ok && threadIdx.x == 0) s_timeout = 1;
    prep_query<KC, D, kWRows, C::NTH>(reinterpret_cast<const QT *>(smem + C::QST_OFF),
                                                     smem + C::QP_OFF, smem + C::QPL_OFF, kb_s, R, q_ok);
    __syncthreads();
    if (lane == 0 && n_st > 1) issue();
    if constexpr (K8) {
        // accumulator inputs of the K groups' first MMAs in C-fragment order
        float *kbd = reinterpret_cast<float *>(smem + C::KBD_OFF);
        for (int i = threadIdx.x; i < NGK * 16; i += C::NTH) {
            const int g = i >> 4, t = (i >> 2) & 3, c = i & 3;
            kbd[i] = kb_s[g * kWRows + 2 * t + (c & 1)];
        }
        __syncthreads();
    }

    // rows 2 tig and 2 tig + 1 of this lane's accumulator columns: visible keys
    // (padding rows see everything; their results are never written)
    int nv0, nv1;
    {
        const int r0 = 2 * tig, r1 = r0 + 1;
        nv0 = r0 < R ? len + a.causal_extra - a.n_q + r0 / G + 1 : 0x7FFFFFFF;
        nv1 = r1 < R ? len + a.causal_extra - a.n_q + r1 / G + 1 : 0x7FFFFFFF;
    }
    const int nv_all = len + a.causal_extra - a.n_q + 1;           // the fewest any row sees
    const float sl2 = a.scale_log2;
    // accumulator inputs of each group's first K MMA (minus the bias terms of
    // rows 2 tig, 2 tig + 1, in the C-fragment order; 4-bit K: four registers per
    // group; q8_0 K, with twice the groups, reads them from shared memory), and
    // the all-ones A operand: made distinct registers so that they stay in place
    constexpr int NKBV = K8 ? 1 : NGK;
    float kbv[NKBV][4];
#pragma unroll
    for (int g = 0; g < NKBV; ++g) {
        const float2 b = *reinterpret_cast<const float2 *>(kb_s + g * kWRows + 2 * tig);
        asm volatile("mov.b32 %0, %1;" : "=f"(kbv[g][0]) : "f"(b.x));
        asm volatile("mov.b32 %0, %1;" : "=f"(kbv[g][1]) : "f"(b.y));
        asm volatile("mov.b32 %0, %1;" : "=f"(kbv[g][2]) : "f"(b.x));
        asm volatile("mov.b32 %0, %1;" : "=f"(kbv[g][3]) : "f"(b.y));
    }
    uint32_t ones[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) asm volatile("mov.b32 %0, 0x3C003C00;" : "=r"(ones[c]));   // fp16x2 (1, 1)
    // per-lane ldmatrix offsets within a stage.  A box's 16-byte chunk index is
    // swizzled by XOR with the row's low bits, so the chunk pair u of a row
    // (u = 0, 1, ...) lies at the pair-0 offset XOR 32 (u % pairs per box) in
    // box u / pairs per box (the XOR only touches bits 5-6).
    const int ktok = (lane & 7) + 8 * ((lane >> 3) & 1), kch = lane >> 4;
    const int vtok = (lane & 7) + 8 * (lane >> 4), vch = (lane >> 3) & 1;
    const uint32_t k_off0 = KG::chunk_addr(0, ktok, kch), v_off0 = VG::chunk_addr(0, vtok, vch);
    constexpr int KPPB = C::KBI / 32, VPPB = C::VRB / 32 > 0 ? C::VRB / 32 : 1;   // chunk pairs per box
    // query B fragments: chunk 8 g + 4 kp + (lane >> 3) of row lane & 7, swizzled by
    // XOR with the row: the kp = 0 and kp = 1 addresses, group g at + 128 g
    const uint32_t qp_base = smem_u32(smem + C::QP_OFF), qpl_base = smem_u32(smem + C::QPL_OFF);
    const uint32_t q_row = (uint32_t)((lane & 7) * D * 2), q_sw = (uint32_t)(lane & 7), q_ch = (uint32_t)(lane >> 3);
    const uint32_t qa0 = q_row + ((q_ch ^ q_sw) << 4), qa1 = q_row + (((4u + q_ch) ^ q_sw) << 4);

    float o[4 * NCP][4];         // O^T, m-tile 4 u + 2 lc + j: chunk 2 u + lc, nibble pairs 2 j / 2 j + 1
    float ps[NGV][4];            // sum over tokens of P' per V group (all accumulator rows equal)
#pragma unroll
    for (int t = 0; t < 4 * NCP; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[t][c] = 0.0f;
#pragma unroll
    for (int g = 0; g < NGV; ++g)
#pragma unroll
        for (int c = 0; c < 4; ++c) ps[g][c] = 0.0f;
    // running reference maximum (log2 units) and sum of rows 2 tig, 2 tig + 1.
    // The reference is raised only when a block's maximum passes it by more
    // than kLazy (p then stays below 2^kLazy), or by anything at all when one
    // of the block's V scales is 256 or more (so that P' = p * scale stays a
    // finite fp16 value).
    constexpr float kLazy = 8.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    bool to = !q_ok;
    int stuck = -1;              // the stage whose wait gave up
    int slot = 0;
    uint32_t par = 0;
    int t0 = lo + kBlk * wb0;    // the block's first token

    for (int j = 0; j < n_st; ++j) {
        if (!to) {
            const bool ok = mbar_wait(bar_ring + 8 * (uint32_t)slot, par);
            if (__any_sync(0xffffffffu, !ok)) {
                to = true;
                stuck = j;
            }
        }
        const int nbl = stage_blocks(j);
#pragma unroll 1
        for (int b = 0; b < nbl; ++b, t0 += kBlk) {
        const uint32_t kb_addr = k_ring + (uint32_t)slot * C::CBK + (uint32_t)(b * kBlk * C::KBI) + k_off0;
        const uint32_t vb_addr = v_ring + (uint32_t)slot * C::CBV + (uint32_t)(b * kBlk * C::VRB) + v_off0;
        const uint32_t ksa = ks_ring + (uint32_t)slot * C::SBK + (uint32_t)(b * C::SBKB) + (uint32_t)gid * (NGK * 2);
        const uint32_t vsa = vs_ring + (uint32_t)slot * C::SBV + (uint32_t)(b * C::SBVB) + (uint32_t)gid * (NGV * 2);
        const bool edge = (t0 + kBlk > hi) || (t0 + kBlk > nv_all);

        // ---- S^T = K Q^T: tokens gid, gid + 8 (rows of the fragment) x rows 2 tig, 2 tig + 1
        uint32_t kw0[(NGK + 1) / 2], kw1[(NGK + 1) / 2];
        lds_scales<NGK>(ksa, kw0);
        lds_scales<NGK>(ksa + 8 * (NGK * 2), kw1);
        float sk0[NGK], sk1[NGK];
        scales_to_float<NGK>(kw0, sk0);
        scales_to_float<NGK>(kw1, sk1);
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int g = 0; g < NGK; ++g) {
            // K group g is the row's chunk pair g: one ldmatrix, KSTEPS_G k-steps
            uint32_t r0, r1, r2, r3;
            ldsm_x4((kb_addr ^ (uint32_t)(32 * (g % KPPB))) + (uint32_t)((g / KPPB) * C::ST * C::KBI), r0, r1, r2, r3);
            uint32_t h0[4], h1[4], h2[4], h3[4];
            if constexpr (K8) {
                uint32_t t2[2];
                unpack_q8_biased(r0, t2); h0[0] = t2[0]; h0[1] = t2[1];
                unpack_q8_biased(r1, t2); h1[0] = t2[0]; h1[1] = t2[1];
                unpack_q8_biased(r2, t2); h2[0] = t2[0]; h2[1] = t2[1];
                unpack_q8_biased(r3, t2); h3[0] = t2[0]; h3[1] = t2[1];
            } else {
                unpack_q4_biased(r0, h0);
                unpack_q4_biased(r1, h1);
                unpack_q4_biased(r2, h2);
                unpack_q4_biased(r3, h3);
            }
            float c0, c1, c2, c3;
            if constexpr (K8) {
                const uint4 kbq = lds128(smem_u32(smem + C::KBD_OFF) + (uint32_t)(g * 64 + tig * 16));
                c0 = __uint_as_float(kbq.x); c1 = __uint_as_float(kbq.y);
                c2 = __uint_as_float(kbq.z); c3 = __uint_as_float(kbq.w);
            } else {
                c0 = kbv[g % NKBV][0]; c1 = kbv[g % NKBV][1]; c2 = kbv[g % NKBV][2]; c3 = kbv[g % NKBV][3];
            }
            float cg[4];
#pragma unroll
            for (int kp = 0; kp < C::KSTEPS_G / 2; ++kp) {
                // B fragments of k-steps 2 p and 2 p + 1 (p = the group's pair kp) in one ldmatrix
                const int p = g * (C::KSTEPS_G / 2) + kp;
                const uint32_t qa = ((p & 1) ? qa1 : qa0) + (uint32_t)(128 * (p >> 1));
                uint32_t b00, b01, b10, b11;
                ldsm_x4(qp_base + qa, b00, b01, b10, b11);
                const int k = 2 * kp;
                if (kp == 0)
                    mma16816_c(cg, h0[k], h1[k], h2[k], h3[k], b00, b01, c0, c1, c2, c3);
                else
                    mma16816(cg, h0[k], h1[k], h2[k], h3[k], b00, b01);
                mma16816(cg, h0[k + 1], h1[k + 1], h2[k + 1], h3[k + 1], b10, b11);
                if constexpr (C::QLO) {
                    ldsm_x4(qpl_base + qa, b00, b01, b10, b11);
                    mma16816(cg, h0[k], h1[k], h2[k], h3[k], b00, b01);
                    mma16816(cg, h0[k + 1], h1[k + 1], h2[k + 1], h3[k + 1], b10, b11);
                }
            }
            sc[0] = fmaf(cg[0], sk0[g], sc[0]);
            sc[1] = fmaf(cg[1], sk0[g], sc[1]);
            sc[2] = fmaf(cg[2], sk1[g], sc[2]);
            sc[3] = fmaf(cg[3], sk1[g], sc[3]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[c] *= sl2;

        // V scales of tokens gid, gid + 8 (0 past the split end, where the plane
        // may hold anything)
        uint32_t vw0[(NGV + 1) / 2], vw1[(NGV + 1) / 2];
        lds_scales<NGV>(vsa, vw0);
        lds_scales<NGV>(vsa + 8 * (NGV * 2), vw1);
        // some V scale of the lane's tokens is 256 or more: a non-negative fp16
        // half h is >= 256 (0x5C00) exactly when h + 0x2400 reaches bit 15 (no
        // carry crosses into the other half); garbage past the split end only
        // makes this answer yes, which is safe
        uint32_t vge = (vw0[0] + 0x24002400u) | (vw1[0] + 0x24002400u);
#pragma unroll
        for (int w = 1; w < (NGV + 1) / 2; ++w) vge |= (vw0[w] + 0x24002400u) | (vw1[w] + 0x24002400u);
        const bool big = (vge & 0x80008000u) != 0u;
        float sv0[NGV], sv1[NGV];
        scales_to_float<NGV>(vw0, sv0);
        scales_to_float<NGV>(vw1, sv1);
        if (edge) {
            const int ta = t0 + gid, tc = ta + 8;
            sc[0] = (ta < hi && ta < nv0) ? sc[0] : -INFINITY;
            sc[1] = (ta < hi && ta < nv1) ? sc[1] : -INFINITY;
            sc[2] = (tc < hi && tc < nv0) ? sc[2] : -INFINITY;
            sc[3] = (tc < hi && tc < nv1) ? sc[3] : -INFINITY;
#pragma unroll
            for (int g = 0; g < NGV; ++g) {
                sv0[g] = ta < hi ? sv0[g] : 0.0f;
                sv1[g] = tc < hi ? sv1[g] : 0.0f;
            }
        }

        // ---- online softmax: the block's row maxima over its 16 tokens
        float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float slack = big ? 0.0f : kLazy;
        if (__any_sync(0xffffffffu, mx0 > m0 + slack || mx1 > m1 + slack)) {
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            // nothing accumulated yet (every reference still -inf): nothing to rescale
            if (__any_sync(0xffffffffu, m0 != -INFINITY || m1 != -INFINITY)) {
                const float c0 = (n0 == -INFINITY) ? 1.0f : ex2(m0 - n0);
                const float c1 = (n1 == -INFINITY) ? 1.0f : ex2(m1 - n1);
#pragma unroll
                for (int t = 0; t < 4 * NCP; ++t) {
                    o[t][0] *= c0;
                    o[t][1] *= c1;
                    o[t][2] *= c0;
                    o[t][3] *= c1;
                }
#pragma unroll
                for (int g = 0; g < NGV; ++g) {
                    ps[g][0] *= c0;
                    ps[g][1] *= c1;
                    ps[g][2] *= c0;
                    ps[g][3] *= c1;
                }
                l0 *= c0;
                l1 *= c1;
            }
            m0 = n0;
            m1 = n1;
        }
        const float b0 = (m0 == -INFINITY) ? 0.0f : m0, b1 = (m1 == -INFINITY) ? 0.0f : m1;
        const float p0 = ex2(sc[0] - b0), p1 = ex2(sc[1] - b1), p2 = ex2(sc[2] - b0), p3 = ex2(sc[3] - b1);
        l0 += p0 + p2;
        l1 += p1 + p3;

        // ---- O^T += V^T P'^T per V chunk pair (one V group for Q4_G64, two for Q4_G32)
#pragma unroll
        for (int u = 0; u < NCP; ++u) {
            uint32_t rv0, rv1, rv2, rv3;     // tokens 0-7 chunks 2u, 2u+1; tokens 8-15 chunks 2u, 2u+1
            ldsm_x4_t(vb_addr ^ (uint32_t)(32 * (u % VPPB)), rv0, rv1, rv2, rv3);
            uint32_t pb0 = 0, pb1 = 0;
#pragma unroll
            for (int lc = 0; lc < 2; ++lc) {
                if (lc == 0 || G32V) {
                    // P' of the chunk's group, tokens gid (rows 2 tig, 2 tig + 1) and
                    // gid + 8, transposed to tokens (2 tig, 2 tig + 1) and (2 tig + 8,
                    // 2 tig + 9) of row gid
                    const int g = G32V ? 2 * u + lc : u;
                    pb0 = movmatrix_t(pack_f16x2(p0 * sv0[g], p1 * sv0[g]));
                    pb1 = movmatrix_t(pack_f16x2(p2 * sv1[g], p3 * sv1[g]));
                }
                const uint32_t ra = lc ? rv1 : rv0, rb = lc ? rv3 : rv2;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t a0 = q4_pair_sub(ra, 2 * j), a1 = q4_pair_sub(ra, 2 * j + 1);
                    const uint32_t a2 = q4_pair_sub(rb, 2 * j), a3 = q4_pair_sub(rb, 2 * j + 1);
                    mma16816(o[4 * u + 2 * lc + j], a0, a1, a2, a3, pb0, pb1);
                }
                if (lc == 1 || G32V)
                    mma16816(ps[G32V ? 2 * u + lc : u], ones[0], ones[1], ones[2], ones[3], pb0, pb1);
            }
        }

        }
        // every lane's reads of this stage are done (their results fed the MMAs
        // above): lane 0 refills it
        __syncwarp();
        if (lane == 0 && !to && n_issued < n_st) issue();
        if (++slot == kWS) {
            slot = 0;
            par ^= 1u;
        }
    }
    // the dependent launch (the merge of the splits) may start now
    pdl_trigger();

    // never reuse the rings while a copy into them could be in flight (only
    // possible after a timeout; otherwise every issued copy was waited on)
    if (to && lane == 0) {
        for (int i = (stuck >= 0 ? stuck : 0); i < n_issued; ++i)
            mbar_wait(bars + 8 * (slot0 + (uint32_t)(i % kWS)), (uint32_t)((i / kWS) & 1));
    }
    if (to && lane == 0) s_timeout = 1;
    __syncwarp();              // (the warp's O goes over its ring below)

    // row sums: each lane summed its two tokens of every block
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // ---- combine the warps: each leaves its reference maxima, sums, sums of P'
    // per V group and raw O^T (odd head_dim indices still 16 times too large,
    // the V codes' offset still in) in shared memory (O^T in its own K ring, so
    // it need not wait for the others); after one barrier every thread forms
    // whole outputs from them.
    if (gid == 0) {
        red[warp * 16 + 2 * tig] = m0;
        red[warp * 16 + 2 * tig + 1] = m1;
        red[warp * 16 + 8 + 2 * tig] = l0;
        red[warp * 16 + 8 + 2 * tig + 1] = l1;
#pragma unroll
        for (int g = 0; g < NGV; ++g)
            *reinterpret_cast<float2 *>(psr + (warp * NGV + g) * 8 + 2 * tig) = make_float2(ps[g][0], ps[g][1]);
    }
    {
        float *cb = reinterpret_cast<float *>(smem + C::K_OFF) + warp * (kWRows * D);
        const bool w0 = 2 * tig < R, w1 = 2 * tig + 1 < R;     // padding rows are never read
#pragma unroll
        for (int t = 0; t < 4 * NCP; ++t) {
            const int d = 32 * (t >> 1) + 4 * gid + 2 * (t & 1);
            if (w0) *reinterpret_cast<float2 *>(cb + (2 * tig) * D + d) = make_float2(o[t][0], o[t][2]);
            if (w1) *reinterpret_cast<float2 *>(cb + (2 * tig + 1) * D + d) = make_float2(o[t][1], o[t][3]);
        }
    }
    __syncthreads();
    const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;
    const float *cb0 = reinterpret_cast<const float *>(smem + C::K_OFF);
    for (int idx = threadIdx.x; idx < R * (D / 4); idx += C::NTH) {
        const int r = idx / (D / 4), d = 4 * (idx % (D / 4)), g = d / C::VGS;
        // common maximum of row r and each warp's weight
        // (rolled loops: this code runs once per CTA, from a cold instruction cache)
        float M = -INFINITY;
#pragma unroll 1
        for (int w = 0; w < kWW; ++w) M = fmaxf(M, red[w * 16 + r]);
        float L = 0.0f, P = 0.0f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll 2
            for (int w = 0; w < kWW; ++w) {
                const float mw = red[w * 16 + r];
                const float f = (mw == -INFINITY) ? 0.0f : ex2(mw - M);
                L = fmaf(f, red[w * 16 + 8 + r], L);
                P = fmaf(f, psr[(w * NGV + g) * 8 + r], P);
                const float4 v = *reinterpret_cast<const float4 *>(cb0 + (w * kWRows + r) * D + d);
                acc.x = fmaf(f, v.x, acc.x);
                acc.y = fmaf(f, v.y, acc.y);
                acc.z = fmaf(f, v.z, acc.z);
                acc.w = fmaf(f, v.w, acc.w);
            }
        }
        const bool empty = (M == -INFINITY || L <= 0.0f);
        // the V codes entered as (q + 8) 2^-24, and 16 times that at odd head_dim
        // indices: remove 8 2^-24 (128 2^-24) per unit of P', scale back
        const float inv = empty ? 0.0f : 0x1p24f / L;
        const float e0 = fmaf(-0x1p-21f, P, 0.0f), e1 = fmaf(-0x1p-17f, P, 0.0f);
        const float4 res = make_float4((acc.x + e0) * inv, (acc.y + e1) * (inv * 0.0625f), (acc.z + e0) * inv,
                                       (acc.w + e1) * (inv * 0.0625f));
        const int i = r / G, jj = r % G;
        const int64_t orow = ((int64_t)s * a.n_q + i) * a.n_heads + kh * G + jj;
        float *dst = (a.n_splits == 1) ? a.out + orow * D : a.part_o + ((int64_t)split * rows_total + orow) * D;
        *reinterpret_cast<float4 *>(dst + d) = res;
        if (d == 0) {
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
template <int KC, int VC, int D, typename QT>
cudaError_t warp_prepare(int *per_sm)
{
    using C = WCfg<KC, VC, D, QT>;
    static PerDevice pd;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int n = per_device(pd, dev, []() -> int {
        auto kern = decode_warp_kernel<KC, VC, D, QT>;
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        int v = 0;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, C::NTH, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        return v > 0 ? v : -(int)cudaErrorInvalidConfiguration;
    });
    if (n <= 0) return (cudaError_t)(-n);
    *per_sm = n;
    return cudaSuccess;
}

template <int KC, int VC, int D, typename QT>
cudaError_t warp_launch(const DecodeArgs &a, cudaStream_t st)
{
    using C = WCfg<KC, VC, D, QT>;
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    // boxes of a whole stage, and of one block (a run's first stage, and its
    // last where the rest of the run is odd)
    CUtensorMap tk, tv, tk1, tv1;
    if (!make_codes_map(&tk, a.k.qs, C::KRB, rows, C::ST) || !make_codes_map(&tv, a.v.qs, C::VRB, rows, C::ST) ||
        !make_codes_map(&tk1, a.k.qs, C::KRB, rows, kBlk) || !make_codes_map(&tv1, a.v.qs, C::VRB, rows, kBlk))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaError_t e = warp_prepare<KC, VC, D, QT>(&per_sm);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_splits, a.n_kv_heads, a.n_seq);
    return launch_pdl(decode_warp_kernel<KC, VC, D, QT>, grid, dim3(C::NTH), C::SMEM, st, a, tk, tv, tk1, tv1);
}

template <int KC, int VC>
int warp_per_sm_d(int head_dim)
{
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (head_dim) {
    case 64: e = warp_prepare<KC, VC, 64, __half>(&n); break;
    case 128: e = warp_prepare<KC, VC, 128, __half>(&n); break;
    case 256: e = warp_prepare<KC, VC, 256, __half>(&n); break;
    default: break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int KC, int VC>
cudaError_t warp_launch_d(const DecodeArgs &a, bool f16, cudaStream_t st)
{
    switch (a.head_dim) {
    case 64: return f16 ? warp_launch<KC, VC, 64, __half>(a, st) : warp_launch<KC, VC, 64, float>(a, st);
    case 128: return f16 ? warp_launch<KC, VC, 128, __half>(a, st) : warp_launch<KC, VC, 128, float>(a, st);
    case 256: return f16 ? warp_launch<KC, VC, 256, __half>(a, st) : warp_launch<KC, VC, 256, float>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Q4_G64 V with Q4_G64 or q8_0 K; Q4_G32 V with q8_0 K (the shipped q8_0 / q4_0
// pair; with 4-bit K the eight V groups' sums of P' and the K groups' four
// accumulator inputs would not fit the registers together).
bool decode_warp_shape(int k_codec, int v_codec, int head_dim, int rows_per_kv_head)
{
    const bool pair = (v_codec == KVQ_CODEC_Q4_G64 && (k_codec == KVQ_CODEC_Q4_G64 || k_codec == KVQ_CODEC_Q8_0)) ||
                      (v_codec == KVQ_CODEC_Q4_G32 && k_codec == KVQ_CODEC_Q8_0);
    return pair && rows_per_kv_head >= 1 && rows_per_kv_head <= kWRows &&
           (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

int decode_warp_ctas_per_sm(int k_codec, int v_codec, int head_dim)
{
    if (v_codec == KVQ_CODEC_Q4_G32) return warp_per_sm_d<KVQ_CODEC_Q8_0, KVQ_CODEC_Q4_G32>(head_dim);
    return k_codec == KVQ_CODEC_Q8_0 ? warp_per_sm_d<KVQ_CODEC_Q8_0, KVQ_CODEC_Q4_G64>(head_dim)
                                     : warp_per_sm_d<KVQ_CODEC_Q4_G64, KVQ_CODEC_Q4_G64>(head_dim);
}

bool decode_warp_takes(const DecodeArgs &a)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    return decode_warp_shape(a.k.codec, a.v.codec, a.head_dim, R) && rows < (1LL << 31) &&
           tensor_maps_available() && decode_warp_ctas_per_sm(a.k.codec, a.v.codec, a.head_dim) > 0;
}

cudaError_t launch_decode_warp(const DecodeArgs &a, int q_dtype, cudaStream_t st)
{
    const bool f16 = q_dtype == KVQ_F16;
    if (a.v.codec == KVQ_CODEC_Q4_G32) return warp_launch_d<KVQ_CODEC_Q8_0, KVQ_CODEC_Q4_G32>(a, f16, st);
    return a.k.codec == KVQ_CODEC_Q8_0 ? warp_launch_d<KVQ_CODEC_Q8_0, KVQ_CODEC_Q4_G64>(a, f16, st)
                                       : warp_launch_d<KVQ_CODEC_Q4_G64, KVQ_CODEC_Q4_G64>(a, f16, st);
}

}  // namespace kvq
