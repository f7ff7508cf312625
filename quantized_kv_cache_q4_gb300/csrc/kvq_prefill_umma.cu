// kvq_prefill_umma.cu -- attention for many query rows per kv head (a prompt
// chunk: n_q tokens x the kv head's G query heads) over a 4-bit packed cache, on
// the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
// (den_llama.cpp, "Results": prefill through the quantized cache; "build3
// (working engine) -- additions": split-KV prefill.)
//
// One CTA takes a block of 128 query rows of one (sequence, kv head) and the
// key range of one split; row r of the block is tensor-memory lane r.  K and
// V are Q4_G64.  Per 64-token tile:
//  * TMA has brought the tile's K and V codes (swizzled 2D boxes) and scales
//    (bulk copies) into a 3-stage ring (the decode kernel's tile format).
//  * All 8 warps turn the K tile into two fp16 operands whose sum is K / 16
//    exactly: each fp16 group scale s is cut into s_hi (its top 7 significant
//    bits) and s_lo = s - s_hi (at most 4), so that q * s_hi / 16 and
//    q * s_lo / 16 are both exact in fp16 for any signed nibble q (the 1/16
//    keeps every product finite for any fp16 scale).  They are laid out as
//    K-major B operands: 128-byte swizzled rows of 64 values.
//  * One thread issues S = Q K_hi^T + Q K_lo^T (M = 128 rows, N = 64
//    tokens, K = head_dim) into 64 tensor-memory columns: the scores are
//    those of the exact dequantized keys, accumulated in fp32.
//  * The warps turn the V tile the same way into V_hi + V_lo in the same
//    buffer (S has finished reading it) -- in these bytes the MN-major B
//    operands of O = P V -- and compute the softmax: each row is read back by
//    two threads (warps w and w + 4 share lane quarter w % 4; one takes tokens
//    0-31, the other 32-63), whose maxima are combined through shared memory;
//    where a row's maximum grows, its O columns are rescaled in tensor memory.
//    p = 2^(s - m) (<= 1, the largest exactly 1) is rounded once to fp16 into
//    shared memory, the K-major A operand of O += P V.
//  * One thread issues O += P V_hi + P V_lo (M = 128, N = head_dim, K = 64
//    tokens) into head_dim tensor-memory columns.
// The tensor core and the CUDA cores take turns inside a CTA (no warp
// specialisation yet); CTAs on other SMs overlap.  Within each 8-value group
// the head_dim order is the one the nibble unpack delivers (value pairs
// (d, d + 4)); the query is written in the same order and the output is put
// back in natural order.
//
// Every mbarrier wait is bounded (about a second); after a timeout the kernel
// sets KVQ_ERR_TIMEOUT, skips further waits and issues, and still frees its
// tensor memory.
#include "kvq_ptx.cuh"

namespace kvq {
using namespace ptx;
namespace {

constexpr int kUT = 256;                 // compute threads (8 warps)
constexpr int kUThreads = kUT + 32;      // + one warp that issues the MMAs and the tile copies
constexpr int kURows = 128;              // query rows per CTA = tensor-memory lanes
constexpr int kUTile = 64;               // tokens per tile (= the decode kernel's TMA box)

// ---- tcgen05 building blocks ------------------------------------------------
// Shared-memory matrix descriptor: start, leading and stride byte offsets (16-byte
// units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp16 A and B, fp32 accumulator, M x N,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t umma_idesc(int m, int n, int b_mn)
{
    return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

// The same with the A operand in tensor memory (row i in lane i, two fp16 of
// consecutive k per 32-bit column; one k-step of 16 is 8 columns).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The compute warps' own barrier (the issuing warp never waits on it).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kUT) : "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void async_proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Offset of 16-byte chunk c (8 values) of row r in a 128-byte-swizzled operand
// whose rows hold 64 values and whose blocks of 64 values are block_bytes apart.
__device__ __forceinline__ uint32_t sw128_off(int r, int c, uint32_t block_bytes)
{
    return (uint32_t)(c >> 3) * block_bytes + (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) << 4);
}

// A code word (values 8c .. 8c+7 of a row, value 2j in the low nibble of byte
// j) as four fp16x2 of exact integers: the pairs (0,4), (2,6) as q and (1,5),
// (3,7) as 16 q -- chunk order (0,4), (1,5), (2,6), (3,7), the order the rest
// of the kernel uses inside a group of 8.
__device__ __forceinline__ uint4 codes_word(uint32_t w)
{
    uint32_t h[4];
    unpack_q4_biased(w, h);          // 1032 + q (pairs 0, 2), 1152 + 16 q (pairs 1, 3): exact
    uint32_t o[4];
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(h[0]), "r"(0x64086408u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(h[1]), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2]) : "r"(h[2]), "r"(0x64086408u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[3]) : "r"(h[3]), "r"(0x64806480u));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int D>
struct UmCfg {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static constexpr int KC = KVQ_CODEC_Q4_G64, VC = KVQ_CODEC_Q4_G64;
    static constexpr int KRB = row_bytes(KC, D), VRB = row_bytes(VC, D);
    static constexpr int KSB = scale_row_bytes(KC, D), VSB = scale_row_bytes(VC, D);
    static constexpr int NG = D / 64;                             // 64-value blocks (= scale groups)
    // shared memory (from a 1024-aligned base)
    static constexpr int X_BLOCK = kUTile * 128;                  // 64 tokens x 64 values, fp16
    static constexpr int X_PAIR = 2 * X_BLOCK;                    // the hi and lo blocks of 64 values
    static constexpr int XK_OFF = 0;                              // K operands: [NG][hi, lo][64 tokens][128 B]
    static constexpr int XV_OFF = XK_OFF + NG * X_PAIR;           // V operands, same layout
    static constexpr int P_OFF = XV_OFF + NG * X_PAIR;            // P: [128 rows][64 tokens] fp16
    static constexpr int RING_OFF = P_OFF + kURows * 128;
    // ring stage: K codes, V codes (TMA boxes), K scales, V scales
    static constexpr int SK_OFF = 0;
    static constexpr int SV_OFF = align_up(kUTile * KRB, 1024);
    static constexpr int SKS_OFF = SV_OFF + align_up(kUTile * VRB, 1024);
    static constexpr int SVS_OFF = SKS_OFF + align_up(kUTile * KSB, 128);
    static constexpr int STAGE = align_up(SVS_OFF + kUTile * VSB, 1024);
    static constexpr int NS = 3;
    static constexpr int RED_OFF = RING_OFF + NS * STAGE;         // fp32 [2][128]: half-row maxima / sums
    // mbarriers: full[NS] (tile landed), S done, O done (MMA commits), K ready,
    // P / V ready (the compute threads' hand-offs to the issuing warp)
    static constexpr int BAR_OFF = RED_OFF + 2 * kURows * 4;
    static constexpr int TMEM_SLOT = BAR_OFF + (NS + 4) * 8;
    static constexpr int SMEM = TMEM_SLOT + 16 + 1024;            // + alignment slack
    // tensor memory: O in [0, D); the scores against K_hi (64 columns) and
    // against K_lo (the next 64) in [D, D + 128); the query rows (A operand of
    // S, two fp16 per column) in [D + 128, D + 128 + D / 2)
    static constexpr int O_COL = 0, S_COL = D, Q_COL = D + 128;
    static constexpr int NCOL_USED = D + 128 + D / 2;
    static constexpr int NCOL = NCOL_USED <= 128 ? 128 : NCOL_USED <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC_S = umma_idesc(kURows, 2 * kUTile, 0);
    static constexpr uint32_t IDESC_O = umma_idesc(kURows, D, 1);
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(NCOL_USED <= 512, "tensor memory");
};

// Bounded mbarrier wait that gives up for good once the CTA has timed out.
__device__ __forceinline__ bool uwait(uint32_t bar, uint32_t parity, volatile int *timed_out)
{
    if (*timed_out) return false;
    if (mbar_wait(bar, parity)) return true;
    *timed_out = 1;
    return false;
}

template <typename C, typename KG, typename VG>
__device__ __forceinline__ void um_issue_tile(uint32_t st, uint32_t full, const CUtensorMap *tmk,
                                              const CUtensorMap *tmv, const uint8_t *ksc, const uint8_t *vsc,
                                              int64_t row0)
{
    const uint64_t pol = evict_first_policy();
    mbar_expect_tx(full, (uint32_t)(KG::BYTES + VG::BYTES + kUTile * (C::KSB + C::VSB)));
#pragma unroll
    for (int b = 0; b < KG::NB; ++b)
        tma_load_2d(st + C::SK_OFF + b * kUTile * KG::BI, tmk, b * KG::BI, (int)row0, full, pol);
#pragma unroll
    for (int b = 0; b < VG::NB; ++b)
        tma_load_2d(st + C::SV_OFF + b * kUTile * VG::BI, tmv, b * VG::BI, (int)row0, full, pol);
    bulk_load_hint(st + C::SKS_OFF, ksc + row0 * C::KSB, kUTile * C::KSB, full, pol);
    bulk_load_hint(st + C::SVS_OFF, vsc + row0 * C::VSB, kUTile * C::VSB, full, pol);
}

// One plane of a ring stage as the two fp16 operands whose sum is the plane's
// values / 16, exactly, stored per block of 64 values as the hi rows of the 64
// tokens followed by their lo rows: thread t takes token t % 64 and the
// quarter t / 64 of its code words (all in one scale group).  q * (s_hi / 16) and q * (s_lo /
// 16) are exact in fp16: s_hi keeps the top 7 significant bits of the fp16
// scale s, s_lo = s - s_hi the rest (at most 4 bits), and |q| <= 8 takes at
// most 4 (odd head_dim indices arrive as 16 q and take scale / 256).  Tokens
// at or past n_valid get scale 0: zero operands.
template <int D, int SB, typename G>
__device__ __forceinline__ void um_split_plane(uint32_t codes, const uint8_t *scales, uint8_t *dst, int n_valid)
{
    constexpr int WPT = D / 32;                      // code words per thread
    constexpr int NW = WPT < 4 ? WPT : 4;            // words per shared-memory load
    const int tok = threadIdx.x & (kUTile - 1), part = threadIdx.x >> 6;
    const int g = (part * WPT) / 8;                  // the thread's scale group (64 values = 8 words)
    __half sc = __ushort_as_half((unsigned short)0);
    if (tok < n_valid) sc = reinterpret_cast<const __half *>(scales + tok * SB)[g];
    const __half sh = __ushort_as_half((unsigned short)(__half_as_ushort(sc) & 0xFFF0u));
    const __half sl = __hsub(sc, sh);
    const __half2 k16 = __float2half2_rn(0.0625f), k256 = __float2half2_rn(0.00390625f);
    const uint32_t h_e = h2_as_u32(__hmul2(__half2half2(sh), k16)), h_o = h2_as_u32(__hmul2(__half2half2(sh), k256));
    const uint32_t l_e = h2_as_u32(__hmul2(__half2half2(sl), k16)), l_o = h2_as_u32(__hmul2(__half2half2(sl), k256));
#pragma unroll
    for (int q = 0; q < WPT; q += NW) {
        const int w0 = part * WPT + q;               // first word, in 16-byte chunk w0 / 4 of the codes row
        const uint32_t addr = G::chunk_addr(codes, tok, w0 >> 2) + (uint32_t)((w0 & 3) * 4);
        uint32_t wv[4];
        if constexpr (NW == 4) {
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(wv[0]), "=r"(wv[1]), "=r"(wv[2]), "=r"(wv[3])
                         : "r"(addr));
        } else {
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(wv[0]), "=r"(wv[1]) : "r"(addr));
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint4 c = codes_word(wv[i]);       // (q, q), (16q, 16q), (q, q), (16q, 16q)
            uint4 hi, lo;
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi.x) : "r"(c.x), "r"(h_e));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi.y) : "r"(c.y), "r"(h_o));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi.z) : "r"(c.z), "r"(h_e));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi.w) : "r"(c.w), "r"(h_o));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(lo.x) : "r"(c.x), "r"(l_e));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(lo.y) : "r"(c.y), "r"(l_o));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(lo.z) : "r"(c.z), "r"(l_e));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(lo.w) : "r"(c.w), "r"(l_o));
            // [block of 64 values][hi, lo][token][128 B]
            const uint32_t off = sw128_off(tok, w0 + i, 2 * kUTile * 128);
            *reinterpret_cast<uint4 *>(dst + off) = hi;
            *reinterpret_cast<uint4 *>(dst + off + kUTile * 128) = lo;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kUThreads, 1)
prefill_umma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv)
{
    using C = UmCfg<D>;
    using KG = TileGeom<C::KRB>;
    using VG = TileGeom<C::VRB>;
    constexpr int NS = C::NS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::BAR_OFF, bar_s = bar_full + 8 * NS, bar_o = bar_s + 8;
    const uint32_t bar_k = bar_o + 8, bar_pv = bar_k + 8;
    float *red = reinterpret_cast<float *>(smem + C::RED_OFF);     // [2][128]
    __shared__ volatile int s_timeout;
    __shared__ int s_issued;
    __shared__ int s_seq;

    const int tid = threadIdx.x, warp = tid >> 5;
    const bool issuer = warp == kUT / 32;                           // the last warp
    // softmax and output: row (= tensor-memory lane) and which 32 tokens of a
    // tile / which half of head_dim this thread takes
    const int row = tid & (kURows - 1), half = (tid >> 7) & 1;
    const int split = blockIdx.x, kh = blockIdx.y / a.n_row_blocks, rblk = blockIdx.y % a.n_row_blocks;
    const int G = a.n_heads / a.n_kv_heads;
    const int r0 = rblk * kURows;
    const int R = min(kURows, a.n_q * G - r0);
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        s_timeout = 0;
        s_issued = 0;
        for (int i = 0; i < NS; ++i) mbar_init(bar_full + 8 * i, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_k, kUT);
        mbar_init(bar_pv, kUT);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sbase + C::TMEM_SLOT),
                     "n"(C::NCOL)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::TMEM_SLOT);
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    pdl_wait();
    // sequences in order of decreasing length (longest first), as in the decode kernel
    int s = blockIdx.z;
    if (a.n_seq > 1 && a.n_seq <= kUT) {
        if (tid < a.n_seq) {
            const int lt = a.kv_len[tid];
            int rank = 0;
            for (int u = 0; u < a.n_seq; ++u) {
                const int lu = a.kv_len[u];
                rank += (lu > lt) || (lu == lt && u < tid);
            }
            if (rank == (int)blockIdx.z) s_seq = tid;
        }
        __syncthreads();
        s = s_seq;
    }
    int len = a.fixed_len >= 0 ? a.fixed_len : a.kv_len[s];
    if (len < 0 || len > a.max_kv_len) {
        if (tid == 0 && split == 0 && blockIdx.y == 0 && a.err) atomicOr(a.err, KVQ_ERR_KV_LEN);
        len = len < 0 ? 0 : a.max_kv_len;
    }
    int lo, hi;
    split_range(len, a.n_splits, split, lo, hi);
    // no row of this block sees past its last query token's keys
    hi = max(lo, min(hi, len + a.causal_extra - a.n_q + (r0 + R - 1) / G + 1));
    const int n_tiles = (int)ceil_div(hi - lo, kUTile);
    const int64_t plane_row = ((int64_t)s * a.n_kv_heads + kh) * a.capacity;
    const uint8_t *ksc = reinterpret_cast<const uint8_t *>(a.k.sc);
    const uint8_t *vsc = reinterpret_cast<const uint8_t *>(a.v.sc);
    auto stage_of = [&](int jj) { return C::RING_OFF + (jj % NS) * C::STAGE; };

    if (issuer) {
        // ---- the issuing warp (one thread): tile copies and MMAs, in the order
        // S(0); then per tile j: S(j + 1) as soon as its K operands are ready
        // (it runs beside the softmax of tile j), O += P V of tile j as soon as
        // P and the V operands are ready (and tile j's ring stage is refilled)
        if ((tid & 31) == 0) {
            const int first = min(NS, n_tiles);
            for (int j = 0; j < first; ++j)
                um_issue_tile<C, KG, VG>(sbase + stage_of(j), bar_full + 8 * j, &tmk, &tmv, ksc, vsc,
                                         plane_row + lo + (int64_t)j * kUTile);
            s_issued = first;
            // descriptors: built once; a k-step adds a constant to the start
            // address field (16-byte units, no carry: shared memory < 256 KB)
            const uint64_t kdesc = umma_desc(sbase + C::XK_OFF, 16, 1024);
            const uint64_t vdesc = umma_desc(sbase + C::XV_OFF, C::X_PAIR, 1024);
            const uint64_t pdesc = umma_desc(sbase + C::P_OFF, 16, 1024);
            // S = Q [K_hi; K_lo]^T: N = 128 (the hi rows of the tile's 64 tokens,
            // then their lo rows), one accumulator; the compute warps add the halves
            auto issue_s = [&](int jj) {
                (void)jj;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16_ta(tmem + C::S_COL, tmem + C::Q_COL + 8 * ks,
                                kdesc + (uint64_t)(((ks >> 2) * C::X_PAIR + (ks & 3) * 32) >> 4), C::IDESC_S,
                                ks > 0 ? 1u : 0u);
                umma_commit(bar_s);
            };
            if (n_tiles > 0 && uwait(bar_k, 0, &s_timeout)) issue_s(0);
            for (int j = 0; j < n_tiles && !s_timeout; ++j) {
                if (j + 1 < n_tiles) {
                    if (!uwait(bar_k, (j + 1) & 1, &s_timeout)) break;
                    issue_s(j + 1);
                }
                if (!uwait(bar_pv, j & 1, &s_timeout)) break;
                if (j + NS < n_tiles) {
                    um_issue_tile<C, KG, VG>(sbase + stage_of(j), bar_full + 8 * (j % NS), &tmk, &tmv, ksc, vsc,
                                             plane_row + lo + (int64_t)(j + NS) * kUTile);
                    s_issued = j + NS + 1;
                }
                tc_fence_after();
#pragma unroll
                for (int hv = 0; hv < 2; ++hv)
#pragma unroll
                    for (int ks = 0; ks < kUTile / 16; ++ks)
                        umma_f16(tmem + C::O_COL, pdesc + (uint64_t)((ks * 32) >> 4),
                                 vdesc + (uint64_t)((hv * C::X_BLOCK + ks * 2048) >> 4), C::IDESC_O,
                                 (j > 0 || hv > 0 || ks > 0) ? 1u : 0u);
                umma_commit(bar_o);
            }
        }
        __syncwarp();
    }
    else {
        // ---- the compute warps
        // the block's query rows into tensor memory as the A operand of S = Q K^T:
        // fp16, head_dim in the unpack order inside each group of 8 (two values a
        // column); rows >= R zero.  Thread (row, half) writes half of its row.
        {
            const __half *q = static_cast<const __half *>(a.q);
            int64_t qrow = 0;
            if (row < R) {
                const int rr = r0 + row;
                qrow = (((int64_t)s * a.n_q + rr / G) * a.n_heads + kh * G + rr % G) * D;
            }
#pragma unroll 1
            for (int cb = 0; cb < D / 4; cb += 32) {              // 32 columns = 8 chunks of 8 values
                float qc[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c = half * (D / 16) + cb / 4 + k;   // value chunk
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (row < R) v = *reinterpret_cast<const uint4 *>(q + qrow + 8 * c);
                    uint32_t o0, o1, o2, o3;
                    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o0) : "r"(v.x), "r"(v.z));   // (x0, x4)
                    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(o1) : "r"(v.x), "r"(v.z));   // (x1, x5)
                    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o2) : "r"(v.y), "r"(v.w));   // (x2, x6)
                    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(o3) : "r"(v.y), "r"(v.w));   // (x3, x7)
                    qc[4 * k] = __uint_as_float(o0);
                    qc[4 * k + 1] = __uint_as_float(o1);
                    qc[4 * k + 2] = __uint_as_float(o2);
                    qc[4 * k + 3] = __uint_as_float(o3);
                }
                tmem_st32(lane_base + C::Q_COL + half * (D / 4) + cb, qc);
            }
            tmem_st_wait();
        }
        // per-row softmax state (the two threads of a row keep the same maximum)
        const int nv_row = row < R ? len + a.causal_extra - a.n_q + (r0 + row) / G + 1 : 0x7FFFFFFF;
        const int lim = min(hi, nv_row);
        float m_run = -INFINITY, l_part = 0.0f;
        const float sc = a.scale_log2 * 16.0f;         // the K operands carry K / 16
        // hand-off to the issuing warp: this thread's shared-memory operand writes
        // (and tensor-memory stores) are done
        auto hand_off = [&](uint32_t bar) {
            async_proxy_fence();
            tc_fence_before();
            mbar_arrive(bar);
        };

        // K operands of tile 0 (and, above, the query rows)
        if (n_tiles > 0) {
            uwait(bar_full, 0, &s_timeout);
            um_split_plane<D, C::KSB, KG>(sbase + stage_of(0) + C::SK_OFF, smem + stage_of(0) + C::SKS_OFF,
                                          smem + C::XK_OFF, min(kUTile, hi - lo));
            hand_off(bar_k);
        }
        for (int j = 0; j < n_tiles; ++j) {
            const int tb = lo + j * kUTile;
            // (1) this thread's 32 scores of tile j (the K_hi and K_lo halves
            //     added), then the K operands of tile j + 1 (S of tile j has read
            //     the buffer; the hand-off also frees S for tile j + 1)
            uwait(bar_s, j & 1, &s_timeout);
            tc_fence_after();
            float x[32];
            {
                float xl[32];
                tmem_ld32(lane_base + C::S_COL + 32 * half, x);
                tmem_ld32(lane_base + C::S_COL + 64 + 32 * half, xl);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] += xl[i];
            }
            if (j + 1 < n_tiles) {
                uwait(bar_full + 8 * ((j + 1) % NS), ((j + 1) / NS) & 1, &s_timeout);
                um_split_plane<D, C::KSB, KG>(sbase + stage_of(j + 1) + C::SK_OFF,
                                              smem + stage_of(j + 1) + C::SKS_OFF, smem + C::XK_OFF,
                                              min(kUTile, hi - tb - kUTile));
                hand_off(bar_k);
            }
            // (2) the V operands of tile j, once O += P V of tile j - 1 is done
            if (j > 0) uwait(bar_o, (j - 1) & 1, &s_timeout);
            tc_fence_after();
            um_split_plane<D, C::VSB, VG>(sbase + stage_of(j) + C::SV_OFF, smem + stage_of(j) + C::SVS_OFF,
                                          smem + C::XV_OFF, min(kUTile, hi - tb));
            // (3) softmax of tile j: scores in log2 units, masked past the split
            //     end and the row's causal limit
            const int t0 = tb + 32 * half;
            if (t0 + 32 > lim) {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = (t0 + i < lim) ? x[i] * sc : -INFINITY;
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] *= sc;
            }
            float mh = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) mh = fmaxf(mh, x[i]);
            red[half * kURows + row] = mh;
            compute_sync();
            const float mt = fmaxf(red[row], red[kURows + row]);
            float f = 1.0f;
            bool resc = false;
            if (mt > m_run) {
                f = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                m_run = mt;
                resc = true;
            }
            l_part *= f;
            const float base = (m_run == -INFINITY) ? 0.0f : m_run;
            uint32_t pk[16];
            float l_tile = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p0 = ex2(x[2 * i] - base), p1 = ex2(x[2 * i + 1] - base);
                l_tile += p0 + p1;
                pk[i] = pack_f16x2(p0, p1);
            }
            l_part += l_tile;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(smem + C::P_OFF + sw128_off(row, 4 * half + k, 0)) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            // O columns of this thread's half of head_dim, rescaled where the
            // maximum grew (whole warps: tensor-memory loads are warp-wide)
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                for (int c = 0; c < D / 2; c += 32) {
                    float ov[32];
                    const uint32_t ta = lane_base + C::O_COL + half * (D / 2) + c;
                    tmem_ld32(ta, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= f;
                    tmem_st32(ta, ov);
                }
                tmem_st_wait();
            }
            // (4) P, the V operands and O are ready for O += P V of tile j; the
            //     maxima buffer is reused by the next tile only after every
            //     thread has read it (the next tile's first hand-off comes later
            //     in program order than these reads, and the next write follows
            //     a wait on O += P V, which needs every thread's hand-off)
            hand_off(bar_pv);
        }
        // the dependent launch (the merge of the splits) may start now
        pdl_trigger();
        if (n_tiles > 0) uwait(bar_o, (n_tiles - 1) & 1, &s_timeout);
        tc_fence_after();
        compute_sync();
        red[half * kURows + row] = l_part;
        compute_sync();
        const float L = red[row] + red[kURows + row];
        const bool empty = (m_run == -INFINITY || L <= 0.0f);
        // the V operands carried V / 16
        const float inv = empty ? 0.0f : 16.0f / L;
        const int64_t rows_total = (int64_t)a.n_seq * a.n_q * a.n_heads;
        float *dst = nullptr;
        int64_t orow = 0;
        if (row < R) {
            const int rr = r0 + row;
            orow = ((int64_t)s * a.n_q + rr / G) * a.n_heads + kh * G + rr % G;
            dst = (a.n_splits == 1) ? a.out + orow * D : a.part_o + ((int64_t)split * rows_total + orow) * D;
        }
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
            float ov[32];
            if (n_tiles > 0) {
                tmem_ld32(lane_base + C::O_COL + half * (D / 2) + c, ov);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] = 0.0f;
            }
            if (dst) {
                // columns 8g + p hold head_dim 8g + (0, 4, 1, 5, 2, 6, 3, 7)[p]
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float *o = dst + half * (D / 2) + c + 8 * g;
                    *reinterpret_cast<float4 *>(o) =
                        make_float4(ov[8 * g] * inv, ov[8 * g + 2] * inv, ov[8 * g + 4] * inv, ov[8 * g + 6] * inv);
                    *reinterpret_cast<float4 *>(o + 4) = make_float4(ov[8 * g + 1] * inv, ov[8 * g + 3] * inv,
                                                                     ov[8 * g + 5] * inv, ov[8 * g + 7] * inv);
                }
            }
        }
        if (dst && half == 0) {
            const float lse = empty ? -INFINITY : (m_run + log2f(L)) * kLn2;
            if (a.n_splits == 1) {
                if (a.out_lse) a.out_lse[orow] = lse;
            } else {
                a.part_lse[(int64_t)split * rows_total + orow] = lse;
            }
        }
    }
    // never leave while a copy into shared memory could be in flight (only
    // possible after a timeout)
    __syncthreads();
    if (tid == kUT && s_timeout) {
        const int issued = s_issued;
        for (int j = issued - 1; j >= 0 && j >= issued - NS; --j) mbar_wait(bar_full + 8 * (j % NS), (j / NS) & 1);
        if (a.err) atomicOr(a.err, KVQ_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(C::NCOL) : "memory");
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D>
int um_ctas_per_sm()
{
    using C = UmCfg<D>;
    static PerDevice pd;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int n = per_device(pd, dev, []() -> int {
        auto kern = prefill_umma_kernel<D>;
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        int v = 0;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kUThreads, C::SMEM);
        if (r != cudaSuccess) return -(int)r;
        // the CTAs sharing an SM must fit its 512 tensor-memory columns
        if (v * C::NCOL > 512) v = 512 / C::NCOL;
        return v > 0 ? v : -(int)cudaErrorInvalidConfiguration;
    });
    if (n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D>
cudaError_t um_launch(const DecodeArgs &a, cudaStream_t st)
{
    using C = UmCfg<D>;
    if (um_ctas_per_sm<D>() <= 0) return cudaErrorInvalidConfiguration;
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    CUtensorMap tk, tv;
    if (!make_codes_map(&tk, a.k.qs, C::KRB, rows, kUTile) || !make_codes_map(&tv, a.v.qs, C::VRB, rows, kUTile))
        return cudaErrorInvalidValue;
    dim3 grid(a.n_splits, a.n_kv_heads * a.n_row_blocks, a.n_seq);
    return launch_pdl(prefill_umma_kernel<D>, grid, dim3(kUThreads), C::SMEM, st, a, tk, tv);
}

}  // namespace

bool prefill_umma_shape(int k_codec, int v_codec, int head_dim, int rows_per_kv_head)
{
    return rows_per_kv_head >= kUmmaMinRows && k_codec == KVQ_CODEC_Q4_G64 && v_codec == KVQ_CODEC_Q4_G64 &&
           (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

int prefill_umma_ctas_per_sm(int k_codec, int v_codec, int head_dim)
{
    if (k_codec != KVQ_CODEC_Q4_G64 || v_codec != KVQ_CODEC_Q4_G64) return 0;
    switch (head_dim) {
    case 64: return um_ctas_per_sm<64>();
    case 128: return um_ctas_per_sm<128>();
    case 256: return um_ctas_per_sm<256>();
    default: return 0;
    }
}

bool prefill_umma_takes(const DecodeArgs &a, int q_dtype)
{
    const int R = a.n_q * (a.n_heads / a.n_kv_heads);
    const int64_t rows = (int64_t)a.n_seq * a.n_kv_heads * a.capacity;
    return q_dtype == KVQ_F16 && prefill_umma_shape(a.k.codec, a.v.codec, a.head_dim, R) && rows < (1LL << 31) &&
           tensor_maps_available() && prefill_umma_ctas_per_sm(a.k.codec, a.v.codec, a.head_dim) > 0;
}

cudaError_t launch_prefill_umma(const DecodeArgs &args, cudaStream_t st)
{
    DecodeArgs a = args;
    a.n_row_blocks = (int)ceil_div(a.n_q * (a.n_heads / a.n_kv_heads), kURows);
    switch (a.head_dim) {
    case 64: return um_launch<64>(a, st);
    case 128: return um_launch<128>(a, st);
    case 256: return um_launch<256>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq
