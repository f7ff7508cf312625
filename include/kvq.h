/*
 * kvq.h -- C ABI of the GB300 quantized-KV-cache decode library (libkvq.so).
 *
 * The library implements the two stages a llama.cpp-style serving engine runs
 * per decode step over a quantized KV cache: the KV-cache append stage, which
 * quantizes the new K/V rows into the cache, and the attention stage, which
 * reads the packed cache (Llaminar, "Graphs and Compute Stages", names both as
 * separate compute stages; den_llama.cpp, "What's in the fork", lists the
 * set-rows/cpy quantize path and the fattn-vec Q4_G64 kernels).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps device memory; it enqueues kernels on
 *     `stream` (a cudaStream_t passed as void*, NULL = legacy default stream)
 *     and returns.  Results are ready once the stream has been synchronized.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns KVQ_EINVAL (or KVQ_EUNSUPPORTED / KVQ_EWORKSPACE) and
 *     launches nothing.  kvq_last_error() then describes the problem.  An
 *     unsupported combination is an error, never a silent change of method
 *     (den_llama.cpp, "What this fork is": an FA quant pair that was not
 *     compiled silently fell back to f16-f16; Llaminar, "GPU Graph Capture":
 *     an unsupported configuration is an error).
 *   - Problems that only the device can see (a position or length held in
 *     device memory that is out of range) are reported by OR-ing a KVQ_ERR_*
 *     bit into the caller's device word `d_err` (nullable); the affected work
 *     is skipped, nothing traps.
 *   - Positions and lengths live in device memory and are advanced by the
 *     caller (Llaminar, "GPU Graph Capture": token positions and KV counters
 *     stay device-owned), so every call can be captured in a CUDA graph.
 *   - The library is stateless apart from cached device attributes and a
 *     per-thread error string; calls on different streams are independent.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,        /* a null pointer, a bad size or an inconsistent shape */
    KVQ_EUNSUPPORTED = 2,  /* a valid request the library does not implement */
    KVQ_EWORKSPACE = 3,    /* workspace missing or smaller than kvq_decode_workspace_bytes() */
    KVQ_ECUDA = 4          /* a CUDA call or kernel launch failed */
} kvq_status;

/* Codecs of a cache plane.
 * KVQ_CODEC_Q4_G64 -- 4-bit signed codes, one fp16 scale per group of 64 values,
 *   4.25 bits per value (den_llama.cpp, "What this fork is", quantized KV
 *   cache bullet; "build3 (working engine) -- additions", Q4_G64 row).
 *   Per group: scale = fp16_rne(absmax / 7) (fp32 quotient, saturated to
 *   65504), code = clamp(rne(x / (float)scale), -8, 7), code 0 if scale == 0.
 *   A row of head_dim values is head_dim/2 code bytes (byte j: value 2j in the
 *   low nibble, value 2j+1 in the high nibble, 4-bit two's complement) plus
 *   head_dim/64 fp16 scales.
 * KVQ_CODEC_Q8_0 -- the q8_0-style K codec of the mixed pair "-ctk q8_0 -ctv
 *   q4_g64" (den_llama.cpp, "Build3 (working engine)"): 32 int8 codes and one
 *   FP16 scale per group, scale = fp16_rne(absmax / 127), code =
 *   clamp(rne(x / (float)scale), -127, 127); a row is head_dim code bytes plus
 *   head_dim/32 fp16 scales (8.5 bits per value).
 * KVQ_CODEC_Q4_G32 -- the "q4_0" V cache of the shipped pair "-ctk q8_0 -ctv
 *   q4_0" (den_llama.cpp, "What's in the fork": the q8_0-q4_0 FlashAttention
 *   pair; "Results": the 65K serve run), whose format the pages do not give:
 *   the Q4_G64 rule and code layout with groups of 32 values (head_dim/32
 *   scales, 4.5 bits per value).  Not llama.cpp's q4_0 byte layout.
 * KVQ_CODEC_NVFP4 -- the NVFP4 KV type of the "-ctk nvfp4 -ctv nvfp4" and
 *   "-ctk q8_0 -ctv nvfp4" runs (den_llama.cpp, "What this fork is";
 *   "build3 (working engine) -- additions", NVFP4 KV row), whose format the
 *   pages do not give: NVIDIA's published NVFP4 without its per-tensor scale.
 *   Per block of 16 values: scale = E4M3(absmax / 6) (fp32 quotient; FP8
 *   E4M3: bias 7, 3 mantissa bits, largest finite 448), code = E2M1(x /
 *   (float)scale) (FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, sign in
 *   bit 3, a negative value that rounds to 0 keeps its sign), both rounded to
 *   nearest, ties to even, and held at the largest finite value; codes 0 when
 *   the scale is 0.  A row is head_dim/2 code bytes (Q4_G64's nibble order)
 *   plus head_dim/16 one-byte E4M3 scales (4.5 bits per value).
 * Dequantized value = (float)scale * code value, exact in fp32. */
typedef enum kvq_codec {
    KVQ_CODEC_Q4_G64 = 1,
    KVQ_CODEC_Q8_0 = 2,
    KVQ_CODEC_Q4_G32 = 3,
    KVQ_CODEC_NVFP4 = 4
} kvq_codec;

typedef enum kvq_dtype { KVQ_F32 = 0, KVQ_F16 = 1 } kvq_dtype;

/* Bits OR-ed into the caller's device error word. */
#define KVQ_ERR_APPEND_POS 1   /* pos0[s] < 0 or pos0[s] + n_new > capacity: sequence s skipped */
#define KVQ_ERR_KV_LEN 2       /* kv_len[s] < 0 or > max_kv_len: sequence s clamped to [0, max_kv_len] */
#define KVQ_ERR_TIMEOUT 4      /* a bounded device wait gave up; the outputs of that call are invalid */

/* Cache capacity (tokens per (sequence, kv head) slot) must be a multiple of this. */
#define KVQ_CAPACITY_ALIGN 64

/* One layer's K (or V) cache: two planes, both in device memory.
 *   qs     : code bytes, [n_seq][n_kv_heads][capacity][kvq_row_bytes(codec, head_dim)]
 *   scales : [n_seq][n_kv_heads][capacity][kvq_scales_per_row(codec, head_dim)] scales
 *            of kvq_scale_bytes(codec) bytes each (fp16; E4M3 bytes for NVFP4)
 * Both planes are 16-byte aligned.  head_dim is a multiple of 64 in
 * [64, 512]; capacity is a positive multiple of KVQ_CAPACITY_ALIGN. */
typedef struct kvq_cache {
    int32_t codec;          /* kvq_codec */
    int32_t n_seq;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t capacity;
    void *qs;
    void *scales;
} kvq_cache;

/* Bytes of one row of the code plane, or 0 for an unknown codec. */
int32_t kvq_row_bytes(int32_t codec, int32_t head_dim);
/* Scales in one row, or 0 for an unknown codec. */
int32_t kvq_scales_per_row(int32_t codec, int32_t head_dim);
/* Bytes of one scale (2: fp16; 1: E4M3 for NVFP4), or 0 for an unknown codec. */
int32_t kvq_scale_bytes(int32_t codec);

/* Failure-path self-test: enqueues one CTA that waits, with the bounded device
 * wait every kernel of the library uses for its copies, on a barrier nothing
 * completes.  After the wait's cycle limit (about 1 s) it ORs
 * KVQ_ERR_TIMEOUT into *d_err (DEVICE int32) and returns; nothing traps and
 * the context stays usable.  KVQ_EINVAL if d_err is NULL. */
kvq_status kvq_selftest_bounded_wait(int32_t *d_err, void *stream);

/* Quantize-on-append (the KV-cache append stage).
 *   k_src, v_src : DEVICE, [n_seq][n_new][n_kv_heads][head_dim], dtype src_dtype
 *                  (KVQ_F32 or KVQ_F16), 16-byte aligned.
 *   d_pos0       : DEVICE int32 [n_seq]; token i of sequence s is written at
 *                  cache position d_pos0[s] + i of every kv head.
 *   d_err        : DEVICE int32, nullable; KVQ_ERR_APPEND_POS is OR-ed in for a
 *                  sequence whose positions leave [0, capacity), and that
 *                  sequence is not written.
 * Either (k, k_src) or (v, v_src) may be NULL to append to one cache only;
 * k and v may use different codecs but must agree on n_seq, n_kv_heads and
 * head_dim.  The packed bytes are identical to the CPU reference rule above,
 * byte for byte.  Whole rows are written, so appends of different tokens never
 * share a byte. */
kvq_status kvq_quantize_append(const kvq_cache *k, const kvq_cache *v,
                               const void *k_src, const void *v_src, int32_t src_dtype,
                               int32_t n_new, const int32_t *d_pos0, int32_t *d_err,
                               void *stream);

/* Split count kvq_decode_attention uses for n_splits = 0 with these caches and
 * arguments on the current device.  One sequence: one wave of the decode
 * kernel's CTAs (which kernel runs, and how many of its CTAs fit on an SM,
 * depends on the codecs, head_dim and the query rows per kv head: one CTA per
 * SM for up to 8 rows over Q4_G64 V, two or three otherwise); a batch, whose
 * lengths may be ragged: up to four waves' worth.  Never fewer than 256 keys
 * per split.
 * Only codec, n_seq, n_kv_heads and head_dim of k and v are read (their plane
 * pointers may be NULL).  Returns 1 for invalid arguments. */
int32_t kvq_decode_default_splits(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q,
                                  int32_t max_kv_len);

/* Device workspace bytes kvq_decode_attention needs for these caches and
 * arguments (n_splits as passed to it, 0 = the default).  0 means none is
 * needed (also returned for invalid arguments). */
size_t kvq_decode_workspace_bytes(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q,
                                  int32_t max_kv_len, int32_t n_splits);

/* Decode / MTP-verify attention over the packed cache (the attention stage);
 * with n_q new prompt tokens it is the attention of a chunked prefill.
 *   k, v          : caches with the same n_seq, n_kv_heads, head_dim, capacity;
 *                   any pair of codecs.
 *   q             : DEVICE, [n_seq][n_q][n_heads][head_dim], dtype q_dtype, 16-byte aligned.
 *                   Query head h reads kv head h / (n_heads / n_kv_heads).
 *   softmax_scale : multiplies q.k (e.g. 1/sqrt(head_dim)).
 *   d_kv_len      : DEVICE int32 [n_seq], keys visible to the LAST query token
 *                   of each sequence; query token i (0-based) sees the first
 *                   d_kv_len[s] - n_q + i + 1 cache positions (the n_q new
 *                   tokens are the last n_q positions and attend causally to
 *                   each other; den_llama.cpp, "Results": MTP n-max 2).  A row
 *                   that sees no key gets out = 0 and out_lse = -inf.
 *   max_kv_len    : host bound on every d_kv_len[s], 1 <= max_kv_len <= capacity.
 *   n_splits      : the sequence range is cut into n_splits chunks per
 *                   (sequence, kv head) that run in parallel and are merged by
 *                   log-sum-exp; 0 = kvq_decode_default_splits(); 1..4096.
 *   out           : DEVICE fp32 [n_seq][n_q][n_heads][head_dim], softmax-weighted V.
 *   out_lse       : DEVICE fp32 [n_seq][n_q][n_heads], natural-log sum of
 *                   exp(scores); nullable.
 *   workspace     : DEVICE scratch of at least kvq_decode_workspace_bytes(),
 *                   256-byte aligned; may be NULL when that size is 0.  Its
 *                   contents need no initialisation and are not kept.
 *   d_err         : DEVICE int32, nullable (KVQ_ERR_KV_LEN, KVQ_ERR_TIMEOUT).
 * Arithmetic: codes (NVFP4: code values times their E4M3 scales) are exact in
 * fp16, dot products accumulate in fp32 and the softmax runs in fp32; the
 * softmax weights enter the weighted sum of V rounded to fp16. */
kvq_status kvq_decode_attention(const kvq_cache *k, const kvq_cache *v,
                                const void *q, int32_t q_dtype, int32_t n_q, int32_t n_heads,
                                float softmax_scale, const int32_t *d_kv_len, int32_t max_kv_len,
                                int32_t n_splits, float *out, float *out_lse,
                                void *workspace, size_t workspace_bytes, int32_t *d_err,
                                void *stream);

/* Log-sum-exp merge of partial attention results (one per split of the key range).
 * The source pages do not describe splitting the key range: this call is the
 * merge step of the library's own split-K decomposition (kvq_decode_attention
 * splits long ranges across CTAs), exposed for callers that split themselves,
 * e.g. a sequence sharded across devices.
 *   part_o   : DEVICE fp32 [n_splits][rows][head_dim], each part normalised over its keys.
 *   part_lse : DEVICE fp32 [n_splits][rows]; -inf marks an empty part (its part_o is ignored).
 *   out      : DEVICE fp32 [rows][head_dim] = sum_s w_s part_o[s] / sum_s w_s with
 *              w_s = exp(part_lse[s] - max_s part_lse[s]); 0 if every part is empty.
 *   out_lse  : DEVICE fp32 [rows], max + ln(sum_s w_s) (-inf if every part is empty); nullable.
 * 1 <= n_splits <= 4096, rows >= 0, head_dim a multiple of 4 in [4, 1024]. */
kvq_status kvq_merge_splits(const float *part_o, const float *part_lse, int32_t n_splits,
                            int32_t rows, int32_t head_dim, float *out, float *out_lse, void *stream);

/* Decode attention that allocates nothing and takes no workspace.
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory where they decode: code enqueuing work
 * while a CUDA graph is being captured (an allocation there is not a stream
 * operation), engines whose memory is all owned by their own pool, and paths
 * that cannot afford an allocation's implicit device synchronisation.
 * Arguments, results and errors are those of kvq_decode_attention; the split
 * scratch comes from a file-scope __device__ array of KVQ_STATIC_SCRATCH_BYTES
 * inside libkvq.so, which every GPU that loads the library keeps until the
 * process exits.  With n_splits = 0 the split count is lowered, if needed, to
 * the largest one whose scratch fits the array; an explicit n_splits whose
 * scratch (kvq_decode_workspace_bytes with the same arguments) exceeds that
 * size returns KVQ_EWORKSPACE before anything is launched.  The first call in
 * each CUDA context looks up the array's device address (with that context's
 * device current) and keeps it for that context; make that first call before
 * any stream capture.  After cudaDeviceReset (a new context) the next call
 * looks the address up again.
 * Every call on a device shares the one array and leaves its contents behind:
 * nothing in it needs to start at zero, but two calls that overlap on the GPU
 * (different streams, no ordering between them) race on it and give wrong
 * results.  The library allocates no memory in this call. */
#define KVQ_STATIC_SCRATCH_BYTES (8u << 20)
size_t kvq_static_scratch_bytes(void);
kvq_status kvq_decode_attention_static(const kvq_cache *k, const kvq_cache *v,
                                       const void *q, int32_t q_dtype, int32_t n_q, int32_t n_heads,
                                       float softmax_scale, const int32_t *d_kv_len, int32_t max_kv_len,
                                       int32_t n_splits, float *out, float *out_lse, int32_t *d_err,
                                       void *stream);

/* Host-tier KV streaming: decode attention for one sequence whose
 * authoritative cache lives in pinned host memory, with a bounded device pool
 * (den_llama.cpp, "Adaptive KV streaming (contributed)": the authoritative KV
 * tensors in pinned host memory, a bounded CUDA pool shared by resident pages
 * and a transfer ring, exact attention over the full context).
 *   k_host, v_host : the caches (n_seq = 1) whose planes are in pinned host
 *                    memory (cudaHostAlloc / cudaHostRegister); the library
 *                    only reads them, with cudaMemcpy2DAsync.
 *   k_dev, v_dev   : device caches of the same codecs and shape holding the
 *                    same first n_resident tokens (the resident part, read in
 *                    place); may be NULL when n_resident = 0.
 *   kv_len         : HOST int, keys visible to the last query token
 *                    (1 <= kv_len <= capacity of the host caches).
 *   page_tokens    : keys per streamed page, a positive multiple of
 *                    KVQ_CAPACITY_ALIGN; tokens n_resident .. kv_len - 1 are
 *                    streamed in pages through n_slots ring slots.
 *   ring           : DEVICE buffer of at least kvq_tiered_ring_bytes(), 256-byte
 *                    aligned (may be NULL when nothing is streamed).
 *   workspace      : DEVICE buffer of at least kvq_tiered_workspace_bytes(),
 *                    256-byte aligned (per-part partials and split scratch).
 *   q, q_dtype, n_q, n_heads, softmax_scale, out, out_lse, d_err: as in
 *                    kvq_decode_attention (one sequence).
 * The result equals kvq_decode_attention over the whole cache up to rounding:
 * the resident prefix and every page are decoded into partials (o, lse) that
 * one merge combines.  Page copies run on a copy stream the library creates
 * once per device and joins to `stream` with events, so the copy of a page
 * overlaps the decode of earlier ones; the copy into a slot waits until the
 * slot's previous page has been decoded.  Arguments are checked on the host
 * before anything is enqueued (KVQ_EINVAL / KVQ_EUNSUPPORTED for n_seq != 1 /
 * KVQ_EWORKSPACE). */
size_t kvq_tiered_ring_bytes(const kvq_cache *k_host, const kvq_cache *v_host, int32_t page_tokens,
                             int32_t n_slots);
size_t kvq_tiered_workspace_bytes(const kvq_cache *k_host, const kvq_cache *v_host, const kvq_cache *k_dev,
                                  const kvq_cache *v_dev, int32_t n_heads, int32_t n_q, int32_t kv_len,
                                  int32_t n_resident, int32_t page_tokens);
kvq_status kvq_decode_attention_tiered(const kvq_cache *k_host, const kvq_cache *v_host,
                                       const kvq_cache *k_dev, const kvq_cache *v_dev, int32_t n_resident,
                                       const void *q, int32_t q_dtype, int32_t n_q, int32_t n_heads,
                                       float softmax_scale, int32_t kv_len, int32_t page_tokens, int32_t n_slots,
                                       void *ring, size_t ring_bytes, float *out, float *out_lse,
                                       void *workspace, size_t workspace_bytes, int32_t *d_err, void *stream);

/* Dequantize a whole cache to fp32 [n_seq][n_kv_heads][capacity][head_dim] on
 * the device (scale * code, exact).  For inspection and testing. */
kvq_status kvq_dequantize(const kvq_cache *c, float *out, void *stream);

/* Static description of a status code. */
const char *kvq_status_string(int32_t status);
/* Detail of the last non-OK status returned on the calling thread ("" if none). */
const char *kvq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
