// kvq_api.cu -- the extern "C" entry points of libkvq.so declared in kvq.h:
// argument checks on the host (nothing is launched on a bad argument), the
// choice of split count and workspace layout, and the kernel launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kvq_internal.cuh"

namespace {

thread_local char g_last_error[512] = "";

kvq_status fail(kvq_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kvq_status cuda_status(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return KVQ_OK;
    return fail(KVQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_codec(int32_t c)
{
    return c == KVQ_CODEC_Q4_G64 || c == KVQ_CODEC_Q8_0 || c == KVQ_CODEC_Q4_G32 || c == KVQ_CODEC_NVFP4;
}

bool valid_head_dim(int32_t d) { return d == 64 || d == 128 || d == 256 || d == 512; }

kvq_status check_cache(const kvq_cache *c, const char *name)
{
    if (!c) return fail(KVQ_EINVAL, "%s: cache is NULL", name);
    if (!valid_codec(c->codec)) return fail(KVQ_EINVAL, "%s: unknown codec %d", name, c->codec);
    if (c->n_seq <= 0 || c->n_kv_heads <= 0)
        return fail(KVQ_EINVAL, "%s: n_seq=%d n_kv_heads=%d must be positive", name, c->n_seq, c->n_kv_heads);
    if (c->head_dim <= 0 || c->head_dim % 64 != 0 || c->head_dim > 512)
        return fail(KVQ_EINVAL, "%s: head_dim=%d must be a multiple of 64 in [64, 512]", name, c->head_dim);
    if (!valid_head_dim(c->head_dim))
        return fail(KVQ_EUNSUPPORTED, "%s: head_dim=%d is not one of 64, 128, 256, 512", name, c->head_dim);
    if (c->capacity <= 0 || c->capacity % KVQ_CAPACITY_ALIGN != 0)
        return fail(KVQ_EINVAL, "%s: capacity=%d must be a positive multiple of %d", name, c->capacity,
                    KVQ_CAPACITY_ALIGN);
    if (!c->qs || !c->scales) return fail(KVQ_EINVAL, "%s: qs/scales plane is NULL", name);
    if (!aligned16(c->qs) || !aligned16(c->scales))
        return fail(KVQ_EINVAL, "%s: qs/scales planes must be 16-byte aligned", name);
    return KVQ_OK;
}

kvq::Plane plane_of(const kvq_cache *c)
{
    return kvq::Plane{c->codec, static_cast<uint8_t *>(c->qs), static_cast<uint8_t *>(c->scales)};
}

int sm_count()
{
    static kvq::PerDevice pd;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    const int n = kvq::per_device(pd, dev, [dev]() -> int {
        int v = 0;
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 0;
    });
    return n > 0 ? n : 148;
}

constexpr int kMaxSplits = 4096;

bool split_args_ok(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q, int32_t max_kv_len)
{
    return k && v && k->n_seq > 0 && k->n_kv_heads > 0 && k->head_dim > 0 && n_heads > 0 && n_q > 0 &&
           n_heads % k->n_kv_heads == 0 && max_kv_len > 0;
}

// Arguments the split policy reads are valid (checked by every caller).
int resolve_splits(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q, int32_t max_kv_len,
                   int32_t n_splits)
{
    if (n_splits > 0) return n_splits;
    const int rows = n_q * (n_heads / k->n_kv_heads);
    // one CTA per (sequence, kv head, block of query rows) and split; prompt
    // chunks the tcgen05 kernel takes come in blocks of 128 rows
    const bool umma = kvq::prefill_umma_shape(k->codec, v->codec, k->head_dim, rows) &&
                      kvq::prefill_umma_ctas_per_sm(k->codec, v->codec, k->head_dim) > 0;
    const int64_t blocks = umma ? kvq::ceil_div(rows, kvq::kUmmaRowsPerCta)
                                : (k->head_dim <= 256 ? kvq::tc_row_blocks(rows) : 1);
    const int64_t units = (int64_t)k->n_seq * k->n_kv_heads * blocks;
    // CTAs of the kernel an SM holds (3 where the occupancy is unknown)
    int per_sm = umma ? kvq::prefill_umma_ctas_per_sm(k->codec, v->codec, k->head_dim)
                      : kvq::decode_ctas_per_sm(k->codec, v->codec, k->head_dim, rows);
    if (per_sm <= 0) per_sm = 3;
    if (umma) {
        // one CTA per SM and many tiles per CTA: the split count whose waves
        // divide the work most evenly (ceil(units * s / slots) / s smallest, the
        // fewest splits among equals; at most 8, so the partials stay small).
        // 96 units on 152 SMs: 3 splits, 2 full waves.
        const int64_t slots = (int64_t)per_sm * sm_count();
        const int64_t max_s = kvq::ceil_div(max_kv_len, 256) < 8 ? kvq::ceil_div(max_kv_len, 256) : 8;
        int64_t best = 1;
        double best_cost = 1e30;
        for (int64_t c = 1; c <= (max_s > 1 ? max_s : 1); ++c) {
            const double cost = (double)kvq::ceil_div(units * c, slots) / (double)c;
            if (cost < best_cost - 1e-9) best_cost = cost, best = c;
        }
        return (int)best;
    }
    int64_t target;
    if (k->n_seq == 1) {
        // one wave of the decode kernel's CTAs
        target = (int64_t)per_sm * sm_count();
    } else {
        // a batch, whose lengths may be ragged: up to four waves so that the
        // longest sequence is cut finely enough (every sequence gets the same
        // number of splits); 16 sequences x 18 rows per kv head (2 CTAs per SM):
        // 19 splits, measured best between 16 and 20 (29, from 3 CTAs per SM,
        // was 9% slower)
        const int64_t waves = k->n_seq < 4 ? k->n_seq : 4;
        target = (int64_t)per_sm * sm_count() * waves;
    }
    int64_t s = kvq::ceil_div(target, units);
    const int64_t max_useful = kvq::ceil_div(max_kv_len, 256);      // at least 256 tokens a split
    if (s > max_useful) s = max_useful;
    if (s < 1) s = 1;
    // splits are whole 64-token tiles (split_range): with t tiles and s splits
    // of ceil(t / s) tiles each, only ceil(t / ceil(t / s)) of them get any;
    // ask for exactly those (the same longest split, no empty ones)
    const int64_t tiles = kvq::ceil_div(max_kv_len, 64);
    if (tiles > 0) s = kvq::ceil_div(tiles, kvq::ceil_div(tiles, s));
    if (s > kMaxSplits) s = kMaxSplits;
    return (int)s;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

void kvq::set_last_error(const char *msg)
{
    snprintf(g_last_error, sizeof g_last_error, "%s", msg);
}

kvq_status kvq::fail_msg(kvq_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

int kvq::resolve_decode_splits(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q,
                               int32_t max_kv_len, int32_t n_splits)
{
    return resolve_splits(k, v, n_heads, n_q, max_kv_len, n_splits);
}

kvq_status kvq::decode_checked(const kvq_cache *k, const kvq_cache *v, const void *q, int q_dtype, int n_q,
                               int n_heads, float softmax_scale, const int32_t *d_kv_len, int fixed_len,
                               int causal_extra, int max_kv_len, int n_splits, float *out, float *out_lse,
                               void *workspace, int32_t *d_err, cudaStream_t cs)
{
    kvq::DecodeArgs a{};
    a.k = plane_of(k);
    a.v = plane_of(v);
    a.q = q;
    a.n_seq = k->n_seq;
    a.n_kv_heads = k->n_kv_heads;
    a.n_heads = n_heads;
    a.n_q = n_q;
    a.head_dim = k->head_dim;
    a.capacity = k->capacity;
    a.scale_log2 = softmax_scale * kvq::kLog2e;
    a.kv_len = d_kv_len;
    a.fixed_len = fixed_len;
    a.causal_extra = causal_extra;
    a.max_kv_len = max_kv_len;
    a.n_splits = n_splits;
    a.out = out;
    a.out_lse = out_lse;
    a.err = d_err;
    const size_t rows = (size_t)k->n_seq * n_q * n_heads;
    if (n_splits > 1) {
        a.part_o = static_cast<float *>(workspace);
        a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                               align256((size_t)n_splits * rows * k->head_dim * sizeof(float)));
    }
    cudaError_t le;
    if (kvq::decode_tc_supported(a)) le = kvq::launch_decode_tc(a, q_dtype, cs);
    else le = kvq::launch_decode_simt(a, q_dtype, cs);
    kvq_status st;
    if ((st = cuda_status(le, "decode launch")) != KVQ_OK) return st;
    if (n_splits > 1)
        return cuda_status(kvq::launch_merge(a.part_o, a.part_lse, n_splits, (int)rows, k->head_dim, out, out_lse, cs),
                           "merge launch");
    return KVQ_OK;
}

kvq_status kvq::check_cache_args(const kvq_cache *c, const char *name) { return check_cache(c, name); }

extern "C" {

int32_t kvq_row_bytes(int32_t codec, int32_t head_dim)
{
    return valid_codec(codec) ? kvq::row_bytes(codec, head_dim) : 0;
}

int32_t kvq_scales_per_row(int32_t codec, int32_t head_dim)
{
    return valid_codec(codec) ? kvq::scales_per_row(codec, head_dim) : 0;
}

int32_t kvq_scale_bytes(int32_t codec)
{
    return valid_codec(codec) ? kvq::scale_bytes(codec) : 0;
}

const char *kvq_status_string(int32_t status)
{
    switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument";
    case KVQ_EUNSUPPORTED: return "unsupported combination";
    case KVQ_EWORKSPACE: return "workspace missing or too small";
    case KVQ_ECUDA: return "CUDA error";
    default: return "unknown status";
    }
}

const char *kvq_last_error(void) { return g_last_error; }

kvq_status kvq_quantize_append(const kvq_cache *k, const kvq_cache *v, const void *k_src, const void *v_src,
                               int32_t src_dtype, int32_t n_new, const int32_t *d_pos0, int32_t *d_err,
                               void *stream)
{
    g_last_error[0] = 0;
    if (!k && !v) return fail(KVQ_EINVAL, "append: both caches are NULL");
    if ((k == nullptr) != (k_src == nullptr)) return fail(KVQ_EINVAL, "append: k and k_src must both be given or both NULL");
    if ((v == nullptr) != (v_src == nullptr)) return fail(KVQ_EINVAL, "append: v and v_src must both be given or both NULL");
    kvq_status st;
    if (k && (st = check_cache(k, "append k")) != KVQ_OK) return st;
    if (v && (st = check_cache(v, "append v")) != KVQ_OK) return st;
    if (k && v && (k->n_seq != v->n_seq || k->n_kv_heads != v->n_kv_heads || k->head_dim != v->head_dim ||
                   k->capacity != v->capacity))
        return fail(KVQ_EINVAL, "append: k and v caches disagree on n_seq/n_kv_heads/head_dim/capacity");
    if (src_dtype != KVQ_F32 && src_dtype != KVQ_F16) return fail(KVQ_EINVAL, "append: src_dtype %d", src_dtype);
    if (n_new < 0) return fail(KVQ_EINVAL, "append: n_new=%d", n_new);
    if (!d_pos0) return fail(KVQ_EINVAL, "append: d_pos0 is NULL");
    if ((k_src && !aligned16(k_src)) || (v_src && !aligned16(v_src)))
        return fail(KVQ_EINVAL, "append: sources must be 16-byte aligned");
    if (n_new == 0) return KVQ_OK;
    const kvq_cache *c0 = k ? k : v;
    if (c0->n_seq > 0 && (int64_t)n_new * c0->n_seq * c0->n_kv_heads * 2 > (int64_t)0x7FFFFFFF * 8)
        return fail(KVQ_EINVAL, "append: too many rows for one call");
    kvq::AppendArgs a{};
    int n = 0;
    if (k) { a.plane[n] = plane_of(k); a.src[n] = k_src; ++n; }
    if (v) { a.plane[n] = plane_of(v); a.src[n] = v_src; ++n; }
    a.n_planes = n;
    a.n_seq = c0->n_seq;
    a.n_new = n_new;
    a.n_kv_heads = c0->n_kv_heads;
    a.head_dim = c0->head_dim;
    a.capacity = c0->capacity;
    a.pos0 = d_pos0;
    a.err = d_err;
    return cuda_status(kvq::launch_append(a, src_dtype == KVQ_F16, static_cast<cudaStream_t>(stream)),
                       "append launch");
}

int32_t kvq_decode_default_splits(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q,
                                  int32_t max_kv_len)
{
    if (!split_args_ok(k, v, n_heads, n_q, max_kv_len)) return 1;
    return resolve_splits(k, v, n_heads, n_q, max_kv_len, 0);
}

size_t kvq_decode_workspace_bytes(const kvq_cache *k, const kvq_cache *v, int32_t n_heads, int32_t n_q,
                                  int32_t max_kv_len, int32_t n_splits)
{
    if (!split_args_ok(k, v, n_heads, n_q, max_kv_len) || n_splits < 0) return 0;
    const int s = resolve_splits(k, v, n_heads, n_q, max_kv_len, n_splits);
    if (s <= 1) return 0;
    const size_t rows = (size_t)k->n_seq * n_q * n_heads;
    return align256((size_t)s * rows * k->head_dim * sizeof(float)) + align256((size_t)s * rows * sizeof(float));
}

kvq_status kvq_decode_attention(const kvq_cache *k, const kvq_cache *v, const void *q, int32_t q_dtype,
                                int32_t n_q, int32_t n_heads, float softmax_scale, const int32_t *d_kv_len,
                                int32_t max_kv_len, int32_t n_splits, float *out, float *out_lse,
                                void *workspace, size_t workspace_bytes, int32_t *d_err, void *stream)
{
    g_last_error[0] = 0;
    kvq_status st;
    if ((st = check_cache(k, "decode k")) != KVQ_OK) return st;
    if ((st = check_cache(v, "decode v")) != KVQ_OK) return st;
    if (k->n_seq != v->n_seq || k->n_kv_heads != v->n_kv_heads || k->head_dim != v->head_dim ||
        k->capacity != v->capacity)
        return fail(KVQ_EINVAL, "decode: k and v caches disagree on n_seq/n_kv_heads/head_dim/capacity");
    if (!q) return fail(KVQ_EINVAL, "decode: q is NULL");
    if (!aligned16(q)) return fail(KVQ_EINVAL, "decode: q must be 16-byte aligned");
    if (q_dtype != KVQ_F32 && q_dtype != KVQ_F16) return fail(KVQ_EINVAL, "decode: q_dtype %d", q_dtype);
    if (n_q <= 0) return fail(KVQ_EINVAL, "decode: n_q=%d", n_q);
    if (n_heads <= 0 || n_heads % k->n_kv_heads != 0)
        return fail(KVQ_EINVAL, "decode: n_heads=%d is not a positive multiple of n_kv_heads=%d", n_heads,
                    k->n_kv_heads);
    if (!std::isfinite(softmax_scale)) return fail(KVQ_EINVAL, "decode: softmax_scale is not finite");
    if (!d_kv_len) return fail(KVQ_EINVAL, "decode: d_kv_len is NULL");
    if (max_kv_len < 1 || max_kv_len > k->capacity)
        return fail(KVQ_EINVAL, "decode: max_kv_len=%d outside [1, capacity=%d]", max_kv_len, k->capacity);
    if (n_splits < 0 || n_splits > kMaxSplits)
        return fail(KVQ_EINVAL, "decode: n_splits=%d outside [0, %d]", n_splits, kMaxSplits);
    if (!out) return fail(KVQ_EINVAL, "decode: out is NULL");
    const int s = resolve_splits(k, v, n_heads, n_q, max_kv_len, n_splits);
    const size_t need = kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, n_splits);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(KVQ_EWORKSPACE, "decode: workspace %zu bytes given, %zu needed", workspace ? workspace_bytes : 0,
                    need);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(KVQ_EINVAL, "decode: workspace must be 256-byte aligned");
    if (s > 65535) return fail(KVQ_EINVAL, "decode: too many splits");
    if (k->n_seq > 65535 || k->n_kv_heads > 65535) return fail(KVQ_EUNSUPPORTED, "decode: grid too large");
    return kvq::decode_checked(k, v, q, q_dtype, n_q, n_heads, softmax_scale, d_kv_len, -1, 0, max_kv_len, s, out,
                               out_lse, workspace, d_err, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_merge_splits(const float *part_o, const float *part_lse, int32_t n_splits, int32_t rows,
                            int32_t head_dim, float *out, float *out_lse, void *stream)
{
    g_last_error[0] = 0;
    if (n_splits < 1 || n_splits > kMaxSplits)
        return fail(KVQ_EINVAL, "merge: n_splits=%d outside [1, %d]", n_splits, kMaxSplits);
    if (rows < 0) return fail(KVQ_EINVAL, "merge: rows=%d", rows);
    if (head_dim < 4 || head_dim > 1024 || head_dim % 4 != 0)
        return fail(KVQ_EINVAL, "merge: head_dim=%d must be a multiple of 4 in [4, 1024]", head_dim);
    if (rows == 0) return KVQ_OK;
    if (!part_o || !part_lse || !out) return fail(KVQ_EINVAL, "merge: NULL pointer");
    if (!aligned16(part_o) || !aligned16(out)) return fail(KVQ_EINVAL, "merge: part_o/out must be 16-byte aligned");
    return cuda_status(kvq::launch_merge(part_o, part_lse, n_splits, rows, head_dim, out, out_lse,
                                         static_cast<cudaStream_t>(stream)),
                       "merge launch");
}

kvq_status kvq_dequantize(const kvq_cache *c, float *out, void *stream)
{
    g_last_error[0] = 0;
    kvq_status st;
    if ((st = check_cache(c, "dequantize")) != KVQ_OK) return st;
    if (!out || !aligned16(out)) return fail(KVQ_EINVAL, "dequantize: out is NULL or not 16-byte aligned");
    const int64_t n_rows = (int64_t)c->n_seq * c->n_kv_heads * c->capacity;
    return cuda_status(kvq::launch_dequant(plane_of(c), n_rows, c->head_dim, out, static_cast<cudaStream_t>(stream)),
                       "dequantize launch");
}

}  // extern "C"
