// kvq_tiered.cu -- decode attention over a cache whose authoritative planes
// live in pinned host memory, with a bounded device pool: the first
// n_resident tokens are kept on the device, the rest are streamed through a
// ring of page slots (den_llama.cpp, "Adaptive KV streaming (contributed)":
// the authoritative KV in pinned host memory, a bounded CUDA pool shared by
// resident pages and a transfer ring, exact attention over the full context).
//
// How: softmax attention over a key range is the log-sum-exp combination of
// attention over its parts, so the context is cut into parts -- the resident
// prefix, then pages of page_tokens keys -- each part is decoded by the
// library's decode kernels into a partial (o, lse) normalised over the part,
// and the partials are merged by the merge kernel.  A page is copied from the
// host planes into ring slot p % n_slots by cudaMemcpy2DAsync (one call per
// plane, all kv heads at once) on copy streams of the library's own (pages
// round-robin over them); the copy of page p waits for the decode of page
// p - n_slots (which read that slot), the decode of page p waits for its copy,
// so copies of later pages run while earlier ones are decoded.  One sequence
// (a single serving slot).
#include <cmath>
#include <cstring>

#include "kvq_internal.cuh"

namespace {

constexpr int kMaxParts = 4096;

struct RingLayout {
    size_t kqs, ksc, vqs, vsc, slot;   // offsets inside a slot, slot size
};

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

RingLayout ring_layout(const kvq_cache *k, const kvq_cache *v, int page_tokens)
{
    const size_t rows = (size_t)k->n_kv_heads * page_tokens;
    RingLayout r{};
    r.kqs = 0;
    r.ksc = r.kqs + a256(rows * kvq::row_bytes(k->codec, k->head_dim));
    r.vqs = r.ksc + a256(rows * kvq::scale_row_bytes(k->codec, k->head_dim));
    r.vsc = r.vqs + a256(rows * kvq::row_bytes(v->codec, v->head_dim));
    r.slot = r.vsc + a256(rows * kvq::scale_row_bytes(v->codec, v->head_dim));
    return r;
}

int n_pages_of(int kv_len, int n_resident, int page_tokens)
{
    return kv_len > n_resident ? (int)kvq::ceil_div(kv_len - n_resident, page_tokens) : 0;
}

// A page-slot view of the caches: one sequence, capacity page_tokens.
void slot_views(const kvq_cache *k, const kvq_cache *v, int page_tokens, uint8_t *slot, const RingLayout &r,
                kvq_cache &ks, kvq_cache &vs)
{
    ks = *k;
    vs = *v;
    ks.capacity = vs.capacity = page_tokens;
    ks.qs = slot + r.kqs;
    ks.scales = slot + r.ksc;
    vs.qs = slot + r.vqs;
    vs.scales = slot + r.vsc;
}

// The split workspace the largest part needs (parts run one after the other
// on the caller's stream and share it).
size_t inner_ws(const kvq_cache *k_dev, const kvq_cache *v_dev, const kvq_cache *k, const kvq_cache *v,
                int32_t n_heads, int32_t n_q, int32_t n_resident, int32_t page_tokens)
{
    size_t need = 0;
    if (n_resident > 0 && k_dev && v_dev)
        need = kvq_decode_workspace_bytes(k_dev, v_dev, n_heads, n_q, n_resident, 0);
    kvq_cache ks = *k, vs = *v;
    ks.capacity = vs.capacity = page_tokens;
    const size_t p = kvq_decode_workspace_bytes(&ks, &vs, n_heads, n_q, page_tokens, 0);
    return need > p ? need : p;
}

// The library's copy streams on the current device (created once per device);
// consecutive pages go to different streams.  One: on GB300 a page copy from
// pinned host memory runs at ~160 GB/s whether 1, 2, 4 or 8 streams share
// the pages (measured), so more streams only add events.
constexpr int kCopyStreams = 1;

struct CopyStreams {
    std::mutex mu;
    cudaStream_t s[kvq::PerDevice::kMaxDevices][kCopyStreams] = {};
};

cudaError_t copy_streams(cudaStream_t (&out)[kCopyStreams])
{
    static CopyStreams cs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kvq::PerDevice::kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(cs.mu);
    for (int i = 0; i < kCopyStreams; ++i) {
        if (!cs.s[dev][i]) {
            e = cudaStreamCreateWithFlags(&cs.s[dev][i], cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                cs.s[dev][i] = nullptr;
                return e;
            }
        }
        out[i] = cs.s[dev][i];
    }
    return cudaSuccess;
}

bool same_shape(const kvq_cache *a, const kvq_cache *b)
{
    return a->codec == b->codec && a->n_seq == b->n_seq && a->n_kv_heads == b->n_kv_heads &&
           a->head_dim == b->head_dim;
}

kvq_status check_tiered(const kvq_cache *k, const kvq_cache *v, const kvq_cache *k_dev, const kvq_cache *v_dev,
                        int32_t n_resident, int32_t n_heads, int32_t n_q, int32_t kv_len, int32_t page_tokens,
                        int32_t n_slots)
{
    kvq_status st;
    if ((st = kvq::check_cache_args(k, "tiered k")) != KVQ_OK) return st;
    if ((st = kvq::check_cache_args(v, "tiered v")) != KVQ_OK) return st;
    if (k->n_seq != 1 || v->n_seq != 1)
        return kvq::fail_msg(KVQ_EUNSUPPORTED, "tiered: one sequence only (n_seq=%d)", k->n_seq);
    if (k->n_kv_heads != v->n_kv_heads || k->head_dim != v->head_dim || k->capacity != v->capacity)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: k and v caches disagree on n_kv_heads/head_dim/capacity");
    if (n_heads <= 0 || n_heads % k->n_kv_heads != 0)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: n_heads=%d is not a positive multiple of n_kv_heads=%d", n_heads,
                             k->n_kv_heads);
    if (n_q <= 0) return kvq::fail_msg(KVQ_EINVAL, "tiered: n_q=%d", n_q);
    if (kv_len < 1 || kv_len > k->capacity)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: kv_len=%d outside [1, capacity=%d]", kv_len, k->capacity);
    if (page_tokens <= 0 || page_tokens % KVQ_CAPACITY_ALIGN != 0)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: page_tokens=%d must be a positive multiple of %d", page_tokens,
                             KVQ_CAPACITY_ALIGN);
    if (n_slots < 1) return kvq::fail_msg(KVQ_EINVAL, "tiered: n_slots=%d", n_slots);
    if (n_resident < 0 || n_resident > kv_len)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: n_resident=%d outside [0, kv_len=%d]", n_resident, kv_len);
    if (n_resident > 0) {
        if (!k_dev || !v_dev) return kvq::fail_msg(KVQ_EINVAL, "tiered: n_resident > 0 needs the device caches");
        if ((st = kvq::check_cache_args(k_dev, "tiered resident k")) != KVQ_OK) return st;
        if ((st = kvq::check_cache_args(v_dev, "tiered resident v")) != KVQ_OK) return st;
        if (!same_shape(k_dev, k) || !same_shape(v_dev, v))
            return kvq::fail_msg(KVQ_EINVAL, "tiered: resident caches differ from the host caches in codec or shape");
        if (k_dev->capacity != v_dev->capacity || n_resident > k_dev->capacity)
            return kvq::fail_msg(KVQ_EINVAL, "tiered: n_resident=%d exceeds the resident capacity", n_resident);
    }
    const int parts = (n_resident > 0 ? 1 : 0) + n_pages_of(kv_len, n_resident, page_tokens);
    if (parts > kMaxParts)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: %d parts (resident + pages) exceed %d", parts, kMaxParts);
    return KVQ_OK;
}

}  // namespace

extern "C" {

size_t kvq_tiered_ring_bytes(const kvq_cache *k_host, const kvq_cache *v_host, int32_t page_tokens,
                             int32_t n_slots)
{
    if (!k_host || !v_host || page_tokens <= 0 || n_slots < 1 || k_host->n_kv_heads <= 0 || k_host->head_dim <= 0)
        return 0;
    return (size_t)n_slots * ring_layout(k_host, v_host, page_tokens).slot;
}

size_t kvq_tiered_workspace_bytes(const kvq_cache *k_host, const kvq_cache *v_host, const kvq_cache *k_dev,
                                  const kvq_cache *v_dev, int32_t n_heads, int32_t n_q, int32_t kv_len,
                                  int32_t n_resident, int32_t page_tokens)
{
    if (!k_host || !v_host || n_heads <= 0 || n_q <= 0 || kv_len < 1 || page_tokens <= 0 || n_resident < 0 ||
        k_host->n_kv_heads <= 0 || n_heads % k_host->n_kv_heads != 0)
        return 0;
    const int parts = (n_resident > 0 ? 1 : 0) + n_pages_of(kv_len, n_resident, page_tokens);
    const size_t rows = (size_t)n_q * n_heads;
    return a256((size_t)parts * rows * k_host->head_dim * sizeof(float)) + a256((size_t)parts * rows * sizeof(float)) +
           a256(inner_ws(k_dev, v_dev, k_host, v_host, n_heads, n_q, n_resident, page_tokens));
}

kvq_status kvq_decode_attention_tiered(const kvq_cache *k_host, const kvq_cache *v_host, const kvq_cache *k_dev,
                                       const kvq_cache *v_dev, int32_t n_resident, const void *q, int32_t q_dtype,
                                       int32_t n_q, int32_t n_heads, float softmax_scale, int32_t kv_len,
                                       int32_t page_tokens, int32_t n_slots, void *ring, size_t ring_bytes,
                                       float *out, float *out_lse, void *workspace, size_t workspace_bytes,
                                       int32_t *d_err, void *stream)
{
    kvq::set_last_error("");
    kvq_status st = check_tiered(k_host, v_host, k_dev, v_dev, n_resident, n_heads, n_q, kv_len, page_tokens, n_slots);
    if (st != KVQ_OK) return st;
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u)) return kvq::fail_msg(KVQ_EINVAL, "tiered: q NULL or unaligned");
    if (q_dtype != KVQ_F32 && q_dtype != KVQ_F16) return kvq::fail_msg(KVQ_EINVAL, "tiered: q_dtype %d", q_dtype);
    if (!std::isfinite(softmax_scale)) return kvq::fail_msg(KVQ_EINVAL, "tiered: softmax_scale is not finite");
    if (!out || (reinterpret_cast<uintptr_t>(out) & 15u)) return kvq::fail_msg(KVQ_EINVAL, "tiered: out NULL or unaligned");
    const int n_pages = n_pages_of(kv_len, n_resident, page_tokens);
    const size_t ring_need = kvq_tiered_ring_bytes(k_host, v_host, page_tokens, n_slots);
    if (n_pages > 0 && (!ring || ring_bytes < ring_need))
        return kvq::fail_msg(KVQ_EWORKSPACE, "tiered: ring %zu bytes given, %zu needed", ring ? ring_bytes : 0,
                             ring_need);
    if (n_pages > 0 && (reinterpret_cast<uintptr_t>(ring) & 255u))
        return kvq::fail_msg(KVQ_EINVAL, "tiered: ring must be 256-byte aligned");
    const size_t ws_need =
        kvq_tiered_workspace_bytes(k_host, v_host, k_dev, v_dev, n_heads, n_q, kv_len, n_resident, page_tokens);
    if (!workspace || workspace_bytes < ws_need)
        return kvq::fail_msg(KVQ_EWORKSPACE, "tiered: workspace %zu bytes given, %zu needed",
                             workspace ? workspace_bytes : 0, ws_need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return kvq::fail_msg(KVQ_EINVAL, "tiered: workspace must be 256-byte aligned");

    const int parts = (n_resident > 0 ? 1 : 0) + n_pages;
    const size_t rows = (size_t)n_q * n_heads;
    const int D = k_host->head_dim;
    float *part_o = static_cast<float *>(workspace);
    float *part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + a256((size_t)parts * rows * D * 4));
    void *inner = static_cast<char *>(workspace) + a256((size_t)parts * rows * D * 4) + a256((size_t)parts * rows * 4);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    auto decode_part = [&](const kvq_cache *kc, const kvq_cache *vc, int len, int end, int idx) -> kvq_status {
        const int s = kvq::resolve_decode_splits(kc, vc, n_heads, n_q, len, 0);
        // query token i sees len + (kv_len - end) - n_q + i + 1 keys of this part
        return kvq::decode_checked(kc, vc, q, q_dtype, n_q, n_heads, softmax_scale, nullptr, len, kv_len - end, len,
                                   s, part_o + (size_t)idx * rows * D, part_lse + (size_t)idx * rows, inner, d_err, cs);
    };
    int idx = 0;
    if (n_resident > 0) {
        if ((st = decode_part(k_dev, v_dev, n_resident, n_resident, idx++)) != KVQ_OK) return st;
    }
    if (n_pages > 0) {
        cudaStream_t cps[kCopyStreams] = {};
        cudaError_t e = copy_streams(cps);
        if (e != cudaSuccess) return kvq::fail_msg(KVQ_ECUDA, "tiered: copy stream: %s", cudaGetErrorString(e));
        const RingLayout rl = ring_layout(k_host, v_host, page_tokens);
        const int kv = k_host->n_kv_heads, cap = k_host->capacity;
        const size_t krb = kvq::row_bytes(k_host->codec, D), ksb = kvq::scale_row_bytes(k_host->codec, D);
        const size_t vrb = kvq::row_bytes(v_host->codec, D), vsb = kvq::scale_row_bytes(v_host->codec, D);
        // events: the copy stream starts after the work the caller enqueued
        // before this call; one "copied" event per page, one "freed" event per
        // slot (its last decode has read it)
        cudaEvent_t start = nullptr;
        cudaEvent_t *ev = new cudaEvent_t[(size_t)n_pages + n_slots]();
        auto cleanup = [&]() {
            if (start) cudaEventDestroy(start);
            for (int i = 0; i < n_pages + n_slots; ++i)
                if (ev[i]) cudaEventDestroy(ev[i]);
            delete[] ev;
        };
        auto cuda_fail = [&](cudaError_t err, const char *what) {
            cleanup();
            return kvq::fail_msg(KVQ_ECUDA, "tiered: %s: %s", what, cudaGetErrorString(err));
        };
        if ((e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e, "event");
        for (int i = 0; i < n_pages + n_slots; ++i)
            if ((e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e, "event");
        cudaEvent_t *copied = ev, *freed = ev + n_pages;
        if ((e = cudaEventRecord(start, cs)) != cudaSuccess) return cuda_fail(e, "stream join");
        for (int i = 0; i < kCopyStreams && i < n_pages; ++i)
            if ((e = cudaStreamWaitEvent(cps[i], start, 0)) != cudaSuccess) return cuda_fail(e, "stream join");
        for (int p = 0; p < n_pages; ++p) {
            const int slot = p % n_slots;
            cudaStream_t cp = cps[p % kCopyStreams];
            const int t0 = n_resident + p * page_tokens;
            const int len = kv_len - t0 < page_tokens ? kv_len - t0 : page_tokens;
            uint8_t *base = static_cast<uint8_t *>(ring) + (size_t)slot * rl.slot;
            if (p >= n_slots && (e = cudaStreamWaitEvent(cp, freed[slot], 0)) != cudaSuccess)
                return cuda_fail(e, "slot wait");
            // all kv heads of the page, one call per plane: rows t0 .. t0 + len of
            // each head's slot (pitch capacity rows) into the slot (pitch page rows)
            const struct { void *dst; const void *src; size_t rb; } planes[4] = {
                {base + rl.kqs, static_cast<const uint8_t *>(k_host->qs) + (size_t)t0 * krb, krb},
                {base + rl.ksc, static_cast<const uint8_t *>(k_host->scales) + (size_t)t0 * ksb, ksb},
                {base + rl.vqs, static_cast<const uint8_t *>(v_host->qs) + (size_t)t0 * vrb, vrb},
                {base + rl.vsc, static_cast<const uint8_t *>(v_host->scales) + (size_t)t0 * vsb, vsb}};
            for (const auto &pl : planes) {
                e = cudaMemcpy2DAsync(pl.dst, (size_t)page_tokens * pl.rb, pl.src, (size_t)cap * pl.rb,
                                      (size_t)len * pl.rb, kv, cudaMemcpyDefault, cp);
                if (e != cudaSuccess) return cuda_fail(e, "page copy");
            }
            if ((e = cudaEventRecord(copied[p], cp)) != cudaSuccess || (e = cudaStreamWaitEvent(cs, copied[p], 0)) != cudaSuccess)
                return cuda_fail(e, "page event");
            kvq_cache ks, vs;
            slot_views(k_host, v_host, page_tokens, base, rl, ks, vs);
            if ((st = decode_part(&ks, &vs, len, t0 + len, idx++)) != KVQ_OK) {
                cleanup();
                return st;
            }
            if ((e = cudaEventRecord(freed[slot], cs)) != cudaSuccess) return cuda_fail(e, "slot event");
        }
        cleanup();      // events are released once their work completes
    }
    if (parts == 1) {
        cudaError_t e = cudaMemcpyAsync(out, part_o, rows * D * sizeof(float), cudaMemcpyDeviceToDevice, cs);
        if (e == cudaSuccess && out_lse)
            e = cudaMemcpyAsync(out_lse, part_lse, rows * sizeof(float), cudaMemcpyDeviceToDevice, cs);
        if (e != cudaSuccess) return kvq::fail_msg(KVQ_ECUDA, "tiered: result copy: %s", cudaGetErrorString(e));
        return KVQ_OK;
    }
    const cudaError_t e = kvq::launch_merge(part_o, part_lse, parts, (int)rows, D, out, out_lse, cs);
    if (e != cudaSuccess) return kvq::fail_msg(KVQ_ECUDA, "tiered: merge launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

}  // extern "C"
