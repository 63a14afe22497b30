// delta_cache.cu -- the delta cache in front of the fused kernels: every
// variant's compressed delta (packed bits + fp32 alpha) lives in host memory
// and is brought into HBM on first use; resident deltas are evicted by a
// request-rate-weighted least-recently-used rule, frequently used ones can be
// pinned, and concurrent requests for a delta that is being loaded share the
// one load.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Détails d'infrastructure": cold start of a variant
// (load of its delta from the host, ~200 ms on the page), LRU eviction weighted
// by request rate, pinning of popular variants, single-flight routing of
// concurrent requests.  Section "Architecture de service": the base stays
// resident and each request names its variant.
//
// Reading of the eviction rule (the page names it only): each variant keeps a
// request rate that decays with half-life H seconds and gains 1 per request;
// the victim is the unpinned, unused resident variant with the lowest decayed
// rate, the least recently requested one on ties.
//
// Host-side runtime, no kernels.  The caller provides the state buffer (host)
// and the device arena; the cache carves the arena first-fit (256-byte
// aligned blocks, freed blocks coalesce).  Ordering with the GPU: a load is
// an async host-to-device copy on the requesting stream followed by an event;
// every later acquirer's stream waits on that event (the single flight).  A
// release records an event on the releasing stream; before a victim's block is
// reused the host waits for the events of its outstanding uses, so a copy can
// never overwrite a delta that queued work still reads.  In host-arena mode
// (for policy studies and CPU tests) the arena is host memory, loads are
// memcpy and no CUDA call is made.
#include <cmath>
#include <cstring>
#include <mutex>
#include <chrono>
#include <new>

#include "bd_internal.h"
#include "bitdelta.h"

#define BD_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kAlign = 256;
constexpr int kUseEvents = 8;  // outstanding releases tracked per variant

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

struct Variant {
    bool registered, resident, pinned, loading;
    const void *host_bits;
    const float *host_alpha;
    size_t bits_bytes, alpha_bytes, block_bytes;
    size_t offset;         // in the arena, when resident
    int32_t refs;          // acquires not yet released
    double rate, last_t;   // decayed request rate and the time it refers to
    cudaEvent_t load_ev;   // CUDA mode: end of the load copy
    cudaEvent_t use_ev[kUseEvents];
    bool use_pending[kUseEvents];
    int use_next;
};

struct Segment {  // free space of the arena
    size_t off, size;
};

struct Cache {
    std::mutex mu;
    int32_t max_variants;
    bool host_arena;
    uint8_t *arena;
    size_t arena_bytes;
    double half_life;
    std::chrono::steady_clock::time_point t0;
    bd_cache_stats stats;
    int32_t n_free;
    Segment *free_segs;  // sorted by offset, max_variants + 1 entries
    Variant *vars;       // max_variants entries
};

size_t state_bytes(int32_t max_variants) {
    return align_up(sizeof(Cache)) + align_up(sizeof(Segment) * (max_variants + 1)) +
           align_up(sizeof(Variant) * max_variants) + kAlign;
}

double now_of(Cache *c, double now_s) {
    if (now_s >= 0.0) return now_s;
    return std::chrono::duration<double>(std::chrono::steady_clock::now() - c->t0).count();
}

double decayed(const Cache *c, const Variant &v, double now) {
    const double dt = now > v.last_t ? now - v.last_t : 0.0;
    return v.rate * std::exp2(-dt / c->half_life);
}

// First fit; returns false when no free segment is large enough.
bool arena_alloc(Cache *c, size_t bytes, size_t *off) {
    for (int32_t i = 0; i < c->n_free; ++i) {
        Segment &s = c->free_segs[i];
        if (s.size < bytes) continue;
        *off = s.off;
        s.off += bytes;
        s.size -= bytes;
        if (s.size == 0) {
            for (int32_t j = i + 1; j < c->n_free; ++j) c->free_segs[j - 1] = c->free_segs[j];
            --c->n_free;
        }
        return true;
    }
    return false;
}

void arena_free(Cache *c, size_t off, size_t bytes) {
    int32_t i = 0;
    while (i < c->n_free && c->free_segs[i].off < off) ++i;
    for (int32_t j = c->n_free; j > i; --j) c->free_segs[j] = c->free_segs[j - 1];
    c->free_segs[i] = Segment{off, bytes};
    ++c->n_free;
    // merge with the neighbours
    if (i + 1 < c->n_free && c->free_segs[i].off + c->free_segs[i].size == c->free_segs[i + 1].off) {
        c->free_segs[i].size += c->free_segs[i + 1].size;
        for (int32_t j = i + 2; j < c->n_free; ++j) c->free_segs[j - 1] = c->free_segs[j];
        --c->n_free;
    }
    if (i > 0 && c->free_segs[i - 1].off + c->free_segs[i - 1].size == c->free_segs[i].off) {
        c->free_segs[i - 1].size += c->free_segs[i].size;
        for (int32_t j = i + 1; j < c->n_free; ++j) c->free_segs[j - 1] = c->free_segs[j];
        --c->n_free;
    }
}

// Wait (host) until queued work that used v's block is done.
int32_t drain_uses(Cache *c, Variant &v) {
    if (c->host_arena) return BD_OK;
    for (int i = 0; i < kUseEvents; ++i)
        if (v.use_pending[i]) {
            if (cudaEventSynchronize(v.use_ev[i]) != cudaSuccess) return BD_ERR_CUDA;
            v.use_pending[i] = false;
        }
    if (v.loading) {
        if (cudaEventSynchronize(v.load_ev) != cudaSuccess) return BD_ERR_CUDA;
        v.loading = false;
    }
    return BD_OK;
}

// The evictable resident variant with the lowest decayed rate (oldest on ties), or -1.
int32_t pick_victim(Cache *c, double now) {
    int32_t best = -1;
    double best_rate = 0.0, best_t = 0.0;
    for (int32_t i = 0; i < c->max_variants; ++i) {
        const Variant &v = c->vars[i];
        if (!v.resident || v.pinned || v.refs > 0) continue;
        const double r = decayed(c, v, now);
        if (best < 0 || r < best_rate || (r == best_rate && v.last_t < best_t)) {
            best = i;
            best_rate = r;
            best_t = v.last_t;
        }
    }
    return best;
}

Cache *as_cache(bd_cache *p) { return reinterpret_cast<Cache *>(p); }

}  // namespace

BD_API size_t bd_cache_state_size(int32_t max_variants) {
    if (max_variants < 1 || max_variants > BD_CACHE_MAX_VARIANTS) return 0;
    return state_bytes(max_variants);
}

BD_API int32_t bd_cache_create(void *state, size_t state_size, int32_t max_variants, void *arena, size_t arena_bytes,
                               double half_life_s, int32_t host_arena, bd_cache **out) {
    if (!state || !arena || !out || arena_bytes == 0 || !(half_life_s > 0.0)) return BD_ERR_INVALID_ARG;
    if (max_variants < 1 || max_variants > BD_CACHE_MAX_VARIANTS) return BD_ERR_INVALID_ARG;
    if (state_size < state_bytes(max_variants)) return BD_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(arena) % kAlign != 0) return BD_ERR_MISALIGNED;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(state) + kAlign - 1) & ~(kAlign - 1));
    Cache *c = new (base) Cache();
    c->max_variants = max_variants;
    c->host_arena = host_arena != 0;
    c->arena = static_cast<uint8_t *>(arena);
    c->arena_bytes = arena_bytes & ~(kAlign - 1);
    c->half_life = half_life_s;
    c->t0 = std::chrono::steady_clock::now();
    std::memset(&c->stats, 0, sizeof c->stats);
    c->free_segs = reinterpret_cast<Segment *>(base + align_up(sizeof(Cache)));
    c->vars = reinterpret_cast<Variant *>(base + align_up(sizeof(Cache)) +
                                          align_up(sizeof(Segment) * (max_variants + 1)));
    c->n_free = 1;
    c->free_segs[0] = Segment{0, c->arena_bytes};
    for (int32_t i = 0; i < max_variants; ++i) {
        Variant *v = new (&c->vars[i]) Variant();
        std::memset(static_cast<void *>(v), 0, sizeof(Variant));
    }
    *out = reinterpret_cast<bd_cache *>(c);
    return BD_OK;
}

BD_API int32_t bd_cache_destroy(bd_cache *cp) {
    if (!cp) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    int32_t rc = BD_OK;
    {
        std::lock_guard<std::mutex> lock(c->mu);
        for (int32_t i = 0; i < c->max_variants; ++i) {
            Variant &v = c->vars[i];
            if (!v.registered || c->host_arena) continue;
            if (drain_uses(c, v) != BD_OK) rc = BD_ERR_CUDA;
            cudaEventDestroy(v.load_ev);
            for (int e = 0; e < kUseEvents; ++e) cudaEventDestroy(v.use_ev[e]);
        }
    }
    c->~Cache();
    return rc;
}

BD_API int32_t bd_cache_register(bd_cache *cp, int32_t variant, const void *host_bits, size_t bits_bytes,
                                 const float *host_alpha, size_t alpha_bytes) {
    if (!cp || !host_bits || !host_alpha || bits_bytes == 0 || alpha_bytes == 0) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    if (variant < 0 || variant >= c->max_variants) return BD_ERR_BAD_VARIANT_ID;
    std::lock_guard<std::mutex> lock(c->mu);
    Variant &v = c->vars[variant];
    if (v.registered) return BD_ERR_INVALID_ARG;
    const size_t block = align_up(bits_bytes) + align_up(alpha_bytes);
    if (block > c->arena_bytes) return BD_ERR_NO_SPACE;
    if (!c->host_arena) {
        if (cudaEventCreateWithFlags(&v.load_ev, cudaEventDisableTiming) != cudaSuccess) return BD_ERR_CUDA;
        for (int e = 0; e < kUseEvents; ++e)
            if (cudaEventCreateWithFlags(&v.use_ev[e], cudaEventDisableTiming) != cudaSuccess) return BD_ERR_CUDA;
    }
    v.registered = true;
    v.host_bits = host_bits;
    v.host_alpha = host_alpha;
    v.bits_bytes = bits_bytes;
    v.alpha_bytes = alpha_bytes;
    v.block_bytes = block;
    return BD_OK;
}

BD_API int32_t bd_cache_set_pinned(bd_cache *cp, int32_t variant, int32_t pinned) {
    if (!cp) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    if (variant < 0 || variant >= c->max_variants) return BD_ERR_BAD_VARIANT_ID;
    std::lock_guard<std::mutex> lock(c->mu);
    if (!c->vars[variant].registered) return BD_ERR_BAD_VARIANT_ID;
    c->vars[variant].pinned = pinned != 0;
    return BD_OK;
}

BD_API int32_t bd_cache_acquire(bd_cache *cp, int32_t variant, double now_s, void *stream, const uint8_t **bits,
                                const float **alpha) {
    if (!cp || !bits || !alpha) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    if (variant < 0 || variant >= c->max_variants) return BD_ERR_BAD_VARIANT_ID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(c->mu);
    Variant &v = c->vars[variant];
    if (!v.registered) return BD_ERR_BAD_VARIANT_ID;
    const double now = now_of(c, now_s);
    v.rate = decayed(c, v, now) + 1.0;
    if (now > v.last_t) v.last_t = now;
    ++c->stats.acquires;
    if (v.resident) {
        ++c->stats.hits;
        if (!c->host_arena && v.loading) {
            const cudaError_t q = cudaEventQuery(v.load_ev);
            if (q == cudaErrorNotReady) {
                ++c->stats.joined;  // single flight: wait on the copy already queued
                if (cudaStreamWaitEvent(s, v.load_ev, 0) != cudaSuccess) return BD_ERR_CUDA;
            } else if (q == cudaSuccess) {
                v.loading = false;
            } else {
                return BD_ERR_CUDA;
            }
        }
    } else {
        ++c->stats.misses;
        size_t off = 0;
        while (!arena_alloc(c, v.block_bytes, &off)) {
            const int32_t victim = pick_victim(c, now);
            if (victim < 0) return BD_ERR_NO_SPACE;
            Variant &w = c->vars[victim];
            const int32_t rc = drain_uses(c, w);
            if (rc != BD_OK) return rc;
            arena_free(c, w.offset, w.block_bytes);
            w.resident = false;
            ++c->stats.evictions;
        }
        uint8_t *dst = c->arena + off;
        if (c->host_arena) {
            std::memcpy(dst, v.host_bits, v.bits_bytes);
            std::memcpy(dst + align_up(v.bits_bytes), v.host_alpha, v.alpha_bytes);
        } else {
            if (cudaMemcpyAsync(dst, v.host_bits, v.bits_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                cudaMemcpyAsync(dst + align_up(v.bits_bytes), v.host_alpha, v.alpha_bytes, cudaMemcpyHostToDevice,
                                s) != cudaSuccess ||
                cudaEventRecord(v.load_ev, s) != cudaSuccess) {
                arena_free(c, off, v.block_bytes);
                return BD_ERR_CUDA;
            }
            v.loading = true;
        }
        v.offset = off;
        v.resident = true;
        ++c->stats.loads;
        c->stats.bytes_loaded += static_cast<int64_t>(v.bits_bytes + v.alpha_bytes);
    }
    ++v.refs;
    *bits = c->arena + v.offset;
    *alpha = reinterpret_cast<const float *>(c->arena + v.offset + align_up(v.bits_bytes));
    return BD_OK;
}

BD_API int32_t bd_cache_release(bd_cache *cp, int32_t variant, void *stream) {
    if (!cp) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    if (variant < 0 || variant >= c->max_variants) return BD_ERR_BAD_VARIANT_ID;
    std::lock_guard<std::mutex> lock(c->mu);
    Variant &v = c->vars[variant];
    if (!v.registered || v.refs <= 0) return BD_ERR_INVALID_ARG;
    if (!c->host_arena) {
        const int e = v.use_next;
        if (v.use_pending[e] && cudaEventSynchronize(v.use_ev[e]) != cudaSuccess) return BD_ERR_CUDA;
        if (cudaEventRecord(v.use_ev[e], static_cast<cudaStream_t>(stream)) != cudaSuccess) return BD_ERR_CUDA;
        v.use_pending[e] = true;
        v.use_next = (e + 1) % kUseEvents;
    }
    --v.refs;
    return BD_OK;
}

BD_API int32_t bd_cache_get_stats(bd_cache *cp, bd_cache_stats *out) {
    if (!cp || !out) return BD_ERR_INVALID_ARG;
    Cache *c = as_cache(cp);
    std::lock_guard<std::mutex> lock(c->mu);
    *out = c->stats;
    out->resident = 0;
    out->in_use = 0;
    out->resident_bytes = 0;
    for (int32_t i = 0; i < c->max_variants; ++i) {
        const Variant &v = c->vars[i];
        if (v.resident) {
            ++out->resident;
            out->resident_bytes += static_cast<int64_t>(v.block_bytes);
        }
        if (v.refs > 0) ++out->in_use;
    }
    return BD_OK;
}

BD_API int32_t bd_cache_is_resident(bd_cache *cp, int32_t variant) {
    if (!cp) return 0;
    Cache *c = as_cache(cp);
    if (variant < 0 || variant >= c->max_variants) return 0;
    std::lock_guard<std::mutex> lock(c->mu);
    return c->vars[variant].resident ? 1 : 0;
}
