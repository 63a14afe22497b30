/*
 * bitdelta.h -- C ABI of libbitdelta.so, the GB300 (sm_103a) BitDelta hot path.
 *
 * BitDelta stores a fine-tuned weight matrix as the shared base W_base plus a
 * 1-bit delta: W_ft ~= W_base + alpha * sign(W_ft - W_base).  Method source:
 * the blog page "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
 * (Hanzo blog); sections cited below:
 *   [math]  "Le fondement mathématique"  Delta = W_ft - W_base; the 1-bit
 *           approximation W_base + alpha*sign(Delta); alpha = mean|Delta|.
 *   [serve] "Architecture de service"    W_eff is rebuilt on the fly inside one
 *           fused kernel that reads W_base and the packed bits together and
 *           never writes W_eff to HBM; the conceptual fused_bitdelta_linear
 *           listing (x [batch, seq, d_in], W_base [d_out, d_in], packed signs,
 *           alpha [d_out] or scalar, result = linear(x, W_eff)).
 *   [infra] "Détails d'infrastructure"   signs packed 8 per byte
 *           (4096x4096 -> 4096x512); alpha stored as fp32, one per output row.
 *
 * Conventions shared by every entry point
 *   - Shapes use n_out = d_out (rows of W) and n_in = d_in (columns).  All
 *     matrices are dense row-major.  bf16 tensors are passed as void*.
 *   - x [batch, seq, d_in] is flattened by the caller to [m, n_in].
 *   - Packed bits [n_out, n_in/8] (uint8): bit i of byte c in row j is the
 *     sign of element k = 8c + i (least significant bit = lowest d_in);
 *     bit = 1 iff Delta >= 0 (zero deltas, either sign of zero, pack as 1)
 *     and unpacks to +1, bit 0 to -1.  The page prints neither the bit order
 *     nor sign(0); these are the readings this library fixes.
 *   - Every pointer is a DEVICE pointer unless marked "host".  The caller
 *     allocates and owns every buffer (inputs, outputs and workspace); the
 *     library allocates nothing, frees nothing and keeps no pointer after a
 *     call returns -- except the delta cache (bd_cache_*), which keeps its
 *     caller-provided state, arena and host deltas until bd_cache_destroy.
 *   - Every device pointer must be 16-byte aligned; n_in must be a multiple of
 *     8 (one packed byte per 8 inputs).  Any n_in that is a multiple of 8, any
 *     n_out >= 1 and any m >= 0 are handled on the GPU (ragged tails included).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL =
 *     the legacy default stream).  Argument errors are returned synchronously
 *     before anything is launched.  Device-side errors (a variant id out of
 *     range, a bounded wait that ran out) are recorded in a sticky per-process
 *     device status word and reported by bd_get_device_status().
 *   - Calls are safe from several host threads on different streams; two
 *     calls must not write the same output or workspace concurrently.
 */
#ifndef BITDELTA_H
#define BITDELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum bd_status {
    BD_OK = 0,
    BD_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad mode      */
    BD_ERR_UNSUPPORTED_SHAPE = 2, /* n_in % 8 != 0, sizes beyond the limits     */
    BD_ERR_MISALIGNED = 3,        /* a device pointer is not 16-byte aligned    */
    BD_ERR_WORKSPACE = 4,         /* workspace missing or smaller than required */
    BD_ERR_CUDA = 5,              /* a CUDA runtime call failed                 */
    BD_ERR_DEVICE_TIMEOUT = 6,    /* a bounded device-side wait ran out         */
    BD_ERR_BAD_VARIANT_ID = 7,    /* a variant id outside [0, n_variants)       */
    BD_ERR_NO_SPACE = 8,          /* delta cache: nothing evictable leaves room  */
    BD_ERR_DEVICE_BOUNDS = 9      /* bounds-checked build only: a device index
                                     failed its check and the access was skipped */
} bd_status;

/* How alpha is stored ([math]: one per matrix; [infra]: one per output row). */
typedef enum bd_alpha_mode {
    BD_ALPHA_SCALAR = 0,  /* alpha: 1 float,     alpha   = mean_{j,k} |Delta_jk| */
    BD_ALPHA_PER_ROW = 1  /* alpha: n_out floats, alpha_j = mean_k |Delta_jk|    */
} bd_alpha_mode;

/* Upper limits checked on entry. */
#define BD_MAX_VARIANTS 64          /* variants per bd_linear_grouped call */
#define BD_MAX_DIM ((int64_t)1 << 31) /* n_out, n_in and m are each below this */

/* ------------------------------------------------------------------------ *
 * Compression  ([math] Delta, sign, alpha; [infra] packing and fp32 alpha)
 *
 * Delta = fp32(W_ft) - fp32(W_base) element-wise (the subtraction is done in
 * fp32 from the bf16 inputs).  Writes the packed sign bits and alpha:
 *   scalar:  alpha[0] = sum_{j,k} |Delta_jk| / (n_out * n_in)
 *   per-row: alpha[j] = sum_k |Delta_jk| / n_in
 * The sums use pairwise fp32 partials over at most 32 elements, widened to
 * fp64 and reduced in a fixed order (relative error below 5e-7), so alpha is
 * bitwise reproducible for a given shape, and is rounded once to fp32.
 *
 *   w_base, w_ft  bf16 [n_out, n_in]   (read)
 *   bits_out      uint8 [n_out, n_in/8] (written)
 *   alpha_out     float [1] or [n_out]  (written)
 *   workspace     device scratch of at least
 *                 bd_compress_workspace_size(n_out, n_in, alpha_mode) bytes;
 *                 its contents on entry are ignored.
 * Errors: BD_ERR_INVALID_ARG, BD_ERR_UNSUPPORTED_SHAPE, BD_ERR_MISALIGNED,
 *         BD_ERR_WORKSPACE, BD_ERR_CUDA (launch failure).
 * ------------------------------------------------------------------------ */
size_t bd_compress_workspace_size(int64_t n_out, int64_t n_in, int32_t alpha_mode);

int32_t bd_compress(const void *w_base, const void *w_ft, int64_t n_out,
                    int64_t n_in, int32_t alpha_mode, uint8_t *bits_out,
                    float *alpha_out, void *workspace, size_t workspace_bytes,
                    void *stream);

/* ------------------------------------------------------------------------ *
 * Batched compression  ([math], [infra]: every matrix of a fine-tune is
 * compressed against its base)
 *
 * Matrix i gets exactly the bits and alpha bd_compress gives it (same
 * per-segment arithmetic and summation order), with up to
 * BD_COMPRESS_BATCH_PER_LAUNCH matrices per launch of each pass instead of
 * two launches per matrix.
 *
 *   descs      host array [n] of bd_compress_desc (read during the call only;
 *              `reserved` must be 0); each as in bd_compress
 *   n          0 <= n <= BD_COMPRESS_BATCH_MAX
 *   workspace  device scratch of at least
 *              bd_compress_batch_workspace_size(descs, n) bytes (each
 *              matrix's bd_compress_workspace_size, rounded up to 256 bytes),
 *              256-byte aligned; its contents on entry are ignored.
 * Ordered on `stream`; buffers caller-owned.  No output may overlap an input
 * or another matrix's output.
 * Errors: the first failing matrix's bd_compress code (nothing launched),
 *         BD_ERR_INVALID_ARG (n out of range, reserved != 0),
 *         BD_ERR_WORKSPACE, BD_ERR_CUDA.
 * ------------------------------------------------------------------------ */
#define BD_COMPRESS_BATCH_MAX 4096
#define BD_COMPRESS_BATCH_PER_LAUNCH 8
typedef struct bd_compress_desc {
    const void *w_base;   /* bf16 [n_out, n_in] */
    const void *w_ft;     /* bf16 [n_out, n_in] */
    uint8_t *bits_out;    /* uint8 [n_out, n_in/8] (written) */
    float *alpha_out;     /* float [1] or [n_out] (written) */
    int64_t n_out;
    int64_t n_in;
    int32_t alpha_mode;
    int32_t reserved;     /* 0 */
} bd_compress_desc;

size_t bd_compress_batch_workspace_size(const bd_compress_desc *descs, int32_t n);
int32_t bd_compress_batch(const bd_compress_desc *descs, int32_t n, void *workspace,
                          size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Compression without a workspace.  The page has no counterpart to this
 * entry point; it exists for callers that cannot hand the library any device
 * memory besides the inputs and outputs -- for example code running under a
 * framework that owns all device memory through a pre-planned arena, or a
 * latency-critical path that must not call cudaMalloc (which can
 * synchronise the device).
 *
 * Same arguments, results and errors as bd_compress, minus the workspace:
 * the partial sums live in a fixed scratch array built into the library,
 * BD_NOALLOC_MAX_PARTIALS doubles (1 MiB) per GPU that loads the library,
 * held until the process exits.  With rows = 1 and chunks = n_out*n_in/8
 * for a scalar alpha, or rows = n_out and chunks = n_in/8 per row, and
 * segs = ceil(chunks / 1024), a shape fits when segs == 1 (each row is one
 * segment and needs no partial sums) or
 *   rows * segs <= BD_NOALLOC_MAX_PARTIALS
 * (a scalar alpha over up to 2^30 elements); larger shapes return
 * BD_ERR_WORKSPACE before launching anything (use bd_compress).
 * The call allocates and frees nothing.  Its first call on a device looks
 * up the scratch array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All
 * calls in the process share the one array, and every slot a call reads is
 * written earlier by the same call, so stale contents never matter -- but
 * calls whose kernels overlap on the GPU (different streams without
 * ordering) race on it: order them on one stream or with events.
 * ------------------------------------------------------------------------ */
#define BD_NOALLOC_MAX_PARTIALS 131072

int32_t bd_compress_noalloc(const void *w_base, const void *w_ft,
                            int64_t n_out, int64_t n_in, int32_t alpha_mode,
                            uint8_t *bits_out, float *alpha_out, void *stream);

/* ------------------------------------------------------------------------ *
 * Fused linear  ([serve] fused reconstruction + matmul, never materialising
 * W_eff in HBM; the conceptual fused_bitdelta_linear listing)
 *
 *   y[t, j] = sum_k x[t, k] * (W_base[j, k] + alpha_(j) * s_jk),
 *   s_jk = +1 if bit(j, k) else -1, alpha_(j) = alpha[0] or alpha[j].
 * Accumulation is fp32; y is rounded once to bf16.  m <= 16 streams W_base
 * and the bits from HBM once (mma.sync, distributive form); larger m runs a
 * tensor-core (tcgen05) kernel that rebuilds each W tile on chip as
 * bf16(W_base + alpha*s), splitting K over a cluster when its tiles are few.
 *
 *   x       bf16 [m, n_in]      (read; m may be 0, then nothing is launched)
 *   w_base  bf16 [n_out, n_in]  (read)
 *   bits    uint8 [n_out, n_in/8] (read)
 *   alpha   float [1] or [n_out] (read)
 *   y       bf16 [m, n_out]     (written)
 * Errors: BD_ERR_INVALID_ARG, BD_ERR_UNSUPPORTED_SHAPE, BD_ERR_MISALIGNED,
 *         BD_ERR_CUDA; BD_ERR_DEVICE_TIMEOUT later via bd_get_device_status.
 * ------------------------------------------------------------------------ */
int32_t bd_linear(const void *x, int64_t m, const void *w_base,
                  const uint8_t *bits, const float *alpha, int32_t alpha_mode,
                  int64_t n_out, int64_t n_in, void *y, void *stream);

/* ------------------------------------------------------------------------ *
 * Batched fused linear  ([serve] fused linear, several independent
 * projections per call -- e.g. q, k and v of a layer, or gate and up)
 *
 * Problem i computes exactly what bd_linear computes for descs[i].
 * Problems with 1 <= m <= 16, n_in a multiple of 128 and x, w_base, bits
 * and y 16-byte aligned are streamed together: up to
 * BD_LINEAR_BATCH_PER_LAUNCH of them per launch (grouped by m <= 8 and
 * m <= 16).  A launch whose 64-row blocks, times one K split shared by all
 * its problems, fit on the GPU at once runs them as one streaming launch
 * with K split over clusters; otherwise their work items -- one 128-column K
 * step of one 64-row block -- are split evenly over the resident CTAs.
 * Either way a row block's fp32 partials are summed in a fixed order, so
 * results are deterministic; they may differ from bd_linear's in the last
 * bits of fp32 rounding (another split of K).  Problems with m > 64 (the
 * tensor-core path) are launched together on the CTA-pair kernel, up to
 * BD_LINEAR_BATCH_PER_LAUNCH per launch, when their 256 x 256 tiles together
 * fill the GPU at least once -- a layer's q, k and v at prefill sizes, or gate
 * and up; such a problem computes what bd_linear computes on that kernel
 * (without a K split).  Every other problem, and a group that would hold a
 * single problem, runs as bd_linear.
 *
 *   descs      host array [n] of bd_linear_desc (read during the call only;
 *              `reserved` must be 0)
 *   n          0 <= n <= BD_LINEAR_BATCH_MAX
 *   workspace  device buffer of at least
 *              bd_linear_batch_workspace_size(descs, n) bytes (the size
 *              depends on the shapes and the current device), 256-byte
 *              aligned and ZERO-FILLED before its first use.  Each call whose
 *              kernels complete without a device error leaves it ready for the
 *              next call (its block counters back at zero; the partial sums it
 *              also holds need no clearing); after BD_ERR_DEVICE_TIMEOUT zero
 *              it again before reuse.  Calls that may run concurrently need
 *              distinct workspaces.  May be NULL when the size is 0.
 *              Caller-owned.
 * No y may overlap any input or another problem's y.  Ordered on `stream`.
 * A launch's CTAs may wait, within the wait limit (bd_set_wait_limit_ns), for
 * other CTAs of the same launch that share a row block; the launch is sized
 * to be resident on the GPU at once, so a launch kept from becoming resident
 * for longer than the limit (long-running kernels on other streams holding
 * the SMs) reports BD_ERR_DEVICE_TIMEOUT instead of completing.
 * Errors: the first failing problem's bd_linear code (nothing launched),
 *         BD_ERR_INVALID_ARG (n out of range, reserved != 0),
 *         BD_ERR_WORKSPACE (missing, misaligned or too small), BD_ERR_CUDA;
 *         BD_ERR_DEVICE_TIMEOUT later via bd_get_device_status.
 * ------------------------------------------------------------------------ */
#define BD_LINEAR_BATCH_MAX 256
#define BD_LINEAR_BATCH_PER_LAUNCH 8
typedef struct bd_linear_desc {
    const void *x;        /* bf16 [m, n_in] */
    const void *w_base;   /* bf16 [n_out, n_in] */
    const uint8_t *bits;  /* uint8 [n_out, n_in/8] */
    const float *alpha;   /* float [1] or [n_out] */
    void *y;              /* bf16 [m, n_out] (written) */
    int64_t m;
    int64_t n_out;
    int64_t n_in;
    int32_t alpha_mode;
    int32_t reserved;     /* 0 */
} bd_linear_desc;

size_t bd_linear_batch_workspace_size(const bd_linear_desc *descs, int32_t n);
int32_t bd_linear_batch(const bd_linear_desc *descs, int32_t n, void *workspace,
                        size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Reconstruct-only pass ([serve]: W_eff = W_base + alpha * unpacked signs,
 * then a plain linear; [latency] reads decode as a standard matmul)
 *
 *   w_eff[j, k] = bf16_rn( fp32(W_base[j, k]) + alpha_(j) * s_jk )
 * with the fp32 add rounded to nearest even and the result rounded once, to
 * nearest even, to bf16 -- the bf16 weight a standard GEMM would consume.
 * Provided to measure that reading against the fused path (which never
 * writes W_eff); the fused path is the one to use.
 *
 *   w_base  bf16 [n_out, n_in]   (read)
 *   bits    uint8 [n_out, n_in/8] (read)
 *   alpha   float [1] or [n_out] (read)
 *   w_eff   bf16 [n_out, n_in]   (written; may not alias the inputs)
 * All device pointers, 16-byte aligned; caller-owned.  Ordered on `stream`.
 * Errors: BD_ERR_INVALID_ARG (null pointer, bad mode, empty shape),
 *         BD_ERR_UNSUPPORTED_SHAPE (n_in % 8 != 0 or a dimension >=
 *         BD_MAX_DIM), BD_ERR_MISALIGNED, BD_ERR_CUDA (launch failure).
 * ------------------------------------------------------------------------ */
int32_t bd_reconstruct(const void *w_base, const uint8_t *bits, const float *alpha,
                       int32_t alpha_mode, int64_t n_out, int64_t n_in,
                       void *w_eff, void *stream);

/* ------------------------------------------------------------------------ *
 * Multi-tenant fused linear  ([serve]: many fine-tuned variants share one
 * resident W_base; each request uses its own variant's packed delta)
 *
 * Token t uses variant v = variant_ids[t]:
 *   y[t, j] = sum_k x[t, k] * (W_base[j, k] + alpha_v(j) * s^v_jk).
 * Tokens are counting-sorted by variant on the device (stable), each
 * variant's segment runs against the shared W_base, and y is written back in
 * the ORIGINAL token order.  Variants with no tokens cost nothing.
 *
 *   x              bf16 [m, n_in]            (read)
 *   variant_ids    int32 [m]                 (read, device)
 *   w_base         bf16 [n_out, n_in]        (read)
 *   bits_v         host array [n_variants] of device pointers, each
 *                  uint8 [n_out, n_in/8]
 *   alpha_v        host array [n_variants] of device pointers, each float
 *                  [1] or [n_out] per alpha_modes_v
 *   alpha_modes_v  host array [n_variants] of bd_alpha_mode values
 *   n_variants     1 .. BD_MAX_VARIANTS
 *   y              bf16 [m, n_out]           (written)
 *   workspace      device scratch of at least
 *                  bd_linear_grouped_workspace_size(m, n_variants, n_out, n_in)
 * An id outside [0, n_variants) sets BD_ERR_BAD_VARIANT_ID in the device
 * status word; the rows of y for such tokens are left unwritten.
 * ------------------------------------------------------------------------ */
size_t bd_linear_grouped_workspace_size(int64_t m, int32_t n_variants,
                                        int64_t n_out, int64_t n_in);

int32_t bd_linear_grouped(const void *x, const int32_t *variant_ids, int64_t m,
                          const void *w_base, const uint8_t *const *bits_v,
                          const float *const *alpha_v,
                          const int32_t *alpha_modes_v, int32_t n_variants,
                          int64_t n_out, int64_t n_in, void *y, void *workspace,
                          size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Delta cache  ([infra] "Détails d'infrastructure": each variant's delta is
 * loaded from host memory into HBM on its first request -- the cold start --
 * resident deltas are evicted least-recently-used weighted by request rate,
 * popular ones can be pinned, and concurrent requests for one variant share a
 * single load; [serve] the base stays resident, a request names its variant)
 *
 * The one stateful part of the library.  The caller provides a host buffer of
 * bd_cache_state_size(max_variants) bytes for the state and a 256-byte
 * aligned device arena that the cache carves first-fit into
 * 256-byte aligned blocks (freed blocks coalesce); the cache keeps pointers to
 * both, and to the registered host deltas, until bd_cache_destroy.  In CUDA
 * mode it creates 9 CUDA events per registered variant (destroyed by
 * bd_cache_destroy); register the host deltas from pinned memory for
 * asynchronous copies.
 *
 * Eviction rule (the page only names it): every variant keeps a request rate
 * that gains 1 per acquire and halves every `half_life_s` seconds; the victim
 * is the resident variant that is not pinned and not acquired, with the lowest
 * decayed rate, the least recently requested one on ties.  Variants are
 * evicted until the new block fits; BD_ERR_NO_SPACE if none is left.
 *
 * Ordering: a load is cudaMemcpyAsync of the bits, then of alpha, on the
 * acquiring stream, followed by an event; an acquirer that finds the load
 * still queued makes its stream wait on that event (single flight, counted in
 * `joined`).  bd_cache_release records an event on the given stream; before
 * an evicted variant's block is reused the host waits for its outstanding
 * releases (and its load), so no copy overwrites a delta that queued work
 * still reads.  host_arena != 0: the arena is host memory, loads are memcpy
 * and no CUDA call is made (policy studies, CPU tests).  All calls are
 * thread-safe (one mutex per cache).
 *
 * `now_s` (acquire) is the request time in seconds for the rate; pass a
 * negative value to use the library's monotonic clock.
 * Errors: BD_ERR_INVALID_ARG, BD_ERR_WORKSPACE (state buffer too small),
 *         BD_ERR_MISALIGNED (arena), BD_ERR_BAD_VARIANT_ID (id outside
 *         [0, max_variants) or not registered), BD_ERR_NO_SPACE, BD_ERR_CUDA.
 * ------------------------------------------------------------------------ */
#define BD_CACHE_MAX_VARIANTS 4096

typedef struct bd_cache bd_cache;

typedef struct bd_cache_stats {
    int64_t acquires, hits, misses, joined, loads, evictions, bytes_loaded;
    int64_t resident_bytes;
    int32_t resident, in_use;
} bd_cache_stats;

size_t  bd_cache_state_size(int32_t max_variants);
int32_t bd_cache_create(void *state_host, size_t state_bytes, int32_t max_variants,
                        void *arena, size_t arena_bytes, double half_life_s,
                        int32_t host_arena, bd_cache **out);
int32_t bd_cache_destroy(bd_cache *cache);
/* host_bits [bits_bytes] and host_alpha [alpha_bytes] stay owned by the caller
 * and must outlive the cache. */
int32_t bd_cache_register(bd_cache *cache, int32_t variant, const void *host_bits, size_t bits_bytes,
                          const float *host_alpha, size_t alpha_bytes);
int32_t bd_cache_set_pinned(bd_cache *cache, int32_t variant, int32_t pinned);
/* Device pointers of the variant's bits and alpha (256-byte aligned), valid
 * until the matching bd_cache_release; loads the delta on a miss. */
int32_t bd_cache_acquire(bd_cache *cache, int32_t variant, double now_s, void *stream,
                         const uint8_t **bits, const float **alpha);
int32_t bd_cache_release(bd_cache *cache, int32_t variant, void *stream);
int32_t bd_cache_get_stats(bd_cache *cache, bd_cache_stats *out);
/* 1 if the variant's delta is in the arena, else 0. */
int32_t bd_cache_is_resident(bd_cache *cache, int32_t variant);

/* ------------------------------------------------------------------------ *
 * Status and debugging
 * ------------------------------------------------------------------------ */

/* Static English text for a status code (never NULL). */
const char *bd_status_string(int32_t status);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device: BD_OK, BD_ERR_DEVICE_BOUNDS (bounds-checked build only),
 * BD_ERR_DEVICE_TIMEOUT or BD_ERR_BAD_VARIANT_ID (in that order of precedence).
 * BD_ERR_CUDA if the sync itself fails. */
int32_t bd_get_device_status(void *stream);

/* Debug knob: wall-clock limit, in nanoseconds, of every bounded device-side
 * wait (mbarrier and pipeline waits) in kernels launched afterwards by this
 * process.  Default 2e9 (2 s).  0 makes any wait that is not already
 * satisfied give up at once; the kernel then records BD_ERR_DEVICE_TIMEOUT,
 * drains its own copies in flight and returns.  Returns the previous value. */
int64_t bd_set_wait_limit_ns(int64_t limit_ns);

/* Debug knob: which fused-linear kernel later bd_linear calls use.
 * 0 = automatic (the HBM-streaming kernel for m <= 16 when it can run, the
 * tensor-core kernel otherwise); 1 = always the streaming kernel (m <= 64;
 * BD_ERR_UNSUPPORTED_SHAPE where it cannot run);
 * 2 = always the tensor-core kernel; 3 = always the register-fed streaming
 * kernel (the fallback of 1 for n_in not a multiple of 128).  Other values
 * are ignored.  Returns the previous value. */
int32_t bd_set_linear_path(int32_t path);

/* Serving knob: when `enable` is non-zero, later bd_linear calls on the
 * streaming path may start reading w_base and bits while the kernel launched
 * just before them on the same stream is still finishing (programmatic
 * dependent launch); x is read, and y written, only after that kernel has
 * completed.  This overlaps the weight stream of back-to-back linears, as in
 * a decode step over static weights.  Enable it only when no kernel that
 * directly precedes a bd_linear on its stream writes that call's w_base or
 * bits (for instance, not right after the bd_compress that produces the
 * bits).  Default 0.  Returns the previous setting. */
int32_t bd_set_weight_prefetch(int32_t enable);

/* Test knob: forces one of the library's kernel choices for calls made
 * afterwards by this process (every choice computes the same result within
 * the documented tolerance, and the compression forms the same bits and
 * alpha bit for bit).  `option` is one of the BD_OPT_* values below, `value`
 * one of the values listed beside it; 0 always restores the automatic
 * choice.  Returns the previous value, or -1 (nothing changed) for an
 * unknown option or a value out of range.  Not synchronised with calls in
 * flight on other host threads.
 *   BD_OPT_COMPRESS_FORM  0 one block per segment; 1 the persistent form
 *                         with a shared-memory copy ring
 *   BD_OPT_GROUPED_PATH   0 automatic; 1 the tcgen05 streaming kernel;
 *                         2 the mma.sync streaming kernel; 3 per-variant
 *                         tensor-core tiles; 4 base product on the tensor
 *                         cores, sign products on the streaming kernel
 *                         (paths that cannot run a shape fall through to
 *                         the automatic choice)
 *   BD_OPT_BATCH_KERNEL   bd_linear_batch launches: 0 automatic; 1 the
 *                         cluster-split kernel; 2 the evenly split kernel
 *   BD_OPT_BATCH_SINGLE   1 keeps a bd_linear_batch group of one problem on
 *                         the batched kernel instead of running it as
 *                         bd_linear
 *   BD_OPT_BATCH_GRID     CTAs of an evenly split batched launch (1 ..
 *                         2^31-1, capped at the CTAs that fit at once)
 *   BD_OPT_PREFILL_KERNEL tensor-core linear (m > 64): 0 automatic; 1 one
 *                         CTA per 128 x 256 tile (K split over a cluster when
 *                         tiles are few); 2 CTA pairs on 256 x 256 tiles
 *   BD_OPT_TEST_STALL     1 makes the first pipeline wait of the kernels
 *                         that support it -- the persistent compression
 *                         form and the multi-tenant streaming kernels --
 *                         wait on a barrier that nothing completes, so that
 *                         the wait runs out after the wait limit and the
 *                         kernel takes its give-up path (tests of failure
 *                         detection; results are then undefined and
 *                         bd_get_device_status reports
 *                         BD_ERR_DEVICE_TIMEOUT)
 *   BD_OPT_PAIR_RING      shape of the CTA-pair tensor-core kernel: 0
 *                         automatic (by K); 1 a 5-deep K-block ring with
 *                         the whole output tile staged; 2 a 6-deep ring
 *                         with the tile staged in two halves */
#define BD_OPT_COMPRESS_FORM 1
#define BD_OPT_GROUPED_PATH 2
#define BD_OPT_BATCH_KERNEL 3
#define BD_OPT_BATCH_SINGLE 4
#define BD_OPT_BATCH_GRID 5
#define BD_OPT_TEST_STALL 6
#define BD_OPT_PREFILL_KERNEL 7
#define BD_OPT_PAIR_RING 8
int64_t bd_set_option(int32_t option, int64_t value);

/* Build flags of the loaded library: bit 0 set in the bounds-checked build
 * (compiled with BD_DEBUG: every kernel checks the indices of its global
 * accesses against the extents it was given, skips an access that fails and
 * records BD_ERR_DEVICE_BOUNDS in the device status word; a stand-in for a
 * memory checker, slower than the release build and not for measurement). */
int32_t bd_build_flags(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t bd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_H */
