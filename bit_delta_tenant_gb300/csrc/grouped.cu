// grouped.cu -- multi-tenant fused linear: a batch whose tokens each carry
// their own variant id, served over one shared W_base.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": fourteen fine-tuned
// variants share one HBM-resident W_base; a request names its variant, and
// the variant's (alpha, sign) delta is applied on the fly by the fused
// kernel.  Here the routing is per token inside one batch.
//
// Steps (all on the device, ordered on the caller's stream):
//   1. sort: a stable counting sort of the tokens by variant id (one block;
//      each warp owns a contiguous token range, ranks equal ids within a
//      32-token slice with __match_any_sync, and per-warp counts give every
//      token its place), writing segment starts, the permutation and the
//      tile tables of the two compute kernels.  Ids outside [0, V) set
//      BD_ERR_BAD_VARIANT_ID in the status word and their tokens are skipped.
//   2. gather: the activations in variant order (a plain row copy).
//   3. compute: small batches (m <= 64) run a streaming kernel that reads
//      W_base and every variant's bits once (grouped_decode.cu on mma.sync;
//      a tcgen05 variant and a base-on-tensor-cores split are selectable);
//      larger batches the tensor-core kernel over per-variant token tiles
//      (prefill.cu).  Outputs go straight back to the original token rows.
#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kTileRows = 256;  // token rows per tensor-core tile
constexpr int kPad = 8;         // tokens per sign tile of the streaming kernel
constexpr int kMaxSignTilesRead = 24;  // the streaming kernel reads this many table entries

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct WsLayout {
    size_t seg, perm, tiles, n_tiles, s_tiles, n_s_tiles, xs, ybase, total;
    int64_t max_slots, max_s_tiles;
};

WsLayout layout(int64_t m, int32_t nv, int64_t n_out, int64_t n_in) {
    WsLayout L;
    L.max_slots = (m + kTileRows - 1) / kTileRows + nv;
    L.max_s_tiles = (m + kPad - 1) / kPad + nv + kMaxSignTilesRead;  // room for the streaming kernel's fixed read
    size_t off = 0;
    L.seg = off;
    off = align256(off + sizeof(int32_t) * (nv + 1));
    L.perm = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(m > 0 ? m : 1));
    L.tiles = off;
    off = align256(off + sizeof(int32_t) * 3 * static_cast<size_t>(L.max_slots));
    L.n_tiles = off;
    off = align256(off + sizeof(int32_t));
    L.s_tiles = off;
    off = align256(off + sizeof(int32_t) * 3 * static_cast<size_t>(L.max_s_tiles));
    L.n_s_tiles = off;
    off = align256(off + sizeof(int32_t));
    L.xs = off;
    off = align256(off + 2 * static_cast<size_t>(m > 0 ? m : 1) * static_cast<size_t>(n_in));
    // fp32 base product of the split small-batch path (only for m <= 64)
    L.ybase = off;
    if (m <= 64) off = align256(off + 4 * static_cast<size_t>(m > 0 ? m : 1) * static_cast<size_t>(n_out));
    L.total = off;
    return L;
}

struct SortArgs {
    const int32_t *ids;
    int64_t m;
    int32_t nv;
    int32_t *seg, *perm, *tiles, *n_tiles, *s_tiles, *n_s_tiles;
    unsigned *status;
};

__global__ void __launch_bounds__(kSortThreads, 1) group_sort_kernel(SortArgs a) {
    __shared__ int32_t cnt[kSortWarps][kMaxVariantsDev];  // per-warp counts, then running offsets
    __shared__ int32_t seg_s[kMaxVariantsDev + 1];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int i = tid; i < kSortWarps * kMaxVariantsDev; i += kSortThreads) (&cnt[0][0])[i] = 0;
    __syncthreads();

    // Contiguous per-warp token ranges, a multiple of 32 long.
    const int64_t per_warp = ((a.m + kSortWarps - 1) / kSortWarps + 31) / 32 * 32;
    const int64_t lo = warp * per_warp;
    const int64_t hi = min(lo + per_warp, a.m);

    // Pass 1: counts per (warp, variant).
    bool bad = false;
    for (int64_t base = lo; base < hi; base += 32) {
        const int64_t t = base + lane;
        int id = -1;
        if (t < hi) {
            id = a.ids[t];
            if (id < 0 || id >= a.nv) {
                bad = true;
                id = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, id);
        if (id >= 0 && (peers & lt_mask) == 0) cnt[warp][id] += __popc(peers);
        __syncwarp();
    }
    if (bad) flag_status(a.status, kDevBadVariant);
    __syncthreads();

    // Segment starts, per-warp offsets, and the two tile tables: up to 256
    // tokens of one variant per tensor-core tile, up to 8 per streaming sign tile.
    if (tid == 0) {
        int32_t s = 0;
        for (int v = 0; v < a.nv; ++v) {
            int32_t tot = 0;
            for (int w = 0; w < kSortWarps; ++w) tot += cnt[w][v];
            seg_s[v] = s;
            s += tot;
        }
        seg_s[a.nv] = s;
        int32_t nt = 0, ns = 0;
        for (int v = 0; v < a.nv; ++v) {
            const int32_t len = seg_s[v + 1] - seg_s[v];
            for (int32_t j = 0; j < len; j += kTileRows) {
                a.tiles[3 * nt] = v;
                a.tiles[3 * nt + 1] = seg_s[v] + j;
                a.tiles[3 * nt + 2] = min(kTileRows, len - j);
                ++nt;
            }
            for (int32_t j = 0; j < len; j += kPad) {
                a.s_tiles[3 * ns] = v;
                a.s_tiles[3 * ns + 1] = seg_s[v] + j;
                a.s_tiles[3 * ns + 2] = min(kPad, len - j);
                ++ns;
            }
        }
        *a.n_tiles = nt;
        *a.n_s_tiles = ns;
    }
    __syncthreads();
    if (tid < a.nv) {
        int32_t off = seg_s[tid];
        for (int w = 0; w < kSortWarps; ++w) {
            const int32_t c = cnt[w][tid];
            cnt[w][tid] = off;
            off += c;
        }
    }
    for (int i = tid; i <= a.nv; i += kSortThreads) a.seg[i] = seg_s[i];
    __syncthreads();

    // Pass 2: the same walk; rank among equal ids in the slice keeps the sort stable.
    for (int64_t base = lo; base < hi; base += 32) {
        const int64_t t = base + lane;
        int id = -1;
        if (t < hi) {
            id = a.ids[t];
            if (id < 0 || id >= a.nv) id = -1;
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, id);
        if (id >= 0) {
            const int32_t pos = cnt[warp][id] + __popc(peers & lt_mask);
            if (in_bounds(pos >= 0 && pos < a.m, a.status)) a.perm[pos] = static_cast<int32_t>(t);
        }
        __syncwarp();
        if (id >= 0 && (peers & lt_mask) == 0) cnt[warp][id] += __popc(peers);
        __syncwarp();
    }
}

// xs[r] = x[map[r]] (a zero row where map[r] < 0), rows r < *n_rows.
__global__ void group_gather_kernel(const uint4 *x, int64_t vec_per_row, const int32_t *map, const int32_t *n_rows,
                                    int64_t max_rows, uint4 *xs, unsigned *status) {
    const int64_t rows = *n_rows;
    const int64_t total = max_rows * vec_per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / vec_per_row;
        if (r >= rows) continue;
        const int64_t c = i - r * vec_per_row;
        const int32_t src = map[r];
        if (!in_bounds(src < max_rows, status)) continue;  // map rows name tokens of x ([max_rows] rows)
        xs[i] = src >= 0 ? x[static_cast<int64_t>(src) * vec_per_row + c] : make_uint4(0, 0, 0, 0);
    }
}

}  // namespace

size_t grouped_workspace_size(int64_t m, int32_t n_variants, int64_t n_out, int64_t n_in) {
    return layout(m, n_variants, n_out, n_in).total;
}

cudaError_t launch_grouped(const void *x, const int32_t *ids, int64_t m, const void *w_base,
                           const GroupedVariants &vars, int64_t n_out, int64_t n_in, void *y, void *ws,
                           size_t ws_bytes, const DevCtx &ctx, cudaStream_t stream) {
    const WsLayout L = layout(m, vars.count, n_out, n_in);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    SortArgs s;
    s.ids = ids;
    s.m = m;
    s.nv = vars.count;
    s.seg = reinterpret_cast<int32_t *>(base + L.seg);
    s.perm = reinterpret_cast<int32_t *>(base + L.perm);
    s.tiles = reinterpret_cast<int32_t *>(base + L.tiles);
    s.n_tiles = reinterpret_cast<int32_t *>(base + L.n_tiles);
    s.s_tiles = reinterpret_cast<int32_t *>(base + L.s_tiles);
    s.n_s_tiles = reinterpret_cast<int32_t *>(base + L.n_s_tiles);
    s.status = ctx.status;
    group_sort_kernel<<<1, kSortThreads, 0, stream>>>(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    uint4 *xs = reinterpret_cast<uint4 *>(base + L.xs);
    const int64_t vec = n_in / 8;
    // compact variant-sorted rows for the tensor-core path (row count = seg[V])
    const int64_t work = m * vec;
    int64_t nblk = (work + 255) / 256;
    if (nblk > 8 * static_cast<int64_t>(ctx.num_sms)) nblk = 8 * static_cast<int64_t>(ctx.num_sms);
    const int blocks = static_cast<int>(nblk);
    group_gather_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(static_cast<const uint4 *>(x), vec, s.perm,
                                                                     s.seg + vars.count, m, xs, ctx.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // Small batches (default): the mma.sync streaming kernel computing the base
    // and every variant's sign products in one pass.  The BD_OPT_GROUPED_PATH
    // option 1/2/3/4 forces the tcgen05 streaming kernel / that default / per-variant
    // tensor-core tiles / a split in which the tensor-core kernel computes the
    // base product (fp32, W_base as stored) and the streaming kernel only the
    // sign products (tests and comparisons; unsupported shapes fall through).
    // Measured on GB300 (14 variants, 64 tokens): the split matches the single
    // kernel (195 us for 8192 x 8192), the sign products dominate; the tcgen05
    // streaming kernel issues ~4 N=16 MMAs per variant and K block, each
    // behind an mbarrier round trip, and ends up latency-bound.
    const int path = static_cast<int>(option_value(BD_OPT_GROUPED_PATH));
    if (path == 1 && grouped_decode_tc_supported(m, vars.count, n_in, xs, w_base, vars))
        return launch_grouped_decode_tc(xs, m, w_base, vars, n_out, n_in, y, s.seg, s.perm, ctx, stream);
    if (path == 4 && m <= 64 && grouped_decode_supported(m, vars.count, n_in, w_base, vars)) {
        float *ybase = reinterpret_cast<float *>(base + L.ybase);
        e = launch_base_product(xs, m, w_base, n_out, n_in, ybase, ctx, stream);
        if (e != cudaSuccess) return e;
        return launch_grouped_decode(xs, m, w_base, vars, n_out, n_in, y, s.s_tiles, s.n_s_tiles, s.perm,
                                     s.seg + vars.count, ybase, ctx, stream);
    }
    if ((path == 0 || path == 1 || path == 2 || path == 4) && grouped_decode_supported(m, vars.count, n_in, w_base, vars))
        return launch_grouped_decode(xs, m, w_base, vars, n_out, n_in, y, s.s_tiles, s.n_s_tiles, s.perm,
                                     s.seg + vars.count, nullptr, ctx, stream);
    GroupTable tab;
    tab.tiles = s.tiles;
    tab.n_tiles = s.n_tiles;
    tab.perm = s.perm;
    tab.max_slots = static_cast<int32_t>(L.max_slots);
    return launch_prefill_grouped(xs, m, w_base, vars, n_out, n_in, y, tab, ctx, stream);
}

}  // namespace bd
