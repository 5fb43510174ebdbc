// Binned ("pull") backward of the deformable-aggregation operator.
//
// The gradients are those of the page "Inside Sparse4D's CUDA core", §4.1:
//   top_grad = grad_out * w; grad_feat[corner i] += w_i * top_grad;
//   grad_loc += (W*(lh*(v4-v3) + hh*(v2-v1)), H*(lw*(v4-v2) + hw*(v3-v1))) * top_grad;
//   grad_weight = grad_out . (w1*v1 + ... + w4*v4).
// The page scatters grad_feat with one atomicAdd per thread. On GB300,
// reductions into L2 move about a third of the bytes per second that loads
// do. So this path never scatters grad_feat. Instead it sorts the corner
// contributions by feature row, and every row is computed once by the lanes
// that own it:
//
//   1. count   one thread per location (b, a, p, k), camera-major, counts the
//              in-map corners of its S samples per feature row (row_off):
//              in shared memory for the maps that fit, then one global
//              atomic per touched row; per corner for larger maps;
//   2. scan    exclusive prefix sum of the counts (three small kernels);
//   3. fill    the same threads claim their slots (one global range per
//              touched row per CTA for the small maps, one global atomic per
//              corner for the large ones) and store the record
//              {sample*4 + corner, corner weight} (one 8-byte store);
//   4. pull    (da_pull.cu) C/8 lanes own one feature row (8 channels each,
//              all groups; a whole warp when C = 256). Per record they read
//              the anchor's grad_out row, accumulate (w * w_i) * grad_out
//              into the row's grad_feat, and form d = feat_row . grad_out
//              per group (a shuffle sum over the D/8 lanes of a group). The
//              grad_feat row is stored once (no zero-fill); the G values of
//              d go to dpix at the record's key, so the four corners of a
//              sample land side by side;
//   5. epilogue one lane per (location, scale) (or one warp per location):
//              it reads the four corners' d of its samples as one
//              contiguous run, and forms grad_weight = sum w_i d_i and the
//              two grad_loc sums, reduced by shuffles. Every output has one
//              owner, so there are no atomics.
#include <algorithm>
#include <climits>

#include "da_internal.cuh"

namespace da {

namespace {
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

BinLayout bin_layout(int64_t B, int64_t rows, int64_t A, int64_t P, int64_t K, int64_t S, int64_t G)
{
    BinLayout L{};
    L.rows_total = B * rows;
    L.nsid = B * A * P * K * S;
    L.ncap = 4 * L.nsid;
    L.ntiles = (L.rows_total + kScanTile - 1) / kScanTile;
    size_t o = 0;
    L.off_row_off = o;
    // Row offsets, the scan's end value, then the sort's three list counters:
    // one zero-fill clears them all.
    o = align256(o + static_cast<size_t>(L.ntiles * kScanTile + kRowOffTail) * 4);
    L.off_tile_sum = o;
    o = align256(o + static_cast<size_t>(L.ntiles + 4) * 4);
    L.off_rec = o;
    o = align256(o + static_cast<size_t>(L.ncap) * 8);
    L.off_dpix = o;
    o = align256(o + static_cast<size_t>(L.ncap) * static_cast<size_t>(G) * 4);
    L.off_left = o;
    o = align256(o + static_cast<size_t>(L.rows_total) * 4);
    // A row holds more than 8 (128, 2048) records in at most ncap/9
    // (ncap/129, ncap/2049) rows.
    L.cap_m = L.ncap / 9 + 1;
    L.cap_s = L.ncap / 129 + 1;
    L.cap_g = L.ncap / 2049 + 1;
    L.off_lists = o;
    o = align256(o + static_cast<size_t>(L.cap_m + L.cap_s + L.cap_g) * 4);
    L.bytes = o;
    return L;
}

namespace {

// ---------------------------------------------------------------- 1. count

// Binning threads run camera-major: CTA (b, k, chunk) takes 256 consecutive
// (a, p) pairs of camera k of batch item b, so all its corners fall in the
// maps of that one camera. The maps of camera k that fit kBinSmemRows
// entries are counted in shared memory first, and each touched row then gets
// one global atomic per CTA. That removes the pile-up of atomics on the rows
// of the coarse maps. Larger maps are counted with a global atomic per
// corner.
constexpr int kBinThreads = 256;
constexpr int kBinSmemRows = 8192;

struct BinCta {
    int b, k, q;         // batch item, camera, (a*P + p) of this thread
    bool valid;          // q < A*P
    int64_t pk;          // location id ((b*A + a)*P + p)*K + k
    int vg;              // a % gsplit: the group of this anchor's virtual rows
};

__device__ __forceinline__ BinCta bin_cta(const Problem &pb, int ctas_per_view)
{
    BinCta c;
    const int bk = static_cast<int>(blockIdx.x) / ctas_per_view;
    const int chunk = static_cast<int>(blockIdx.x) - bk * ctas_per_view;
    c.b = static_cast<int>(pb.div_K.div(bk));
    c.k = bk - c.b * pb.K;
    c.q = chunk * kBinThreads + threadIdx.x;
    c.valid = c.q < pb.A * pb.P;
    const int a = c.valid ? static_cast<int>(pb.div_P.div(c.q)) : 0;
    const int p = c.q - a * pb.P;
    c.pk = ((static_cast<int64_t>(c.b) * pb.A + a) * pb.P + p) * pb.K + c.k;
    c.vg = pb.gsplit > 1 ? a % pb.gsplit : 0;
    return c;
}

// Location (x, y) of location id pk: [.., 2] in the standard layout, the
// first two of 2 + S entries in the fused one.
template <bool FUSED>
__device__ __forceinline__ float2 bin_xy(const Problem &pb, int64_t pk)
{
    if constexpr (FUSED) {
        const float *e = pb.loc + pk * (2 + pb.S);
        return make_float2(e[0], e[1]);
    }
    return *reinterpret_cast<const float2 *>(pb.loc + pk * 2);
}

// Shared-memory offsets of the small maps of camera k (-1: counted globally).
__host__ __device__ inline void small_map_offsets(int S, const MapInfo *maps_s, int k, int *hoff, int &nsmall,
                                                  int gs)
{
    // Smallest maps first: their rows take the most corners each, so they
    // gain most from counting in shared memory.
    for (int s = 0; s < S; ++s) hoff[s] = -1;
    int off = 0;
    for (;;) {
        int best = -1, bn = 0;
        for (int s = 0; s < S; ++s) {
            const int n = maps_s[k * S + s].H * maps_s[k * S + s].W * gs;
            if (hoff[s] < 0 && off + n <= kBinSmemRows && (best < 0 || n < bn)) {
                best = s;
                bn = n;
            }
        }
        if (best < 0) break;
        hoff[best] = off;
        off += bn;
    }
    nsmall = off;
}

// Adds the shared counts of the small maps into row_off: one global atomic
// per touched row. Needs a __syncthreads() before it.
__device__ __forceinline__ void flush_small_counts(const Problem &pb, const MapInfo *maps_s, const int *hoff,
                                                   int k, const int *hist, int32_t *row_base, int gs)
{
    for (int s = 0; s < pb.S; ++s) {
        if (hoff[s] < 0) continue;
        const MapInfo m = maps_s[k * pb.S + s];
        const int n = m.H * m.W * gs;
        for (int r = threadIdx.x; r < n; r += kBinThreads) {
            const int v = hist[hoff[s] + r];
            if (v && DA_CHECK(pb.dbg_err, static_cast<int64_t>(m.start) * gs + r, pb.rows, kBoundsRowCount))
                atomicAdd(row_base + m.start * gs + r, v);
        }
    }
}

template <bool FUSED>
__global__ void __launch_bounds__(kBinThreads) bin_count_kernel(const Problem pb, const BinArgs w,
                                                                 int ctas_per_view, int hist_rows)
{
    pdl_wait();
    pdl_trigger();
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    extern __shared__ int hist[];  // hist_rows entries
    __shared__ int hoff[DA_MAX_MAPS];
    __shared__ int nsmall_s;
    stage_maps(pb, maps_s);
    const BinCta c = bin_cta(pb, ctas_per_view);
    __syncthreads();
    // Virtual rows per pixel row: gsplit in the fused rewrite, else 1.
    const int gs = FUSED ? pb.gsplit : 1;
    const int vg = FUSED ? c.vg : 0;
    if (threadIdx.x == 0) small_map_offsets(pb.S, maps_s, c.k, hoff, nsmall_s, gs);
    __syncthreads();
    for (int i = threadIdx.x; i < nsmall_s; i += kBinThreads) hist[i] = 0;
    __syncthreads();
    int32_t *cnt = w.row_off + static_cast<int64_t>(c.b) * pb.rows;
    if (c.valid) {
        const float2 xy = bin_xy<FUSED>(pb, c.pk);
        for (int s = 0; s < pb.S; ++s) {
            const MapInfo m = maps_s[c.k * pb.S + s];
            Footprint f;
            footprint(xy.x, xy.y, m, f);
            const int ho = hoff[s];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                if (f.row[cc] < 0) continue;
                if (ho >= 0) {
                    const int hi = ho + (f.row[cc] - m.start) * gs + vg;
                    if (DA_CHECK(pb.dbg_err, hi, hist_rows, kBoundsShared)) atomicAdd(&hist[hi], 1);
                } else {
                    const int64_t ri = static_cast<int64_t>(f.row[cc]) * gs + vg;
                    if (DA_CHECK(pb.dbg_err, ri, pb.rows, kBoundsRowCount)) atomicAdd(cnt + ri, 1);
                }
            }
        }
    }
    __syncthreads();
    flush_small_counts(pb, maps_s, hoff, c.k, hist, cnt, gs);
}

// ---------------------------------------------------------------- 2. scan

// Block-wide inclusive scan of one value per thread (1024 threads).
__device__ __forceinline__ int block_incl_scan(int v, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += n;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    total = warp_tot[31];
    return incl + (warp > 0 ? warp_tot[warp - 1] : 0);
}

// Each CTA turns kScanTile counts into tile-local exclusive offsets.
__global__ void __launch_bounds__(1024) scan_tiles_kernel(int32_t *data, int32_t *tile_sum)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[32];
    int4 *p = reinterpret_cast<int4 *>(data + static_cast<int64_t>(blockIdx.x) * kScanTile) + threadIdx.x;
    const int4 v = *p;
    const int s1 = v.x, s2 = s1 + v.y, s3 = s2 + v.z, s4 = s3 + v.w;
    int total;
    const int incl = block_incl_scan(s4, warp_tot, total);
    const int e = incl - s4;
    *p = make_int4(e, e + s1, e + s2, e + s3);
    if (threadIdx.x == 0) tile_sum[blockIdx.x] = total;
}

// One CTA: exclusive scan of the tile totals; the grand total goes to `end`.
__global__ void __launch_bounds__(1024) scan_sums_kernel(int32_t *tile_sum, int64_t ntiles, int32_t *end)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[32];
    int carry = 0;
    for (int64_t base = 0; base < ntiles; base += 1024) {
        const int64_t i = base + threadIdx.x;
        const int v = i < ntiles ? tile_sum[i] : 0;
        int total;
        const int incl = block_incl_scan(v, warp_tot, total);
        if (i < ntiles) tile_sum[i] = carry + incl - v;
        carry += total;
        __syncthreads();  // warp_tot is reused by the next chunk
    }
    if (threadIdx.x == 0) *end = carry;
}

__global__ void __launch_bounds__(256) scan_add_kernel(int32_t *data, const int32_t *tile_sum, int64_t n4)
{
    pdl_wait();
    pdl_trigger();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    const int add = tile_sum[(i * 4) / kScanTile];
    int4 *p = reinterpret_cast<int4 *>(data) + i;
    int4 v = *p;
    v.x += add;
    v.y += add;
    v.z += add;
    v.w += add;
    *p = v;
}

// ---------------------------------------------------------------- 3. fill

// The fill runs the same threads. For the small maps it counts again in
// shared memory, claims one contiguous range per touched row with a single
// global atomic, and then hands out slots inside the range with shared
// atomics. Every corner of a large map claims its slot with a global atomic.
template <bool FUSED>
__global__ void __launch_bounds__(kBinThreads) bin_fill_kernel(const Problem pb, const BinArgs w,
                                                                int ctas_per_view, int hist_rows)
{
    pdl_wait();
    pdl_trigger();
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    extern __shared__ int hist[];  // hist_rows entries
    __shared__ int hoff[DA_MAX_MAPS];
    __shared__ int nsmall_s;
    stage_maps(pb, maps_s);
    const BinCta c = bin_cta(pb, ctas_per_view);
    __syncthreads();
    // Virtual rows per pixel row: gsplit in the fused rewrite, else 1.
    const int gs = FUSED ? pb.gsplit : 1;
    const int vg = FUSED ? c.vg : 0;
    if (threadIdx.x == 0) small_map_offsets(pb.S, maps_s, c.k, hoff, nsmall_s, gs);
    __syncthreads();
    for (int i = threadIdx.x; i < nsmall_s; i += kBinThreads) hist[i] = 0;
    __syncthreads();
    float2 xy = make_float2(0.f, 0.f);
    if (c.valid) {
        xy = bin_xy<FUSED>(pb, c.pk);
        for (int s = 0; s < pb.S; ++s) {
            const int ho = hoff[s];
            if (ho < 0) continue;
            const MapInfo m = maps_s[c.k * pb.S + s];
            Footprint f;
            footprint(xy.x, xy.y, m, f);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int hi = ho + (f.row[cc] - m.start) * gs + vg;
                if (f.row[cc] >= 0 && DA_CHECK(pb.dbg_err, hi, hist_rows, kBoundsShared)) atomicAdd(&hist[hi], 1);
            }
        }
    }
    __syncthreads();
    // Claim each touched row's range: hist[] switches from counts to bases.
    int32_t *cursor = w.row_off + static_cast<int64_t>(c.b) * pb.rows;
    for (int s = 0; s < pb.S; ++s) {
        if (hoff[s] < 0) continue;
        const MapInfo m = maps_s[c.k * pb.S + s];
        const int n = m.H * m.W * gs;
        for (int r = threadIdx.x; r < n; r += kBinThreads) {
            const int v = hist[hoff[s] + r];
            if (v && DA_CHECK(pb.dbg_err, static_cast<int64_t>(m.start) * gs + r, pb.rows, kBoundsRowCount))
                hist[hoff[s] + r] = atomicAdd(cursor + m.start * gs + r, v);
        }
    }
    __syncthreads();
    if (!c.valid) return;
    for (int s = 0; s < pb.S; ++s) {
        const MapInfo m = maps_s[c.k * pb.S + s];
        Footprint f;
        footprint(xy.x, xy.y, m, f);
        const int ho = hoff[s];
        const int64_t sid = c.pk * pb.S + s;
        int pos[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            pos[cc] = -1;
            if (f.row[cc] < 0) continue;
            if (ho >= 0) {
                const int hi = ho + (f.row[cc] - m.start) * gs + vg;
                if (DA_CHECK(pb.dbg_err, hi, hist_rows, kBoundsShared)) pos[cc] = atomicAdd(&hist[hi], 1);
            } else {
                const int64_t ri = static_cast<int64_t>(f.row[cc]) * gs + vg;
                if (DA_CHECK(pb.dbg_err, ri, pb.rows, kBoundsRowCount)) pos[cc] = atomicAdd(cursor + ri, 1);
            }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            if (pos[cc] >= 0 && DA_CHECK(pb.dbg_err, pos[cc], w.ncap, kBoundsRecord))
                w.rec[pos[cc]] = make_int2(static_cast<int>(sid) * 4 + cc, __float_as_int(f.cw[cc]));
    }
}

// ------------------------------------------- 3b. sort (deterministic mode)

// The fill hands out slots inside a row with atomics, so the order of a
// row's records, and with it the rounding of the pull's sums, changes from
// run to run. In deterministic mode the records of every row are put in
// ascending order of their first field (sample id * 4 + corner, unique per
// record) before the pull. The sum over a
// row then always runs in the same order, so grad_feat (and everything
// computed from it) is the same bit for bit on every run.
//
// A row's records all come from the A*P locations of one view at one scale,
// and a location puts at most one corner in a row, so a row holds at most
// A*P records. Three tiers, by row length n:
//   n <= 8      one thread per row: rank = number of smaller keys;
//   n <= 128    one warp per row, records staged in shared memory, ranks;
//   n <= 2048   one CTA per row, bitonic sort in shared memory;
//   larger      one CTA per row, bitonic sort in place in global memory.
// The first kernel runs over all rows and lists the longer ones for the
// other three.

constexpr int kSortThreads = 256;
constexpr int kSortWarpMax = 128;
constexpr int kSortSmemMax = 2048;

__device__ __forceinline__ int row_begin(const BinArgs &w, int64_t r) { return r > 0 ? w.row_off[r - 1] : 0; }

__global__ void __launch_bounds__(kSortThreads) sort_short_rows_kernel(const Problem pb, const BinArgs w)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int n_list[3], base[3];
    if (threadIdx.x < 3) n_list[threadIdx.x] = 0;
    __syncthreads();
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kSortThreads + threadIdx.x;
    int n = 0, jb = 0;
    if (r < w.rows_total) {
        jb = row_begin(w, r);
        n = w.row_off[r] - jb;
    }
    const int tier = n <= 8 ? -1 : n <= kSortWarpMax ? 0 : n <= kSortSmemMax ? 1 : 2;
    int slot = 0;
    if (tier >= 0) slot = atomicAdd(&n_list[tier], 1);
    __syncthreads();
    if (threadIdx.x < 3 && n_list[threadIdx.x] > 0)
        base[threadIdx.x] = atomicAdd(w.sort_counts + threadIdx.x, n_list[threadIdx.x]);
    __syncthreads();
    if (tier >= 0) {
        const int64_t off = tier == 0 ? 0 : tier == 1 ? w.cap_m : w.cap_m + w.cap_s;
        w.sort_lists[off + base[tier] + slot] = static_cast<int32_t>(r);
        return;
    }
    if (n < 2) return;
    int2 e[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e[u] = u < n ? w.rec[jb + u] : make_int2(INT_MAX, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        if (u >= n) break;
        int rank = 0;
#pragma unroll
        for (int v = 0; v < 8; ++v) rank += (e[v].x < e[u].x) ? 1 : 0;  // padding keys are never smaller
        if (rank != u && DA_CHECK(pb.dbg_err, jb + rank, w.ncap, kBoundsRecord)) w.rec[jb + rank] = e[u];
    }
}

// Rows of 9..128 records: one warp per row. The records are staged in
// shared memory; each lane ranks its records against all of them.
__global__ void __launch_bounds__(kSortThreads) sort_warp_rows_kernel(const Problem pb, const BinArgs w)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int2 buf[kSortThreads / 32][kSortWarpMax];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int count = w.sort_counts[0];
    const int nwarps = gridDim.x * (kSortThreads / 32);
    for (int i = blockIdx.x * (kSortThreads / 32) + warp; i < count; i += nwarps) {
        const int64_t r = w.sort_lists[i];
        const int jb = row_begin(w, r);
        const int n = w.row_off[r] - jb;
        if (!DA_CHECK(pb.dbg_err, n - 1, kSortWarpMax, kBoundsShared)) continue;  // the tier bounds n
        for (int j = lane; j < n; j += 32) buf[warp][j] = w.rec[jb + j];
        __syncwarp();
        for (int j = lane; j < n; j += 32) {
            const int2 e = buf[warp][j];
            int rank = 0;
            for (int v = 0; v < n; ++v) rank += (buf[warp][v].x < e.x) ? 1 : 0;
            if (rank != j && DA_CHECK(pb.dbg_err, jb + rank, w.ncap, kBoundsRecord)) w.rec[jb + rank] = e;
        }
        __syncwarp();
    }
}

// Compare-exchange of a bitonic network: the smaller key goes to index lo.
template <typename Ptr>
__device__ __forceinline__ void cmp_swap(Ptr a, int lo, int hi)
{
    const int2 x = a[lo], y = a[hi];
    if (x.x > y.x) {
        a[lo] = y;
        a[hi] = x;
    }
}

// Ascending bitonic sort of a[0..n) by the block's threads, in the variant
// whose first step of every merge compares mirrored elements: every
// comparator then points the same way, and positions past n act as +inf
// that no comparator moves, so n need not be a power of two. `sync` is
// __syncthreads; a[] is shared or global memory.
template <typename Ptr>
__device__ void block_bitonic_sort(Ptr a, int n)
{
    int64_t np = 1;
    while (np < n) np <<= 1;
    const int half = static_cast<int>(np >> 1);
    for (int64_t k = 2; k <= np; k <<= 1) {
        const int lk = __ffsll(k) - 2;  // log2(k / 2)
        const int hk = static_cast<int>(k >> 1);
        for (int i = threadIdx.x; i < half; i += blockDim.x) {
            const int blk = i >> lk, o = i & (hk - 1);
            const int64_t lo = static_cast<int64_t>(blk) * k + o, hi = static_cast<int64_t>(blk) * k + k - 1 - o;
            if (hi < n) cmp_swap(a, static_cast<int>(lo), static_cast<int>(hi));
        }
        __syncthreads();
        for (int j = hk >> 1; j > 0; j >>= 1) {
            const int lj = __ffs(j) - 1;
            for (int i = threadIdx.x; i < half; i += blockDim.x) {
                const int blk = i >> lj, o = i & (j - 1);
                const int64_t lo = (static_cast<int64_t>(blk) << (lj + 1)) + o, hi = lo + j;
                if (hi < n) cmp_swap(a, static_cast<int>(lo), static_cast<int>(hi));
            }
            __syncthreads();
        }
    }
}

// Rows of 129..2048 records: one CTA per row, sorted in shared memory.
__global__ void __launch_bounds__(kSortThreads) sort_cta_rows_kernel(const Problem pb, const BinArgs w)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int2 buf[kSortSmemMax];
    const int count = w.sort_counts[1];
    const int32_t *list = w.sort_lists + w.cap_m;
    for (int i = blockIdx.x; i < count; i += gridDim.x) {
        const int64_t r = list[i];
        const int jb = row_begin(w, r);
        const int n = w.row_off[r] - jb;
        if (!DA_CHECK(pb.dbg_err, n - 1, kSortSmemMax, kBoundsShared)) continue;  // the tier bounds n
        for (int j = threadIdx.x; j < n; j += kSortThreads) buf[j] = w.rec[jb + j];
        __syncthreads();
        block_bitonic_sort(static_cast<int2 *>(buf), n);
        for (int j = threadIdx.x; j < n; j += kSortThreads) w.rec[jb + j] = buf[j];
        __syncthreads();
    }
}

// Rows of more than 2048 records (crowded pixels): one CTA per row, sorted
// in place in global memory (plain loads: the data changes under the
// kernel, so no read-only cache path).
__global__ void __launch_bounds__(1024) sort_long_rows_kernel(const Problem pb, const BinArgs w)
{
    pdl_wait();
    pdl_trigger();
    const int count = w.sort_counts[2];
    const int32_t *list = w.sort_lists + w.cap_m + w.cap_s;
    for (int i = blockIdx.x; i < count; i += gridDim.x) {
        const int64_t r = list[i];
        const int jb = row_begin(w, r);
        const int n = w.row_off[r] - jb;
        block_bitonic_sort(w.rec + jb, n);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- 5. epilogue

// The pull's leftover-row count is spent once the pull has finished; the
// epilogue, which follows it, clears it for the next pull of this workspace.
__device__ __forceinline__ void reset_left_count(const BinArgs &w)
{
    if (blockIdx.x == 0 && threadIdx.x == 0 && w.left_count) *w.left_count = 0;
}

__global__ void __launch_bounds__(256) epilogue_kernel(const Problem pb, const BinArgs w, float *grad_loc,
                                                       float *grad_weight, int64_t pk_begin, int64_t pk_end)
{
    pdl_wait();
    pdl_trigger();
    reset_left_count(w);
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t pk64 = pk_begin + ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (pk64 >= pk_end) return;  // whole warps leave together
    const int pk = static_cast<int>(pk64);
    const int k = pk - static_cast<int>(pb.div_K.div(pk)) * pb.K;
    const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + pk64 * 2);
    float gx = 0.f, gy = 0.f;
    const int sg = pb.S * pb.G;
    for (int i = lane; i < sg; i += 32) {
        const int s = static_cast<int>(pb.div_G.div(i));
        const int g = i - s * pb.G;
        const int64_t sid = pk64 * pb.S + s;
        const MapInfo m = maps_s[k * pb.S + s];
        Footprint f;
        footprint(xy.x, xy.y, m, f);
        const float wt = pb.weights[sid * pb.G + g];
        const float *dp = w.dpix + sid * 4 * pb.G + g;  // corner c at dp[c * G]
        const float d0 = f.row[0] >= 0 ? dp[0] : 0.f;
        const float d1 = f.row[1] >= 0 ? dp[pb.G] : 0.f;
        const float d2 = f.row[2] >= 0 ? dp[2 * pb.G] : 0.f;
        const float d3 = f.row[3] >= 0 ? dp[3 * pb.G] : 0.f;
        grad_weight[sid * pb.G + g] = f.cw[0] * d0 + f.cw[1] * d1 + f.cw[2] * d2 + f.cw[3] * d3;
        gx += static_cast<float>(m.W) * wt * (f.lh * (d3 - d2) + f.hh * (d1 - d0));
        gy += static_cast<float>(m.H) * wt * (f.lw * (d3 - d1) + f.hw * (d2 - d0));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        gx += __shfl_xor_sync(0xffffffffu, gx, o);
        gy += __shfl_xor_sync(0xffffffffu, gy, o);
    }
    if (lane == 0) {
        grad_loc[pk64 * 2] = gx;
        grad_loc[pk64 * 2 + 1] = gy;
    }
}

// The same with one lane per (location, scale), carrying all G groups in
// 16-byte vectors (G = 4 or 8, S dividing 32): a warp covers 32/S
// locations. The weights of a sample, its grad_weight and its four corners'
// d are 1 and 4 runs of G contiguous floats (the corners' side by side, the
// lanes' samples consecutive), so every access is a 16-byte vector, and
// the footprint and the bookkeeping run once per sample instead of once per
// (sample, group). The S lanes of a location sum grad_loc with shuffles.
template <int G>
__global__ void __launch_bounds__(256) epilogue_vec_kernel(const Problem pb, const BinArgs w, float *grad_loc,
                                                           float *grad_weight, int64_t npk, int s_log2)
{
    pdl_wait();
    pdl_trigger();
    reset_left_count(w);
    static_assert(G == 4 || G == 8, "16-byte vectors of G floats");
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int S = pb.S;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t pk64 = t >> s_log2;
    const int s = static_cast<int>(t & (S - 1));
    const bool live = pk64 < npk;
    // Lanes past the end run on the last location (whole locations, so the
    // shuffles stay within live lanes) and store nothing.
    const int pk = static_cast<int>(live ? pk64 : npk - 1);
    const int k = pk - static_cast<int>(pb.div_K.div(pk)) * pb.K;
    const int64_t sid = static_cast<int64_t>(pk) * S + s;
    const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + static_cast<int64_t>(pk) * 2);
    const MapInfo m = maps_s[k * S + s];
    Footprint f;
    footprint(xy.x, xy.y, m, f);
    float wt[G], d[4][G];
#pragma unroll
    for (int h = 0; h < G / 4; ++h) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(pb.weights + sid * G) + h);
        wt[4 * h] = v.x; wt[4 * h + 1] = v.y; wt[4 * h + 2] = v.z; wt[4 * h + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int h = 0; h < G / 4; ++h) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f.row[c] >= 0) v = __ldg(reinterpret_cast<const float4 *>(w.dpix + (sid * 4 + c) * G) + h);
            d[c][4 * h] = v.x; d[c][4 * h + 1] = v.y; d[c][4 * h + 2] = v.z; d[c][4 * h + 3] = v.w;
        }
    }
    float gw[G];
    float gx = 0.f, gy = 0.f;
    const float fw = static_cast<float>(m.W), fh = static_cast<float>(m.H);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        gw[g] = f.cw[0] * d[0][g] + f.cw[1] * d[1][g] + f.cw[2] * d[2][g] + f.cw[3] * d[3][g];
        gx += fw * wt[g] * (f.lh * (d[3][g] - d[2][g]) + f.hh * (d[1][g] - d[0][g]));
        gy += fh * wt[g] * (f.lw * (d[3][g] - d[1][g]) + f.hw * (d[2][g] - d[0][g]));
    }
    if (live) {
#pragma unroll
        for (int h = 0; h < G / 4; ++h)
            reinterpret_cast<float4 *>(grad_weight + sid * G)[h] =
                make_float4(gw[4 * h], gw[4 * h + 1], gw[4 * h + 2], gw[4 * h + 3]);
    }
    for (int o = 1; o < S; o <<= 1) {
        gx += __shfl_xor_sync(0xffffffffu, gx, o);
        gy += __shfl_xor_sync(0xffffffffu, gy, o);
    }
    if (live && s == 0) {
        grad_loc[static_cast<int64_t>(pk) * 2] = gx;
        grad_loc[static_cast<int64_t>(pk) * 2 + 1] = gy;
    }
}

// The fused layout's rewrite (G = 1): a location has S samples of one group,
// too few for a warp, so one thread takes a location. The gradients go to
// grad_loc_weight [.., 2 + S]: (dL/dx, dL/dy, dL/dw_0 .. dL/dw_{S-1}).
__global__ void __launch_bounds__(256) epilogue_fused_kernel(const Problem pb, const BinArgs w, float *glw,
                                                             int64_t npk)
{
    pdl_wait();
    pdl_trigger();
    reset_left_count(w);
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t pk64 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (pk64 >= npk) return;
    const int pk = static_cast<int>(pk64);
    const int k = pk - static_cast<int>(pb.div_K.div(pk)) * pb.K;
    const int E = 2 + pb.S;
    float *e = glw + pk64 * E;
    const float *le = pb.loc + pk64 * E;
    const float x = le[0], y = le[1];
    float gx = 0.f, gy = 0.f;
    for (int s = 0; s < pb.S; ++s) {
        const MapInfo m = maps_s[k * pb.S + s];
        Footprint f;
        footprint(x, y, m, f);
        const float wt = le[2 + s];
        const float *dp = w.dpix + (pk64 * pb.S + s) * 4;  // G = 1: corner c at dp[c]
        const float d0 = f.row[0] >= 0 ? dp[0] : 0.f;
        const float d1 = f.row[1] >= 0 ? dp[1] : 0.f;
        const float d2 = f.row[2] >= 0 ? dp[2] : 0.f;
        const float d3 = f.row[3] >= 0 ? dp[3] : 0.f;
        e[2 + s] = f.cw[0] * d0 + f.cw[1] * d1 + f.cw[2] * d2 + f.cw[3] * d3;
        gx += static_cast<float>(m.W) * wt * (f.lh * (d3 - d2) + f.hh * (d1 - d0));
        gy += static_cast<float>(m.H) * wt * (f.lw * (d3 - d1) + f.hw * (d2 - d0));
    }
    e[0] = gx;
    e[1] = gy;
}

// ---------------------------------------------------------------- launch

}  // namespace

cudaError_t launch_backward_binned(const BwdArgs &a, const BinArgs &w, int feat_dtype, cudaStream_t st, int stages)
{
    const Problem &pb = a.pb;
    cudaError_t e;
    const int64_t npk = static_cast<int64_t>(pb.num_ba) * pb.P * pb.K;
    if (!(stages & kStageBin)) goto pull_stage;
    // 1. counts
    if (w.ntiles > 0) {
        e = launch_zero_fill(reinterpret_cast<float *>(w.row_off), w.ntiles * kScanTile + kRowOffTail, st);
        if (e != cudaSuccess) return e;
    }
    {
    const int ctas_per_view = (pb.A * pb.P + kBinThreads - 1) / kBinThreads;
    const int64_t bin_grid = static_cast<int64_t>(pb.B) * pb.K * ctas_per_view;
    // Shared histogram: as many entries as the largest set of small maps of
    // any camera needs (the kernels pick the same maps).
    int hist_rows = 0;
    for (int k = 0; k < pb.K; ++k) {
        int hoff[DA_MAX_MAPS], nsmall = 0;
        small_map_offsets(pb.S, pb.maps, k, hoff, nsmall, pb.layout == kLayoutFused ? pb.gsplit : 1);
        hist_rows = nsmall > hist_rows ? nsmall : hist_rows;
    }
    const size_t hist_bytes = static_cast<size_t>(hist_rows) * sizeof(int);
    if (w.nsid > 0) {
        if (pb.layout == kLayoutFused)
            e = launch_pdl(bin_count_kernel<true>, dim3(static_cast<unsigned>(bin_grid)), dim3(kBinThreads),
                hist_bytes, st, pb, w, ctas_per_view, hist_rows);
        else
            e = launch_pdl(bin_count_kernel<false>, dim3(static_cast<unsigned>(bin_grid)), dim3(kBinThreads),
                hist_bytes, st, pb, w, ctas_per_view, hist_rows);
        if (e != cudaSuccess) return e;
    }
    // 2. offsets
    if (w.ntiles > 0) {
        e = launch_pdl(scan_tiles_kernel, dim3(static_cast<unsigned>(w.ntiles)), dim3(1024), 0, st,
            w.row_off, w.tile_sum);
        if (e != cudaSuccess) return e;
        e = launch_pdl(scan_sums_kernel, dim3(1), dim3(1024), 0, st,
            w.tile_sum, w.ntiles, w.row_off + w.ntiles * kScanTile);
        if (e != cudaSuccess) return e;
        const int64_t n4 = w.ntiles * kScanTile / 4;
        e = launch_pdl(scan_add_kernel, dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, st,
            w.row_off, w.tile_sum, n4);
        if (e != cudaSuccess) return e;
    }
    // 3. records
    if (w.nsid > 0) {
        if (pb.layout == kLayoutFused)
            e = launch_pdl(bin_fill_kernel<true>, dim3(static_cast<unsigned>(bin_grid)), dim3(kBinThreads),
                hist_bytes, st, pb, w, ctas_per_view, hist_rows);
        else
            e = launch_pdl(bin_fill_kernel<false>, dim3(static_cast<unsigned>(bin_grid)), dim3(kBinThreads),
                hist_bytes, st, pb, w, ctas_per_view, hist_rows);
        if (e != cudaSuccess) return e;
    }
    // 3b. deterministic order inside every row
    if (w.sort_lists && w.nsid > 0 && w.rows_total > 0) {
        const int64_t g1 = (w.rows_total + kSortThreads - 1) / kSortThreads;
        e = launch_pdl(sort_short_rows_kernel, dim3(static_cast<unsigned>(g1)), dim3(kSortThreads), 0, st, pb, w);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        // Persistent grids over the row lists (their lengths are on the device).
        e = launch_pdl(sort_warp_rows_kernel, dim3(static_cast<unsigned>(sms * 8)), dim3(kSortThreads), 0, st, pb, w);
        if (e != cudaSuccess) return e;
        // Sixteen CTAs per SM, twice the resident maximum: each row's bitonic
        // network is a chain of short barrier-separated stages, so the kernel
        // is latency-bound and more CTAs in flight help. Deterministic
        // backward at the 6-camera training shape: 947 us with 4 CTAs per SM,
        // 931 us with 8, 927 us with 16.
        e = launch_pdl(sort_cta_rows_kernel, dim3(static_cast<unsigned>(sms * 16)), dim3(kSortThreads), 0, st, pb, w);
        if (e != cudaSuccess) return e;
        e = launch_pdl(sort_long_rows_kernel, dim3(static_cast<unsigned>(sms)), dim3(1024), 0, st, pb, w);
        if (e != cudaSuccess) return e;
    }
    }
pull_stage:
    if (!(stages & kStagePull)) return cudaSuccess;
    // 4. grad_feat and d
    if (w.rows_total > 0) {
        e = launch_pull(a, w, feat_dtype, st);
        if (e != cudaSuccess) return e;
    }
    // 5. grad_weight and grad_loc
    if (npk > 0 && pb.layout == kLayoutFused) {
        e = launch_pdl(epilogue_fused_kernel, dim3(static_cast<unsigned>((npk + 255) / 256)), dim3(256), 0, st,
            pb, w, a.grad_loc, npk);
        if (e != cudaSuccess) return e;
    } else if (npk > 0) {
        // The vector kernel reads weights and writes grad_weight as 16-byte
        // vectors; the interface promises only 4-byte alignment for those.
        const bool aligned16 = (reinterpret_cast<uintptr_t>(pb.weights) % 16) == 0 &&
                               (reinterpret_cast<uintptr_t>(a.grad_weight) % 16) == 0;
        const bool vec = aligned16 && (pb.G == 4 || pb.G == 8) && pb.S >= 1 && pb.S <= 32 &&
                         (32 % pb.S) == 0;
        if (vec) {
            int s_log2 = 0;
            while ((1 << s_log2) < pb.S) ++s_log2;
            const int64_t threads = npk << s_log2;
            const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
            if (pb.G == 8)
                e = launch_pdl(epilogue_vec_kernel<8>, dim3(grid), dim3(256), 0, st,
                    pb, w, a.grad_loc, a.grad_weight, npk, s_log2);
            else
                e = launch_pdl(epilogue_vec_kernel<4>, dim3(grid), dim3(256), 0, st,
                    pb, w, a.grad_loc, a.grad_weight, npk, s_log2);
        } else {
            e = launch_pdl(epilogue_kernel, dim3(static_cast<unsigned>((npk * 32 + 255) / 256)), dim3(256), 0, st,
                pb, w, a.grad_loc, a.grad_weight, 0, npk);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace da
