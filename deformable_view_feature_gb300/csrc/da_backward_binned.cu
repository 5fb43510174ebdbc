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
//   1. count   one thread per sample (all groups at once) counts its in-map
//              corners per feature row (row_off, one integer red per corner);
//   2. scan    exclusive prefix sum of the counts (three small kernels);
//   3. fill    the same threads claim a slot in their rows (atomic add with
//              return) and write the record {sample*4 + corner, corner
//              weight}, plus the slot of each corner (pos4);
//   4. pull    a CTA owns a batch item b, a group g and a range of rows of
//              about equal record count. grad_out[b, :, g] sits in shared
//              memory. Four lanes own one row (8 channels each): per record
//              they read the anchor's grad_out slice, accumulate
//              (w * w_i) * grad_out into the row's grad_feat, and form
//              d = feat_row . grad_out. The grad_feat row is stored once
//              (no zero-fill); d goes to dpix at the record's index;
//   5. epilogue one warp per location (b, a, p, k): its lanes take the
//              (s, g) samples, gather the four corners' d through pos4, and
//              form grad_weight = sum w_i d_i and the two grad_loc sums,
//              reduced by shuffles. Every output has one owner, so there
//              are no atomics.
#include <algorithm>

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
    o = align256(o + static_cast<size_t>(L.ntiles * kScanTile + 4) * 4);
    L.off_tile_sum = o;
    o = align256(o + static_cast<size_t>(L.ntiles + 4) * 4);
    L.off_rec_cid = o;
    o = align256(o + static_cast<size_t>(L.ncap) * 4);
    L.off_rec_cw = o;
    o = align256(o + static_cast<size_t>(L.ncap) * 4);
    L.off_pos4 = o;
    o = align256(o + static_cast<size_t>(L.nsid) * 16);
    L.off_dpix = o;
    o = align256(o + static_cast<size_t>(L.ncap) * static_cast<size_t>(G) * 4);
    L.bytes = o;
    return L;
}

namespace {

// Sample id -> (location id (b*A+a)*P+p)*K+k, scale s, camera k, batch item b).
struct SampleIdx {
    int pk, s, k, b;
};

__device__ __forceinline__ SampleIdx split_sample(const Problem &pb, int sid)
{
    SampleIdx r;
    r.pk = static_cast<int>(pb.div_S.div(sid));
    r.s = sid - r.pk * pb.S;
    const int bap = static_cast<int>(pb.div_K.div(r.pk));
    r.k = r.pk - bap * pb.K;
    const int ba = static_cast<int>(pb.div_P.div(bap));
    r.b = static_cast<int>(pb.div_A.div(ba));
    return r;
}

// ---------------------------------------------------------------- 1. count

__global__ void __launch_bounds__(256) bin_count_kernel(const Problem pb, const BinArgs w)
{
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t sid64 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (sid64 >= w.nsid) return;
    const int sid = static_cast<int>(sid64);
    const SampleIdx si = split_sample(pb, sid);
    const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + static_cast<int64_t>(si.pk) * 2);
    Footprint f;
    footprint(xy.x, xy.y, maps_s[si.k * pb.S + si.s], f);
    int32_t *cnt = w.row_off + static_cast<int64_t>(si.b) * pb.rows;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (f.row[c] >= 0) atomicAdd(cnt + f.row[c], 1);
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

__global__ void __launch_bounds__(256) bin_fill_kernel(const Problem pb, const BinArgs w)
{
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t sid64 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (sid64 >= w.nsid) return;
    const int sid = static_cast<int>(sid64);
    const SampleIdx si = split_sample(pb, sid);
    const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + static_cast<int64_t>(si.pk) * 2);
    Footprint f;
    footprint(xy.x, xy.y, maps_s[si.k * pb.S + si.s], f);
    int32_t *cursor = w.row_off + static_cast<int64_t>(si.b) * pb.rows;
    int pos[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        pos[c] = -1;
        if (f.row[c] >= 0) {
            pos[c] = atomicAdd(cursor + f.row[c], 1);
            w.rec_cid[pos[c]] = sid * 4 + c;
            w.rec_cw[pos[c]] = f.cw[c];
        }
    }
    reinterpret_cast<int4 *>(w.pos4)[sid64] = make_int4(pos[0], pos[1], pos[2], pos[3]);
}

// ---------------------------------------------------------------- 4. pull

constexpr int kPullThreads = 1024;

// Sum d[0..3] over the LPP lanes of one row, as in the gather kernels: each
// halving step sends half of the values still held. The lane left holding
// record u's sum stores it to dst[u] when u < nvalid.
template <int LPP>
__device__ __forceinline__ void pixel_sum_store(const float (&d)[4], int sub, int nvalid, float *dst)
{
    if constexpr (LPP >= 4) {
        const bool hA = (sub & (LPP / 2)) != 0;
        float a0 = hA ? d[2] : d[0], a1 = hA ? d[3] : d[1];
        const float s0 = hA ? d[0] : d[2], s1 = hA ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, LPP / 2);
        a1 += __shfl_xor_sync(0xffffffffu, s1, LPP / 2);
        const bool hB = (sub & (LPP / 4)) != 0;
        float r = hB ? a1 : a0;
        const float t = hB ? a0 : a1;
        r += __shfl_xor_sync(0xffffffffu, t, LPP / 4);
#pragma unroll
        for (int m = LPP / 8; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
        const int u = (hA ? 2 : 0) + (hB ? 1 : 0);
        if ((sub & (LPP / 4 - 1)) == 0 && u < nvalid) dst[u] = r;
    } else if constexpr (LPP == 2) {
        const bool h = (sub & 1) != 0;
        float a0 = h ? d[2] : d[0], a1 = h ? d[3] : d[1];
        const float s0 = h ? d[0] : d[2], s1 = h ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        a1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        const int u0 = h ? 2 : 0;
        if (u0 < nvalid) dst[u0] = a0;
        if (u0 + 1 < nvalid) dst[u0 + 1] = a1;
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u < nvalid) dst[u] = d[u];
    }
}

// Feature values of one 4-channel chunk, widened to fp32.
template <typename T>
__device__ __forceinline__ float4 load_feat4(const void *p);

template <>
__device__ __forceinline__ float4 load_feat4<float>(const void *p)
{
    return __ldg(reinterpret_cast<const float4 *>(p));
}

template <>
__device__ __forceinline__ float4 load_feat4<Bf16Tag>(const void *p)
{
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
}

// First row R in [lo, hi] whose records start at or after t. The records of
// row R start at row_end[R-1] (0 for R = 0) once the fill has run.
__device__ int64_t first_row_from(const int32_t *row_end, int64_t lo, int64_t hi, int64_t t)
{
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        const int64_t st = mid > 0 ? row_end[mid - 1] : 0;
        if (st >= t) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

struct PullArgs {
    Problem pb;
    const float *grad_out;
    float *grad_feat;
    BinArgs w;
    int npieces;
};

// LPP lanes own one feature row of one group; each holds DPL channels.
// For DPL = 8, a lane holds two 4-channel chunks. Rows in odd slots of the
// warp take them in swapped order. Then the two shared loads of a record
// touch complementary bank halves for even and odd rows, and the eight rows
// of a warp read conflict-free.
template <typename T, int LPP, int DPL, bool GO_SMEM>
__global__ void __launch_bounds__(kPullThreads, 1) pull_kernel(const PullArgs args)
{
    constexpr int PPW = 32 / LPP;      // rows per warp
    constexpr int NCH = DPL / 4;       // 4-channel chunks per lane
    constexpr int ESZ = sizeof(T) == 4 ? 4 : 2;
    constexpr int RPL = LPP >= 4 ? 1 : 4 / LPP;  // records a lane loads per batch of 4
    const Problem &pb = args.pb;
    const BinArgs &w = args.w;
    extern __shared__ __align__(16) float go_s[];  // [A][D] when GO_SMEM

    const int bg = static_cast<int>(blockIdx.x) / args.npieces;
    const int piece = static_cast<int>(blockIdx.x) - bg * args.npieces;
    const int b = static_cast<int>(pb.div_G.div(bg));
    const int g = bg - b * pb.G;
    const int D = pb.D;

    const float *go_g = args.grad_out + static_cast<int64_t>(b) * pb.A * pb.C + static_cast<int64_t>(g) * D;
    if constexpr (GO_SMEM) {
        const int n4 = pb.A * (D / 4);
        for (int i = threadIdx.x; i < n4; i += kPullThreads) {
            const int a = i / (D / 4);
            const int c4 = i - a * (D / 4);
            reinterpret_cast<float4 *>(go_s)[i] =
                *reinterpret_cast<const float4 *>(go_g + static_cast<int64_t>(a) * pb.C + c4 * 4);
        }
        __syncthreads();
    }

    // This CTA's rows: about 1/npieces of the batch item's records.
    const int64_t R0 = static_cast<int64_t>(b) * pb.rows, R1 = R0 + pb.rows;
    const int64_t s0 = R0 > 0 ? w.row_off[R0 - 1] : 0;
    const int64_t s1 = R1 > 0 ? w.row_off[R1 - 1] : 0;
    const int64_t tot = s1 - s0;
    const int64_t r_lo = piece == 0 ? R0 : first_row_from(w.row_off, R0, R1, s0 + tot * piece / args.npieces);
    const int64_t r_hi = piece == args.npieces - 1
                             ? R1
                             : first_row_from(w.row_off, R0, R1, s0 + tot * (piece + 1) / args.npieces);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane / LPP, sub = lane % LPP;
    const int par = NCH == 2 ? (q & 1) : 0;
    int coff[NCH];  // channel offset of logical chunk h within the group
#pragma unroll
    for (int h = 0; h < NCH; ++h) coff[h] = sub * DPL + (h ^ par) * 4;
    float *dpix_g = w.dpix + static_cast<int64_t>(g) * w.ncap;

    for (int64_t base = r_lo + static_cast<int64_t>(warp) * PPW; base < r_hi;
         base += static_cast<int64_t>(kPullThreads / 32) * PPW) {
        const int64_t R = base + q;
        const bool active = R < r_hi;
        const int jb = active ? (R > 0 ? w.row_off[R - 1] : 0) : 0;
        const int je = active ? w.row_off[R] : 0;
        const int n = je - jb;

        float v[DPL], acc[DPL];
        {
            const char *fp = static_cast<const char *>(pb.feat) +
                             (R * pb.C + static_cast<int64_t>(g) * D) * ESZ;
#pragma unroll
            for (int h = 0; h < NCH; ++h) {
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                if (active) t = load_feat4<T>(fp + static_cast<int64_t>(coff[h]) * ESZ);
                v[4 * h] = t.x;
                v[4 * h + 1] = t.y;
                v[4 * h + 2] = t.z;
                v[4 * h + 3] = t.w;
            }
        }
#pragma unroll
        for (int m = 0; m < DPL; ++m) acc[m] = 0.f;

        int nmax = n;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));

        for (int k0 = 0; k0 < nmax; k0 += 4) {
            // Records k0..k0+3 of this row: lane `sub` loads those with
            // index = sub (mod LPP), then every lane of the row gets them by
            // shuffles.
            int ra[RPL];
            float rt[RPL];
#pragma unroll
            for (int r = 0; r < RPL; ++r) {
                const int u = sub + r * LPP;
                ra[r] = 0;
                rt[r] = 0.f;
                if (u < 4 && k0 + u < n) {
                    const int cid = w.rec_cid[jb + k0 + u];
                    const int sid = cid >> 2;
                    const int ba = static_cast<int>(pb.div_PKS.div(sid));
                    ra[r] = ba - b * pb.A;
                    rt[r] = w.rec_cw[jb + k0 + u] * pb.weights[static_cast<int64_t>(sid) * pb.G + g];
                }
            }
            float d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int src = q * LPP + (u % LPP);
                const int a = LPP > 1 ? __shfl_sync(0xffffffffu, ra[u / LPP], src) : ra[u / LPP];
                const float tw = LPP > 1 ? __shfl_sync(0xffffffffu, rt[u / LPP], src) : rt[u / LPP];
                const bool valid = k0 + u < n;
                float gov[DPL];
#pragma unroll
                for (int h = 0; h < NCH; ++h) {
                    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (valid) {
                        if constexpr (GO_SMEM)
                            t = *reinterpret_cast<const float4 *>(&go_s[a * D + coff[h]]);
                        else
                            t = __ldg(reinterpret_cast<const float4 *>(go_g + static_cast<int64_t>(a) * pb.C + coff[h]));
                    }
                    gov[4 * h] = t.x;
                    gov[4 * h + 1] = t.y;
                    gov[4 * h + 2] = t.z;
                    gov[4 * h + 3] = t.w;
                }
                float dd = 0.f;
#pragma unroll
                for (int m = 0; m < DPL; ++m) {
                    dd = fmaf(v[m], gov[m], dd);
                    acc[m] = fmaf(tw, gov[m], acc[m]);
                }
                d[u] = dd;
            }
            pixel_sum_store<LPP>(d, sub, n - k0, dpix_g + jb + k0);
        }

        if (active) {
            float *gp = args.grad_feat + R * pb.C + static_cast<int64_t>(g) * D;
#pragma unroll
            for (int h = 0; h < NCH; ++h)
                *reinterpret_cast<float4 *>(gp + coff[h]) =
                    make_float4(acc[4 * h], acc[4 * h + 1], acc[4 * h + 2], acc[4 * h + 3]);
        }
    }
}

// ---------------------------------------------------------------- 5. epilogue

__global__ void __launch_bounds__(256) epilogue_kernel(const Problem pb, const BinArgs w, float *grad_loc,
                                                       float *grad_weight, int64_t npk)
{
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t pk64 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (pk64 >= npk) return;  // whole warps leave together
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
        const int4 pos = reinterpret_cast<const int4 *>(w.pos4)[sid];
        const float *dp = w.dpix + static_cast<int64_t>(g) * w.ncap;
        const float d0 = pos.x >= 0 ? dp[pos.x] : 0.f;
        const float d1 = pos.y >= 0 ? dp[pos.y] : 0.f;
        const float d2 = pos.z >= 0 ? dp[pos.z] : 0.f;
        const float d3 = pos.w >= 0 ? dp[pos.w] : 0.f;
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

// ---------------------------------------------------------------- launch

template <typename T, int LPP, int DPL>
cudaError_t launch_pull(const PullArgs &pa, int64_t grid, size_t go_bytes, cudaStream_t st)
{
    constexpr size_t kMaxGo = 200 * 1024;
    if (go_bytes <= kMaxGo) {
        auto kern = pull_kernel<T, LPP, DPL, true>;
        if (go_bytes > 48 * 1024) {
            const cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(go_bytes));
            if (e != cudaSuccess) return e;
        }
        kern<<<static_cast<unsigned>(grid), kPullThreads, go_bytes, st>>>(pa);
    } else {
        pull_kernel<T, LPP, DPL, false><<<static_cast<unsigned>(grid), kPullThreads, 0, st>>>(pa);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_pull(const PullArgs &pa, int64_t grid, size_t go_bytes, cudaStream_t st)
{
    switch (pa.pb.D) {
        case 4: return launch_pull<T, 1, 4>(pa, grid, go_bytes, st);
        case 8: return launch_pull<T, 1, 8>(pa, grid, go_bytes, st);
        case 16: return launch_pull<T, 2, 8>(pa, grid, go_bytes, st);
        case 32: return launch_pull<T, 4, 8>(pa, grid, go_bytes, st);
        case 64: return launch_pull<T, 8, 8>(pa, grid, go_bytes, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_backward_binned(const BwdArgs &a, const BinArgs &w, int feat_dtype, cudaStream_t st)
{
    const Problem &pb = a.pb;
    cudaError_t e;
    // 1. counts
    if (w.ntiles > 0) {
        e = launch_zero_fill(reinterpret_cast<float *>(w.row_off), w.ntiles * kScanTile + 4, st);
        if (e != cudaSuccess) return e;
    }
    if (w.nsid > 0) {
        bin_count_kernel<<<static_cast<unsigned>((w.nsid + 255) / 256), 256, 0, st>>>(pb, w);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 2. offsets
    if (w.ntiles > 0) {
        scan_tiles_kernel<<<static_cast<unsigned>(w.ntiles), 1024, 0, st>>>(w.row_off, w.tile_sum);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        scan_sums_kernel<<<1, 1024, 0, st>>>(w.tile_sum, w.ntiles, w.row_off + w.ntiles * kScanTile);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int64_t n4 = w.ntiles * kScanTile / 4;
        scan_add_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, st>>>(w.row_off, w.tile_sum, n4);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 3. records
    if (w.nsid > 0) {
        bin_fill_kernel<<<static_cast<unsigned>((w.nsid + 255) / 256), 256, 0, st>>>(pb, w);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 4. grad_feat and d
    if (w.rows_total > 0) {
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        PullArgs pa{pb, a.grad_out, a.grad_feat, w, 1};
        const int64_t pairs = static_cast<int64_t>(pb.B) * pb.G;
        pa.npieces = static_cast<int>(std::max<int64_t>(1, (6 * static_cast<int64_t>(sms) + pairs - 1) / pairs));
        const size_t go_bytes = static_cast<size_t>(pb.A) * pb.D * sizeof(float);
        e = feat_dtype == DA_BF16 ? dispatch_pull<Bf16Tag>(pa, pairs * pa.npieces, go_bytes, st)
                                  : dispatch_pull<float>(pa, pairs * pa.npieces, go_bytes, st);
        if (e != cudaSuccess) return e;
    }
    // 5. grad_weight and grad_loc
    const int64_t npk = static_cast<int64_t>(pb.num_ba) * pb.P * pb.K;
    if (npk > 0) {
        epilogue_kernel<<<static_cast<unsigned>((npk * 32 + 255) / 256), 256, 0, st>>>(pb, w, a.grad_loc,
                                                                                         a.grad_weight, npk);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace da
