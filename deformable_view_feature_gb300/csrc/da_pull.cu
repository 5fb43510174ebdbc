// Pull step of the binned backward of the deformable-aggregation operator:
// grad_feat (the page "Inside Sparse4D's CUDA core", §4.1: every corner
// adds w_i * grad_out * w to its feature row) computed row by row from the
// corner contributions that the binning (da_backward_binned.cu) sorted by
// feature row, together with d = feat_row . grad_out per record and group,
// from which grad_weight and grad_loc follow.
#include <algorithm>
#include <cmath>


#include "da_internal.cuh"

namespace da {

namespace {

// Sum d[0..3] over the L lanes of one group, as in the gather kernels: each
// halving step sends half of the values still held. The lane left holding
// record u's sum stores it to base[key[u] * stride] when u < nvalid.
__device__ __forceinline__ int pick4(const int (&k)[4], int u)
{
    return u == 0 ? k[0] : u == 1 ? k[1] : u == 2 ? k[2] : k[3];
}

// err, kcap: a bounds-checking build checks every key against kcap records.
template <int L>
__device__ __forceinline__ void group_sum_store(const float (&d)[4], int sub, int nvalid, float *base,
                                                const int (&key)[4], int stride, uint32_t *err, int64_t kcap)
{
    if constexpr (L >= 4) {
        const bool hA = (sub & (L / 2)) != 0;
        float a0 = hA ? d[2] : d[0], a1 = hA ? d[3] : d[1];
        const float s0 = hA ? d[0] : d[2], s1 = hA ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, L / 2);
        a1 += __shfl_xor_sync(0xffffffffu, s1, L / 2);
        const bool hB = (sub & (L / 4)) != 0;
        float r = hB ? a1 : a0;
        const float t = hB ? a0 : a1;
        r += __shfl_xor_sync(0xffffffffu, t, L / 4);
#pragma unroll
        for (int m = L / 8; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
        const int u = (hA ? 2 : 0) + (hB ? 1 : 0);
        const int ku = pick4(key, u);
        if ((sub & (L / 4 - 1)) == 0 && u < nvalid && DA_CHECK(err, ku, kcap, kBoundsSample))
            base[static_cast<int64_t>(ku) * stride] = r;
    } else if constexpr (L == 2) {
        const bool h = (sub & 1) != 0;
        float a0 = h ? d[2] : d[0], a1 = h ? d[3] : d[1];
        const float s0 = h ? d[0] : d[2], s1 = h ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        a1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        const int u0 = h ? 2 : 0;
        const int k0 = pick4(key, u0), k1 = pick4(key, u0 + 1);
        if (u0 < nvalid && DA_CHECK(err, k0, kcap, kBoundsSample)) base[static_cast<int64_t>(k0) * stride] = a0;
        if (u0 + 1 < nvalid && DA_CHECK(err, k1, kcap, kBoundsSample)) base[static_cast<int64_t>(k1) * stride] = a1;
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u < nvalid && DA_CHECK(err, key[u], kcap, kBoundsSample)) base[static_cast<int64_t>(key[u]) * stride] = d[u];
    }
}

// 32 contiguous bytes (8 floats) at a 32-byte aligned address, in one
// 256-bit read-only load (sm_100 and later).
__device__ __forceinline__ void ldg_v8(const void *p, float4 &x, float4 &y)
{
    asm("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w), "=f"(y.x), "=f"(y.y), "=f"(y.z), "=f"(y.w)
        : "l"(p));
}

// The same with an L1 policy: no_allocate for data read once (feature rows,
// sample weights, records), so it does not push grad_out rows out of L1;
// evict_last for the grad_out rows, which neighbouring rows' warps read
// again. Pull + epilogue at the 6-camera training shape: 618 us with the
// default policy, 610 with no_allocate alone, 604 with both.
__device__ __forceinline__ void ldg_v8_stream(const void *p, float4 &x, float4 &y)
{
    asm("ld.global.nc.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w), "=f"(y.x), "=f"(y.y), "=f"(y.z), "=f"(y.w)
        : "l"(p));
}

__device__ __forceinline__ void ldg_v8_keep(const void *p, float4 &x, float4 &y)
{
    asm("ld.global.nc.L1::evict_last.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w), "=f"(y.x), "=f"(y.y), "=f"(y.z), "=f"(y.w)
        : "l"(p));
}

__device__ __forceinline__ int2 ldg_record_stream(const int2 *p)
{
    int2 r;
    asm("ld.global.nc.L1::no_allocate.v2.s32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// 8 floats to a 32-byte aligned address in one 256-bit store.
__device__ __forceinline__ void stg_v8(void *p, const float4 x, const float4 y)
{
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :
                 : "l"(p), "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w), "f"(y.x), "f"(y.y), "f"(y.z), "f"(y.w)
                 : "memory");
}

// The 8 floats at p: one 256-bit load when V8 (p 32-byte aligned), else two
// 128-bit loads. With a lane's 8 channels contiguous and the lanes of a row
// side by side, the 256-bit form reads a whole row segment in one warp-wide
// instruction whose every 32-byte sector is fully used; the two 128-bit
// loads each touch every sector of the segment half.
template <bool V8>
__device__ __forceinline__ void ldg_f32x8(const float *p, float4 &x, float4 &y)
{
    if constexpr (V8) {
        ldg_v8(p, x, y);
    } else {
        x = __ldg(reinterpret_cast<const float4 *>(p));
        y = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
}

// Eight feature values of one lane, widened to fp32.
template <typename T, bool V8>
__device__ __forceinline__ void load_feat8(const void *p, float (&v)[8])
{
    if constexpr (sizeof(T) == 4) {
        float4 a, c;
        if constexpr (V8) ldg_v8_stream(p, a, c);
        else ldg_f32x8<V8>(static_cast<const float *>(p), a, c);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    } else {
        Chunk<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(p)), v);
    }
}

// How the rows are shared out. kRowsAll: one warp per feature row (LPR
// lanes per row), over every row. With row groups (pull_plan) the maps whose
// rows hold few records each are pulled in runs of consecutive pixels, one
// run per warp and four vertically adjacent runs per CTA (kRowGroups,
// pull_groups), and the other maps one row per warp (kRowsCoarse, the
// rows enumerated through pb.maps[].pad). Rows past a run's record cap are
// pulled one warp per row from a list afterwards (kRowsListed, w.left).
constexpr int kRowsAll = 0, kRowsCoarse = 1, kRowGroups = 2, kRowsListed = 3;

struct PullArgs {
    Problem pb;  // with row groups, pb.maps[i].pad: map i's first unit (row or block) of its kind
    const float *grad_out;
    float *grad_feat;
    BinArgs w;
    int64_t row_begin, row_end;  // units this launch covers: rows (kRowsAll, kRowsCoarse) or blocks
    int weights_v8;              // G == 8 and weights 32-byte aligned: one 256-bit load per sample
    int mode;                    // kRowsAll, kRowsCoarse or kRowGroups
    int64_t units_per_b;         // kRowsCoarse, kRowGroups: units per batch item
    uint64_t group_maps;         // bit i: map i is pulled in row groups
    uint8_t rw_log[DA_MAX_MAPS]; // log2 of the pixels per run (block width) of each grouped map
};

// 4 warps per CTA. The register-limited occupancy (32 warps per SM) is the
// same for any CTA size, but rows hold from 1 to a few hundred records and a
// CTA retires with its slowest warp: smaller CTAs free their slots sooner.
// Training shape: 775 us with 128 threads, 805 with 256, 917 with 512
// (787 with 64 and 781 with 32).
constexpr int kPullThreads = 128;


// One record's contribution to a lane's 8 channels: acc += tw * go, and the
// lane's part of d = feat_row . go. Packed two-wide fp32 FMAs (each half
// rounded on its own) halve the instruction count of this, the pull's
// innermost step; the dot product runs as two partial sums (even and odd
// channels) added at the end.
__device__ __forceinline__ float record_fma2(const float2 (&v)[4], const float4 x, const float4 y, float tw,
                                             float2 (&acc)[4])
{
    const float2 go[4] = {make_float2(x.x, x.y), make_float2(x.z, x.w), make_float2(y.x, y.y),
                          make_float2(y.z, y.w)};
    const float2 t = make_float2(tw, tw);
    float2 dd = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        dd = __ffma2_rn(v[m], go[m], dd);
        acc[m] = __ffma2_rn(t, go[m], acc[m]);
    }
    return dd.x + dd.y;
}

// Shared memory of one pull warp, per chunk: for each of its RPW rows, CH
// records (see pull_kernel), each with
//   meta  {anchor a of the record within its batch item, corner weight bits},
//   ksm   the record's key (sample id * 4 + corner),
//   wsm   the G weights of the record's sample, group-major: wsm[g][slot],
//         each group's row padded by 4 floats. The walk reads four slots of
//         every group at once (one 16-byte load per lane, the G groups at G
//         addresses): rows 4 banks apart keep that one wavefront instead of G.
// slot = row in warp * CH + record in chunk.
__host__ __device__ constexpr int pull_wpitch(int slots) { return slots + 4; }

__host__ __device__ inline size_t pull_smem_per_warp(int slots, int G)
{
    return (static_cast<size_t>(slots) * 3 + static_cast<size_t>(G) * pull_wpitch(slots)) * 4;
}

// LPR = C/8 lanes own one feature row, 8 channels each, all groups; a warp
// holds RPW = 32/LPR rows. LPG = D/8 lanes hold one group. The records of a
// row are taken in chunks of CH = max(LPR, 4):
//   1. each lane of the row decodes CH/LPR records of the chunk: the
//      record, its anchor, its sample's G weights. The loads of one lane are
//      independent of every other lane's, so the chunk costs one round trip
//      of record loads and one of weight loads, and each record is decoded
//      once instead of by every lane of the row. The results go to the
//      warp's shared-memory table;
//   2. the lanes walk the chunk four records at a time: shared-memory reads
//      of the table, the four anchors' grad_out rows (independent loads that
//      issue together), then acc += (w * w_i) * grad_out and the lane's part
//      of d = feat_row . grad_out, summed over a group's lanes by shuffles;
//      the lane left with a record's sum stores it to dpix at the record's
//      key, next to the sample's other corners.
// Slots past a row's last record hold anchor 0 and weight 0: their loads
// are of a valid row and their products add zero, so the walk needs no
// predicates.
// V8: grad_out, grad_feat (and fp32 features) are 32-byte aligned, so each
// lane moves its 8 channels with one 256-bit access.
template <typename T, int LPR, int LPG, bool FUSED, bool V8>
__device__ __forceinline__ void pull_rows(const PullArgs &args, int64_t warp_id, unsigned char *pull_smem)
{
    constexpr int RPW = 32 / LPR;
    constexpr int CH = LPR >= 4 ? LPR : 4;
    constexpr int RPL = CH / LPR;  // records each lane decodes per chunk
    constexpr int SLOTS = RPW * CH;
    constexpr int ESZ = sizeof(T) == 4 ? 4 : 2;
    const Problem &pb = args.pb;
    const BinArgs &w = args.w;
    const int G = pb.G;
    const int lane = threadIdx.x & 31;
    const int q = lane / LPR, sub = lane % LPR;
    const int g = sub / LPG, gsub = sub % LPG;
    int2 *meta = reinterpret_cast<int2 *>(pull_smem + (threadIdx.x >> 5) * pull_smem_per_warp(SLOTS, G));
    int *ksm = reinterpret_cast<int *>(meta + SLOTS);
    float *wsm = reinterpret_cast<float *>(ksm + SLOTS);
    constexpr int WP = pull_wpitch(SLOTS);
    // Rows are taken from the end: each camera's block of rows ends with its
    // coarsest maps, whose rows hold the most records (a sample lands in
    // every scale, and a coarse map has few pixels). Taken last to first,
    // the long rows start early and the launch ends on short rows, not on a
    // tail of long ones (2 % of the backward at the 6-camera training shape).
    // Consecutive rows go to the warps of one CTA: neighbouring pixels share
    // samples, whose grad_out rows the CTA's warps then find in L1 (a
    // footprint covers 2x2 pixels). Walking 2x2 pixel blocks one pixel after
    // another in one warp instead measured slower (L1 hit rate 21 % against
    // 38 %): the reuse comes from warps running side by side.
    int64_t R = args.row_end - 1 - (warp_id * RPW + q);
    bool active = R >= args.row_begin;
    if (args.mode == kRowsListed) {
        // Entry warp_id of the leftover-row list (one row per warp: RPW = 1).
        const int64_t cnt = min(static_cast<int64_t>(*reinterpret_cast<volatile int32_t *>(w.left_count)),
                                w.rows_total);
        active = warp_id < cnt;
        R = active ? w.left[warp_id] : 0;
    }
    if (args.mode == kRowsCoarse && active) {
        // Unit R is row ul of the ungrouped maps of batch item bu.
        const int64_t bu = R / args.units_per_b;
        const int64_t ul = R - bu * args.units_per_b;
        int64_t rr = 0;
        for (int i = 0; i < pb.nmaps; ++i) {
            const MapInfo mm = pb.maps[i];
            if (!((args.group_maps >> i) & 1) && ul >= mm.pad && ul < mm.pad + static_cast<int64_t>(mm.H) * mm.W)
                rr = mm.start + (ul - mm.pad);
        }
        R = bu * pb.rows + rr;
    }
    const int b = active ? static_cast<int>(pb.div_rows.div(static_cast<uint32_t>(R))) : 0;
    const int jb = active ? (R > 0 ? w.row_off[R - 1] : 0) : 0;
    const int je = active ? w.row_off[R] : 0;
    const int n = je - jb;
    const float *go_b = args.grad_out + static_cast<int64_t>(b) * pb.A * pb.C + sub * 8;
    const int abase = b * pb.A;
    const int row_slot = q * CH;

    float v[8];
    if (active) {
        load_feat8<T, V8>(static_cast<const char *>(pb.feat) + (R * pb.C + sub * 8) * ESZ, v);
    } else {
#pragma unroll
        for (int m = 0; m < 8; ++m) v[m] = 0.f;
    }
    float2 v2[4], acc2[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        v2[m] = make_float2(v[2 * m], v[2 * m + 1]);
        acc2[m] = make_float2(0.f, 0.f);
    }

    int nmax = n;
    if constexpr (RPW > 1) {
#pragma unroll
        for (int o = 16; o >= LPR; o >>= 1) nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
    }

    // With one record per lane per chunk (RPL = 1), the next chunk's record
    // is loaded one chunk ahead, so a chunk's decode waits only for weights.
    int2 rnext = make_int2(0, 0);
    if constexpr (RPL == 1) {
        if (sub < n && DA_CHECK(pb.dbg_err, jb + sub, w.ncap, kBoundsRecord)) rnext = ldg_record_stream(&w.rec[jb + sub]);
    }
    for (int k0 = 0; k0 < nmax; k0 += CH) {
        // 1. decode: lane sub takes records k0 + sub + LPR*j of its row.
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
            const int c = sub + LPR * j;
            bool valid = k0 + c < n && DA_CHECK(pb.dbg_err, jb + k0 + c, w.ncap, kBoundsRecord);
            int2 r;
            if constexpr (RPL == 1) {
                r = valid ? rnext : make_int2(0, 0);
                const int kn = k0 + CH + c;
                rnext = make_int2(0, 0);
                if (kn < n && DA_CHECK(pb.dbg_err, jb + kn, w.ncap, kBoundsRecord)) rnext = ldg_record_stream(&w.rec[jb + kn]);
            } else {
                r = valid ? ldg_record_stream(&w.rec[jb + k0 + c]) : make_int2(0, 0);
            }
            const int sid = r.x >> 2;
            int a = valid ? static_cast<int>(pb.div_PKS.div(sid)) - abase : 0;
            // A bounds-checking build drops a record whose anchor or sample
            // is outside the problem (its weight 0, anchor 0).
            if (valid && !(DA_CHECK(pb.dbg_err, a, pb.A, kBoundsAnchor) &&
                           DA_CHECK(pb.dbg_err, sid, w.nsid, kBoundsSample))) {
                valid = false;
                a = 0;
            }
            meta[row_slot + c] = make_int2(a, valid ? r.y : 0);
            ksm[row_slot + c] = r.x;
            if constexpr (!FUSED) {
                const float *wp = pb.weights + static_cast<int64_t>(sid) * G;
                if (args.weights_v8) {
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
                    if (valid) ldg_v8_stream(wp, x, y);
                    const float wv[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int gg = 0; gg < 8; ++gg) wsm[gg * WP + row_slot + c] = wv[gg];
                } else {
                    for (int gg = 0; gg < G; ++gg) wsm[gg * WP + row_slot + c] = valid ? __ldg(wp + gg) : 0.f;
                }
            } else {
                wsm[row_slot + c] = valid ? bin_weight<true>(pb, sid, 0) : 0.f;
            }
        }
        __syncwarp();
        // 2. walk the chunk four records at a time.
        const int nb = min(CH, nmax - k0);
        const float *wrow = wsm + g * WP + row_slot;
        for (int u0 = 0; u0 < nb; u0 += 4) {
            const int4 m01 = *reinterpret_cast<const int4 *>(meta + row_slot + u0);
            const int4 m23 = *reinterpret_cast<const int4 *>(meta + row_slot + u0 + 2);
            const float4 w4 = *reinterpret_cast<const float4 *>(wrow + u0);
            const int an[4] = {m01.x, m01.z, m23.x, m23.z};
            const float tw[4] = {__int_as_float(m01.y) * w4.x, __int_as_float(m01.w) * w4.y,
                                 __int_as_float(m23.y) * w4.z, __int_as_float(m23.w) * w4.w};
            float4 x[4], y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if constexpr (V8) ldg_v8_keep(go_b + static_cast<int64_t>(an[u]) * pb.C, x[u], y[u]);
                else ldg_f32x8<V8>(go_b + static_cast<int64_t>(an[u]) * pb.C, x[u], y[u]);
            }
            float d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) d[u] = record_fma2(v2, x[u], y[u], tw[u], acc2);
            const int4 k4 = *reinterpret_cast<const int4 *>(ksm + row_slot + u0);
            const int keys[4] = {k4.x, k4.y, k4.z, k4.w};
            group_sum_store<LPG>(d, gsub, n - k0 - u0, w.dpix + g, keys, G, pb.dbg_err, w.ncap);
        }
        __syncwarp();
    }

    if (active) {
        const float4 a0 = make_float4(acc2[0].x, acc2[0].y, acc2[1].x, acc2[1].y);
        const float4 a1 = make_float4(acc2[2].x, acc2[2].y, acc2[3].x, acc2[3].y);
        float *gf = args.grad_feat + R * pb.C + sub * 8;
        if constexpr (V8) {
            stg_v8(gf, a0, a1);
        } else {
            reinterpret_cast<float4 *>(gf)[0] = a0;
            reinterpret_cast<float4 *>(gf)[1] = a1;
        }
    }
}

template <typename T, int LPR, int LPG, bool FUSED, bool V8>
__global__ void __launch_bounds__(kPullThreads, 8) pull_kernel(const PullArgs args)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char pull_smem[];
    pull_rows<T, LPR, LPG, FUSED, V8>(args, (static_cast<int64_t>(blockIdx.x) * kPullThreads + threadIdx.x) >> 5,
                                      pull_smem);
}

// ------------------------------------------------------------ row groups
//
// A feature row of a fine map holds few records (at the 6-camera training
// shape, 4 on the 64x176 maps): a warp that pulls one such row spends most of
// its time on the chain of dependent loads that precedes its walk (row
// offsets, then records, then weights and grad_out rows). There a warp takes
// a run of consecutive pixels of one map row instead, whose records are one
// contiguous run of the record array: it walks that run as one stream, in
// chunks and batches as the per-row pull does, and switches rows where the
// row offsets say. The four warps of a CTA take the same columns of four
// consecutive map rows, so vertically adjacent pixels, which share the
// samples whose footprints straddle them, are walked side by side and their
// grad_out rows meet in L1.

constexpr int kGroupMaxRows = 16;    // pixels per warp: the warp's lanes hold their row offsets
constexpr int kRunMaxRecs = 256;     // records a run walks before it hands rows on

__host__ __device__ inline size_t group_smem_per_warp(int G) { return pull_smem_per_warp(32, G); }

// One CTA per block of 4 map rows x RW columns of a grouped map, C = 256
// (lane l: channels 8l..8l+7 of all groups); warp w takes the RW (or fewer,
// at the right edge) pixels of map row 4*by + w. Blocks are taken from the
// end, as rows are in pull_kernel.
//   - lanes 0..nr load the begin offsets of the warp's rows and of the next
//     row, so the record run is [J0, J1) and row k ends where row k+1 begins;
//     the warp keeps its first rows up to kRunMaxRecs records and lists the
//     rest for pull_listed_kernel;
//   - the first row's features are loaded, and the next row's one row ahead
//     (with an L2 prefetch four rows ahead);
//   - the run is decoded 32 records at a time into the warp's table (as in
//     pull_kernel) and walked four at a time; before a record is applied,
//     every row that ends at or before it is finished: its grad_feat is
//     stored and the next row's features take its place;
//   - rows after the last record are stored as zeros.
// In pull_hybrid_kernel: 80 registers, 6 CTAs (24 warps) per SM. Pull +
// epilogue at the training shape: 589 us; 605 us with 5 CTAs per SM (94
// registers); with one warp per
// 16 pixels of a map row and the CTA's warps on consecutive runs of one map
// row, 615 us (feature rows in registers) or 608 us (through a shared-memory
// ring of cp.async copies).
template <typename T, int LPG, bool V8>
__device__ __forceinline__ void pull_groups(const PullArgs &args, int64_t block, unsigned char *pull_smem)
{
    constexpr int CH = 32;
    constexpr int WP = pull_wpitch(CH);
    const Problem &pb = args.pb;
    const BinArgs &w = args.w;
    const int G = pb.G;
    const int lane = threadIdx.x & 31;
    const int g = lane / LPG, gsub = lane % LPG;
    unsigned char *wbase = pull_smem + (threadIdx.x >> 5) * group_smem_per_warp(G);
    int2 *meta = reinterpret_cast<int2 *>(wbase);
    int *ksm = reinterpret_cast<int *>(meta + CH);
    float *wsm = reinterpret_cast<float *>(ksm + CH);

    // CTA unit: a block of 4 map rows x RW columns; warp w takes map row
    // 4*by + w, so the CTA's warps walk vertically adjacent pixels side by side.
    const int64_t cid = args.row_end - 1 - block;
    if (cid < args.row_begin) return;
    const int b = static_cast<int>(cid / args.units_per_b);
    const int64_t gl = cid - static_cast<int64_t>(b) * args.units_per_b;
    int mi = 0;
    for (int i = 0; i < pb.nmaps; ++i) {
        const MapInfo mm = pb.maps[i];
        const int rl = args.rw_log[i];
        const int64_t nbx = (mm.W + (1 << rl) - 1) >> rl;
        const int64_t ng = ((mm.H + 3) / 4) * nbx;
        if (((args.group_maps >> i) & 1) && gl >= mm.pad && gl < mm.pad + ng) mi = i;
    }
    const MapInfo m = pb.maps[mi];
    const int rl = args.rw_log[mi];
    const int nbx = (m.W + (1 << rl) - 1) >> rl;
    const int ul = static_cast<int>(gl - m.pad);
    const int by = ul / nbx, bx = ul - by * nbx;
    const int my = 4 * by + (threadIdx.x >> 5);
    if (my >= m.H) return;  // the whole warp
    const int first = my * m.W + (bx << rl);
    const int nr = min(1 << rl, m.W - (bx << rl));
    const int64_t R0 = static_cast<int64_t>(b) * pb.rows + m.start + first;
    int rb = 0;  // lane k <= nr: where row R0 + k begins
    if (lane <= nr) rb = R0 + lane > 0 ? w.row_off[R0 + lane - 1] : 0;
    const int J0 = __shfl_sync(0xffffffffu, rb, 0);
    // The run keeps its first rows up to kRunMaxRecs records (row offsets
    // grow with k, so the rows that fit are a prefix); the rest go to the
    // leftover list, to be pulled one warp per row. Uniform locations never
    // get there; clustered ones (projected key points) do.
    const int kc = 31 - __clz(__ballot_sync(0xffffffffu, lane <= nr && rb - J0 <= kRunMaxRecs));
    if (kc < nr) {
        int base = 0;
        if (lane == 0) base = atomicAdd(w.left_count, nr - kc);
        base = __shfl_sync(0xffffffffu, base, 0);
        if (lane >= kc && lane < nr && DA_CHECK(pb.dbg_err, base + lane - kc, w.rows_total, kBoundsRowCount))
            w.left[base + lane - kc] = static_cast<int32_t>(R0 + lane);
        if (kc == 0) return;
    }
    const int nrw = kc;  // rows walked here
    const int J1 = __shfl_sync(0xffffffffu, rb, nrw);
    const float *go_b = args.grad_out + static_cast<int64_t>(b) * pb.A * pb.C + lane * 8;
    const int abase = b * pb.A;

    constexpr int ESZ = sizeof(T) == 4 ? 4 : 2;
    auto feat_ptr = [&](int k) {
        return static_cast<const char *>(pb.feat) + ((R0 + k) * pb.C + lane * 8) * ESZ;
    };
    // Lanes 0..(row bytes / 128 - 1) each prefetch one 128-byte line of row k.
    auto l2_prefetch = [&](int k) {
        if (k < nrw && lane * 128 < 256 * ESZ) {
            const char *p = static_cast<const char *>(pb.feat) + (R0 + k) * pb.C * ESZ + lane * 128;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    };
    int cur = 0;
    int cur_end = __shfl_sync(0xffffffffu, rb, 1);
    float2 v2[4], acc2[4];
    float vn[8];
    {
        float v[8];
        load_feat8<T, V8>(feat_ptr(0), v);
#pragma unroll
        for (int c = 0; c < 4; ++c) v2[c] = make_float2(v[2 * c], v[2 * c + 1]);
    }
    if (nrw > 1) load_feat8<T, V8>(feat_ptr(1), vn);
    else {
#pragma unroll
        for (int c = 0; c < 8; ++c) vn[c] = 0.f;
    }
    for (int k = 2; k < 5; ++k) l2_prefetch(k);
    auto next_feats = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) v2[c] = make_float2(vn[2 * c], vn[2 * c + 1]);
        if (cur + 1 < nrw) load_feat8<T, V8>(feat_ptr(cur + 1), vn);
        l2_prefetch(cur + 4);
    };
    auto store_row = [&](int k) {
        const float4 a0 = make_float4(acc2[0].x, acc2[0].y, acc2[1].x, acc2[1].y);
        const float4 a1 = make_float4(acc2[2].x, acc2[2].y, acc2[3].x, acc2[3].y);
        float *gf = args.grad_feat + (R0 + k) * pb.C + lane * 8;
        if constexpr (V8) {
            stg_v8(gf, a0, a1);
        } else {
            reinterpret_cast<float4 *>(gf)[0] = a0;
            reinterpret_cast<float4 *>(gf)[1] = a1;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) acc2[c] = make_float2(0.f, 0.f);
    };
#pragma unroll
    for (int c = 0; c < 4; ++c) acc2[c] = make_float2(0.f, 0.f);

    // Each lane's record of the next round is loaded one round ahead, so a
    // round's decode waits only for the weights.
    int2 rnext = make_int2(0, 0);
    if (J0 + lane < J1 && DA_CHECK(pb.dbg_err, J0 + lane, w.ncap, kBoundsRecord))
        rnext = ldg_record_stream(&w.rec[J0 + lane]);
    for (int k0 = J0; k0 < J1; k0 += CH) {
        // 1. decode: lane c takes record k0 + c of the run.
        {
            const int c = lane;
            bool valid = k0 + c < J1 && DA_CHECK(pb.dbg_err, k0 + c, w.ncap, kBoundsRecord);
            const int2 r = valid ? rnext : make_int2(0, 0);
            const int kn = k0 + CH + c;
            rnext = make_int2(0, 0);
            if (kn < J1 && DA_CHECK(pb.dbg_err, kn, w.ncap, kBoundsRecord)) rnext = ldg_record_stream(&w.rec[kn]);
            const int sid = r.x >> 2;
            int a = valid ? static_cast<int>(pb.div_PKS.div(sid)) - abase : 0;
            if (valid && !(DA_CHECK(pb.dbg_err, a, pb.A, kBoundsAnchor) &&
                           DA_CHECK(pb.dbg_err, sid, w.nsid, kBoundsSample))) {
                valid = false;
                a = 0;
            }
            meta[c] = make_int2(a, valid ? r.y : 0);
            ksm[c] = r.x;
            const float *wp = pb.weights + static_cast<int64_t>(sid) * G;
            if (args.weights_v8) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
                if (valid) ldg_v8_stream(wp, x, y);
                const float wv[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
                for (int gg = 0; gg < 8; ++gg) wsm[gg * WP + c] = wv[gg];
            } else {
                for (int gg = 0; gg < G; ++gg) wsm[gg * WP + c] = valid ? __ldg(wp + gg) : 0.f;
            }
        }
        __syncwarp();
        // 2. walk four records at a time, finishing rows as their ends pass.
        const int nb = min(CH, J1 - k0);
        const float *wrow = wsm + g * WP;
        for (int u0 = 0; u0 < nb; u0 += 4) {
            const int4 m01 = *reinterpret_cast<const int4 *>(meta + u0);
            const int4 m23 = *reinterpret_cast<const int4 *>(meta + u0 + 2);
            const float4 w4 = *reinterpret_cast<const float4 *>(wrow + u0);
            const int an[4] = {m01.x, m01.z, m23.x, m23.z};
            const float tw[4] = {__int_as_float(m01.y) * w4.x, __int_as_float(m01.w) * w4.y,
                                 __int_as_float(m23.y) * w4.z, __int_as_float(m23.w) * w4.w};
            float4 x[4], y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if constexpr (V8) ldg_v8_keep(go_b + static_cast<int64_t>(an[u]) * pb.C, x[u], y[u]);
                else ldg_f32x8<V8>(go_b + static_cast<int64_t>(an[u]) * pb.C, x[u], y[u]);
            }
            float d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                d[u] = 0.f;
                if (u0 + u < nb) {
                    while (k0 + u0 + u >= cur_end) {  // the same for every lane
                        store_row(cur);
                        ++cur;
                        cur_end = __shfl_sync(0xffffffffu, rb, cur + 1);
                        next_feats();
                    }
                    d[u] = record_fma2(v2, x[u], y[u], tw[u], acc2);
                }
            }
            const int4 k4 = *reinterpret_cast<const int4 *>(ksm + u0);
            const int keys[4] = {k4.x, k4.y, k4.z, k4.w};
            group_sum_store<LPG>(d, gsub, nb - u0, w.dpix + g, keys, G, pb.dbg_err, w.ncap);
        }
        __syncwarp();
    }
    // The row being summed, then the rows with no records left.
    store_row(cur);
    for (int k = cur + 1; k < nrw; ++k) store_row(k);
}

// Both kinds of unit in one launch: CTAs below n_coarse take coarse rows
// (one warp per row, longest first), the rest take blocks of grouped maps.
// One launch lets the blocks fill the SMs while the coarse maps' longest
// rows are still being walked; as two launches, each ended on its own tail
// (large_bf16, whose 10x25 maps' rows hold ~370 records: 399 us per step
// against 358 us with one warp per row everywhere).
template <typename T, int LPG, bool V8>
__global__ void __launch_bounds__(kPullThreads, 6)
    pull_hybrid_kernel(const PullArgs coarse, const PullArgs grouped, int64_t n_coarse)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char pull_smem[];
    if (static_cast<int64_t>(blockIdx.x) < n_coarse)
        pull_rows<T, 32, LPG, false, V8>(coarse, (static_cast<int64_t>(blockIdx.x) * kPullThreads + threadIdx.x) >> 5,
                                         pull_smem);
    else
        pull_groups<T, LPG, V8>(grouped, static_cast<int64_t>(blockIdx.x) - n_coarse, pull_smem);
}

// The leftover rows of the runs: one warp per listed row, a grid of at most
// eight CTAs per SM looping over the list (its length is known only on the
// device). Launched after the hybrid kernel; with no leftovers it only reads
// the count.
template <typename T, int LPG, bool V8>
__global__ void __launch_bounds__(kPullThreads, 8) pull_listed_kernel(const PullArgs args)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char pull_smem[];
    const int64_t cnt = min(static_cast<int64_t>(*reinterpret_cast<volatile int32_t *>(args.w.left_count)),
                            args.w.rows_total);
    const int64_t nw = static_cast<int64_t>(gridDim.x) * (kPullThreads / 32);
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * kPullThreads + threadIdx.x) >> 5; i < cnt; i += nw)
        pull_rows<T, 32, LPG, false, V8>(args, i, pull_smem);
}

// Row groups serve the standard layout with C = 256 when the maps cover a
// batch item's feature rows exactly (every row a pixel of one map). A map
// whose rows would hold fewer than kGroupMaxRho records each on average
// (4*A*P samples' corners spread over H*W rows) is grouped, with about
// kGroupTargetRecs records per warp (runs of a power of two of pixels, 2 to
// kGroupMaxRows). Pull + epilogue at the 6-camera training shape (runs of 16
// pixels on the 64x176 maps, 8 on the 32x88 maps): 589 us against 636 us
// with one warp per row. With the earlier one-warp-per-run layout, 128
// records per run measured as 64 (610, 612 us), 32 slower (659 us), 256
// slower (629 us).
constexpr double kGroupMaxRho = 24.0;
constexpr double kGroupTargetRecs = 128.0;

bool pull_plan(Problem &pb, PullArgs &coarse, PullArgs &grouped)
{
    if (pb.layout != kLayoutStd || pb.C != 256 || pb.nmaps <= 0 || pb.rows <= 0 || pb.A <= 0 || pb.P <= 0)
        return false;
    int order[DA_MAX_MAPS];
    for (int i = 0; i < pb.nmaps; ++i) order[i] = i;
    std::sort(order, order + pb.nmaps, [&](int x, int y) { return pb.maps[x].start < pb.maps[y].start; });
    int64_t end = 0;
    for (int i = 0; i < pb.nmaps; ++i) {
        const MapInfo &m = pb.maps[order[i]];
        if (m.start != end) return false;
        end += static_cast<int64_t>(m.H) * m.W;
    }
    if (end != pb.rows) return false;
    uint64_t gm = 0;
    uint8_t rwl[DA_MAX_MAPS] = {};
    int64_t rows = 0, groups = 0;
    for (int i = 0; i < pb.nmaps; ++i) {
        const MapInfo &m = pb.maps[i];
        const int64_t px = static_cast<int64_t>(m.H) * m.W;
        const double rho = 4.0 * pb.A * pb.P / static_cast<double>(px);
        if (rho < kGroupMaxRho) {
            int l = static_cast<int>(std::lround(std::log2(kGroupTargetRecs / rho)));
            l = std::min(std::max(l, 1), 4);  // 2..kGroupMaxRows pixels
            rwl[i] = static_cast<uint8_t>(l);
            gm |= 1ull << i;
            // Units of a grouped map: blocks of 4 map rows x 2^l columns.
            pb.maps[i].pad = static_cast<int32_t>(groups);
            groups += static_cast<int64_t>((m.H + 3) / 4) * ((m.W + (1 << l) - 1) >> l);
        } else {
            pb.maps[i].pad = static_cast<int32_t>(rows);
            rows += px;
        }
    }
    if (gm == 0) return false;
    for (PullArgs *p : {&coarse, &grouped}) {
        p->pb = pb;
        p->group_maps = gm;
        std::copy(rwl, rwl + DA_MAX_MAPS, p->rw_log);
        p->row_begin = 0;
    }
    coarse.mode = kRowsCoarse;
    coarse.units_per_b = rows;
    coarse.row_end = rows * pb.B;
    grouped.mode = kRowGroups;
    grouped.units_per_b = groups;
    grouped.row_end = groups * pb.B;
    return true;
}

template <typename T, int LPG>
cudaError_t launch_pull_hybrid(const PullArgs &coarse, const PullArgs &grouped, cudaStream_t st)
{
    const int64_t n_coarse = (coarse.row_end - coarse.row_begin + kPullThreads / 32 - 1) / (kPullThreads / 32);
    const int64_t grid = n_coarse + (grouped.row_end - grouped.row_begin);  // one CTA per block
    if (grid == 0) return cudaSuccess;
    const bool v8 = aligned(coarse.grad_out, 32) && aligned(coarse.grad_feat, 32) &&
                    (sizeof(T) != 4 || aligned(coarse.pb.feat, 32));
    PullArgs c = coarse, g = grouped;
    c.weights_v8 = g.weights_v8 = coarse.pb.G == 8 && aligned(coarse.pb.weights, 32);
    const size_t smem = group_smem_per_warp(coarse.pb.G) * (kPullThreads / 32);
    const dim3 gd(static_cast<unsigned>(grid));
    const dim3 blk(kPullThreads);
    cudaError_t e = v8 ? launch_pdl(pull_hybrid_kernel<T, LPG, true>, gd, blk, smem, st, c, g, n_coarse)
                       : launch_pdl(pull_hybrid_kernel<T, LPG, false>, gd, blk, smem, st, c, g, n_coarse);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t rows_grouped = coarse.pb.B * coarse.pb.rows - (coarse.row_end - coarse.row_begin);
    const int64_t lgrid =
        std::max<int64_t>(1, std::min<int64_t>((rows_grouped + 3) / 4, static_cast<int64_t>(sms) * 8));
    PullArgs l = c;
    l.mode = kRowsListed;
    const size_t lsmem = pull_smem_per_warp(32, coarse.pb.G) * (kPullThreads / 32);
    const dim3 lg(static_cast<unsigned>(lgrid));
    return v8 ? launch_pdl(pull_listed_kernel<T, LPG, true>, lg, blk, lsmem, st, l)
              : launch_pdl(pull_listed_kernel<T, LPG, false>, lg, blk, lsmem, st, l);
}

template <typename T>
cudaError_t dispatch_hybrid(const PullArgs &coarse, const PullArgs &grouped, cudaStream_t st)
{
    switch (coarse.pb.D / 8) {
        case 1: return launch_pull_hybrid<T, 1>(coarse, grouped, st);
        case 2: return launch_pull_hybrid<T, 2>(coarse, grouped, st);
        case 4: return launch_pull_hybrid<T, 4>(coarse, grouped, st);
        case 8: return launch_pull_hybrid<T, 8>(coarse, grouped, st);
        case 16: return launch_pull_hybrid<T, 16>(coarse, grouped, st);
        case 32: return launch_pull_hybrid<T, 32>(coarse, grouped, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int LPR, int LPG>
cudaError_t launch_pull_kernel(const PullArgs &pa, cudaStream_t st)
{
    if constexpr (LPG > LPR) {
        return cudaErrorInvalidValue;
    } else {
        constexpr int RPW = 32 / LPR;
        const int64_t warps = (pa.row_end - pa.row_begin + RPW - 1) / RPW;
        const int64_t grid = (warps + kPullThreads / 32 - 1) / (kPullThreads / 32);
        if (grid == 0) return cudaSuccess;
        // 256-bit accesses need 32-byte alignment of every row segment: rows
        // are C*4 >= 32 bytes of fp32 (grad_out, grad_feat) or C*elem bytes of
        // features (a 16-byte load per lane when 16-bit), so the base
        // addresses decide.
        const bool v8 = aligned(pa.grad_out, 32) && aligned(pa.grad_feat, 32) &&
                        (sizeof(T) != 4 || aligned(pa.pb.feat, 32));
        PullArgs p = pa;
        p.weights_v8 = pa.pb.layout != kLayoutFused && pa.pb.G == 8 && aligned(pa.pb.weights, 32);
        constexpr int CH = LPR >= 4 ? LPR : 4;
        const size_t smem = pull_smem_per_warp(RPW * CH, pa.pb.G) * (kPullThreads / 32);
        const dim3 g(static_cast<unsigned>(grid));
        const dim3 blk(kPullThreads);
        if (pa.pb.layout == kLayoutFused)
            return v8 ? launch_pdl(pull_kernel<T, LPR, LPG, true, true>, g, blk, smem, st, p)
                      : launch_pdl(pull_kernel<T, LPR, LPG, true, false>, g, blk, smem, st, p);
        return v8 ? launch_pdl(pull_kernel<T, LPR, LPG, false, true>, g, blk, smem, st, p)
                  : launch_pdl(pull_kernel<T, LPR, LPG, false, false>, g, blk, smem, st, p);
    }
}

template <typename T, int LPR>
cudaError_t dispatch_lpg(const PullArgs &pa, cudaStream_t st)
{
    switch (pa.pb.D / 8) {
        case 1: return launch_pull_kernel<T, LPR, 1>(pa, st);
        case 2: return launch_pull_kernel<T, LPR, 2>(pa, st);
        case 4: return launch_pull_kernel<T, LPR, 4>(pa, st);
        case 8: return launch_pull_kernel<T, LPR, 8>(pa, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dispatch_pull(const PullArgs &pa, cudaStream_t st)
{
    switch (pa.pb.C / 8) {
        case 1: return dispatch_lpg<T, 1>(pa, st);
        case 2: return dispatch_lpg<T, 2>(pa, st);
        case 4: return dispatch_lpg<T, 4>(pa, st);
        case 8: return dispatch_lpg<T, 8>(pa, st);
        case 16: return dispatch_lpg<T, 16>(pa, st);
        case 32: return dispatch_lpg<T, 32>(pa, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_pull(const BwdArgs &a, const BinArgs &w, int feat_dtype, cudaStream_t st)
{
    PullArgs pa{};
    pa.pb = a.pb;
    pa.grad_out = a.grad_out;
    pa.grad_feat = a.grad_feat;
    pa.w = w;
    pa.row_begin = 0;
    pa.row_end = w.rows_total;
    pa.mode = kRowsAll;
    Problem pb = a.pb;
    PullArgs grouped = pa;
    if (pull_plan(pb, pa, grouped)) {
        return feat_dtype == DA_BF16  ? dispatch_hybrid<Bf16Tag>(pa, grouped, st)
               : feat_dtype == DA_F16 ? dispatch_hybrid<F16Tag>(pa, grouped, st)
                                      : dispatch_hybrid<float>(pa, grouped, st);
    }
    return feat_dtype == DA_BF16  ? dispatch_pull<Bf16Tag>(pa, st)
           : feat_dtype == DA_F16 ? dispatch_pull<F16Tag>(pa, st)
                                  : dispatch_pull<float>(pa, st);
}

}  // namespace da
