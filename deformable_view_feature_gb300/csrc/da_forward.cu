// Forward sampling kernel of the deformable-aggregation operator.
//
// out[b,a,c] = sum_{p,k,s} weights[b,a,p,k,s,g] * bilinear(map (b,k,s), loc[b,a,p,k], c)
// (page "Inside Sparse4D's CUDA core", §3.2 for the sample and §5.1 for the
// dimensions summed over). In the fused layout every group has its own
// location and both come from one tensor: the DCNv4 form
// y_g = sum_k m_gk x_g(p_gk) of the DCNv4 page ("Defining the problem"),
// whose offsets and weights one linear layer produces together ("Solving the
// problem: 1"). In the projected layout the kernel itself projects the
// anchors' key points into the cameras (the Sparse4D page, §1 and §6) and
// takes the softmax of the weight logits over each task's P*K*S samples, so
// no location or weight tensor is read.
//
// Work decomposition (the page's kernel uses one thread per sample; here a
// warp owns one (b*A+a, g) task and its P*K*S samples):
//   * A CTA of 8 warps owns `anchors_per_cta` whole anchors: all their groups.
//     Where a group's slice of a feature row is at most half a 128-byte line
//     (bf16 or fp16 with D = 32), a warp takes two neighbouring groups of an
//     anchor and a CTA twice the anchors, so every corner read is one whole
//     line (the 6-camera bf16 forward: 114 -> 106 us).
//   * Footprints: 32 samples at a time, one per lane. Each lane writes its
//     sample's four {row, weight * corner weight} pairs to a per-warp,
//     corner-major table in shared memory.
//   * Gather: the D channels of one corner row are D*sizeof(T) bytes, i.e.
//     CH 16-byte chunks. Lane l reads chunk l % CH of corner (l / CH) % 4 for
//     the samples of slot l / (4*CH). So one warp-wide 16-byte load reads the
//     four corner rows of 8/CH samples, every row as one coalesced segment
//     (the vectorised channel-last access of the DCNv4 page, "Solving the
//     problem: 2. let the GPU move less data"). Each lane walks U consecutive
//     samples per step, so U loads are in flight per lane. Their table
//     entries arrive in U/2 16-byte shared loads.
//   * Each lane accumulates its chunk in fp32 registers. At the end, shuffles
//     sum over corners and slots, and the CH lanes of slot 0 write the group's
//     D outputs with 16-byte stores.
//   * Camera parts (standard layout, a batch item's maps of 48 MB or more,
//     K even): CTAs run in the order (batch item, camera half, anchors), each
//     over half the cameras, and add their partial sums into the zeroed out
//     with vector reductions. The CTAs resident at once cover about one batch
//     item's anchors, so only half its maps are live in L2: at the 6-camera
//     training shape the forward reads 609 MB of DRAM instead of 977 MB (the
//     compulsory bytes are 614 MB), in the same time. Two addends on an exact
//     zero give the same bits in either order, so the forward stays
//     deterministic.
#include "da_internal.cuh"

// Samples a lane walks per step (loads in flight per lane), at most 32 per
// warp-wide step.
#ifndef DA_FWD_UNROLL
#define DA_FWD_UNROLL 16
#endif

namespace da {
namespace {

// SPLIT: the camera-part decomposition (FwdArgs::parts == 2), standard layout.
// GPT: groups per task. A group's slice of a feature row is CH 16-byte
// chunks; when that is at most half a 128-byte line (bf16 or fp16 with
// D = 32, fp32 with D = 16), GPT = 2 gives one warp two neighbouring groups
// of an anchor (standard layout: the groups share the sample locations). Each
// corner read is then one whole line from one warp, not two half-line
// requests from two warps.
template <typename T, int CH, bool FUSED, bool SPLIT, int GPT>
__global__ void __launch_bounds__(kThreads) fwd_kernel(const FwdArgs args)
{
    static_assert(!(SPLIT && FUSED), "camera parts serve the standard layout");
    static_assert(GPT == 1 || (GPT == 2 && !FUSED && CH <= 4), "paired groups share locations");
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;   // channels per 16-byte chunk
    constexpr int ESZ = 16 / VEC;   // bytes per feature element
    constexpr int TCH = CH * GPT;   // 16-byte chunks of one task's corner row
    constexpr int SPP = 8 / TCH;    // samples per warp-wide load
    // Samples per lane per step; a warp-wide step covers U * SPP <= 32.
    constexpr int U = DA_FWD_UNROLL * SPP <= 32 ? DA_FWD_UNROLL : 32 / SPP;
    // The steps of U*SPP samples must tile the 32 table entries exactly.
    static_assert(U % 2 == 0 && 32 % (U * SPP) == 0, "unroll must divide the 32-sample table");
    const Problem &pb = args.pb;

    __shared__ __align__(16) int2 tab[kWarps][4][kTabPitch];
    // GPT = 2: weight * corner weight of the task's second group.
    __shared__ __align__(16) float tab2[GPT > 1 ? kWarps : 1][4][kTabPitch];
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane % TCH;
    const int corner = (lane / TCH) & 3;
    const int slot = lane / (4 * TCH);
    const bool second = GPT > 1 && chunk >= CH;  // the lane's chunk is in the task's second group

    int ba0, na, part = 0;
    if constexpr (SPLIT) {
        const int c = static_cast<int>(blockIdx.x);
        const int bq = static_cast<int>(args.div_cpp.div(c));  // b * parts + part
        const int ci = c - bq * args.ctas_per_part;
        const int bb = bq / args.parts;
        part = bq - bb * args.parts;
        ba0 = bb * pb.A + ci * pb.anchors_per_cta;
        na = min(pb.anchors_per_cta, pb.A - ci * pb.anchors_per_cta);
    } else {
        ba0 = static_cast<int>(blockIdx.x) * pb.anchors_per_cta;
        na = min(pb.anchors_per_cta, pb.num_ba - ba0);
    }
    // Samples of a task: all P*K*S, or the P*kpart*S of this CTA's cameras.
    const int nsamp = SPLIT ? pb.P * args.kpart * pb.S : pb.pks;
    const int ntask = na * (pb.G / GPT);
    const uint32_t row_bytes = static_cast<uint32_t>(pb.C) * ESZ;

    for (int task = warp; task < ntask; task += kWarps) {
        // Task (anchor tq, groups g .. g + GPT - 1): task * GPT = tq * G + g.
        const int tq = static_cast<int>(pb.div_G.div(task * GPT));
        const int g = task * GPT - tq * pb.G;
        const int ba = ba0 + tq;
        const int b = static_cast<int>(pb.div_A.div(ba));
        const char *base = static_cast<const char *>(pb.feat) +
                           (static_cast<int64_t>(b) * pb.rows * pb.C + static_cast<int64_t>(g) * pb.D) * ESZ +
                           chunk * 16;
        float acc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = 0.f;

        for (int j0 = 0; j0 < nsamp; j0 += 32) {
            const int n = min(32, nsamp - j0);
            {
                int row[4] = {-1, -1, -1, -1};
                float tw[4] = {0.f, 0.f, 0.f, 0.f};
                float tw2[4] = {0.f, 0.f, 0.f, 0.f};
                if (lane < n) {
                    const int j = j0 + lane;
                    int jk = static_cast<int>(pb.div_S.div(j));  // p*K + k (p*kpart + k' with parts)
                    const int s = j - jk * pb.S;
                    int k;
                    if constexpr (SPLIT) {
                        const int p = static_cast<int>(args.div_kpart.div(jk));
                        k = part * args.kpart + (jk - p * args.kpart);
                        jk = p * pb.K + k;
                    } else {
                        k = jk - static_cast<int>(pb.div_K.div(jk)) * pb.K;
                    }
                    float2 xy;
                    float w;
                    sample_xyw<FUSED>(pb, ba, g, jk, s, xy, w);
                    Footprint f;
                    footprint(xy.x, xy.y, maps_s[k * pb.S + s], f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        row[c] = f.row[c];
                        tw[c] = w * f.cw[c];
                    }
                    if constexpr (GPT > 1) {
                        const float w2 = pb.weights[((static_cast<int64_t>(ba) * pb.pk + jk) * pb.S + s) * pb.G + g + 1];
#pragma unroll
                        for (int c = 0; c < 4; ++c) tw2[c] = w2 * f.cw[c];
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) tab[warp][c][lane] = make_int2(row[c], __float_as_int(tw[c]));
                if constexpr (GPT > 1) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tab2[warp][c][lane] = tw2[c];
                }
            }
            __syncwarp();

            for (int i0 = 0; i0 < n; i0 += U * SPP) {
                const int i = i0 + U * slot;
                int r[U];
                float cw[U];
#pragma unroll
                for (int h = 0; h < U / 2; ++h) {
                    const int4 e = *reinterpret_cast<const int4 *>(&tab[warp][corner][i + 2 * h]);
                    r[2 * h] = e.x;
                    cw[2 * h] = __int_as_float(e.y);
                    r[2 * h + 1] = e.z;
                    cw[2 * h + 1] = __int_as_float(e.w);
                    if constexpr (GPT > 1) {
                        const float2 e2 = *reinterpret_cast<const float2 *>(&tab2[warp][corner][i + 2 * h]);
                        if (second) {
                            cw[2 * h] = e2.x;
                            cw[2 * h + 1] = e2.y;
                        }
                    }
                }
                uint4 raw[U];
#pragma unroll
                for (int u = 0; u < U; ++u) raw[u] = ldg16_if(feat_row_ok(pb, r[u]), row_addr(base, r[u], row_bytes));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float v[VEC];
                    Ck::unpack(raw[u], v);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] = fmaf(cw[u], v[q], acc[q]);
                }
            }
            __syncwarp();
        }

        // Sum the corner and slot partials: lanes that differ only above the
        // chunk bits hold the same channels.
#pragma unroll
        for (int m = TCH; m < 32; m <<= 1) {
#pragma unroll
            for (int q = 0; q < VEC; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], m);
        }
        if (lane < TCH) {
            float *o = args.out + static_cast<int64_t>(ba) * pb.C + static_cast<int64_t>(g) * pb.D + chunk * VEC;
            if constexpr (SPLIT) {
                // Exactly two partial sums meet on a zeroed output: 0 + x is
                // exact and x + y = y + x, so the bits do not depend on the
                // order the two parts arrive in (parts is 1 or 2).
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q)
                    red_add_v4_if(true, o + 4 * q, acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            } else {
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q)
                    reinterpret_cast<float4 *>(o)[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2],
                                                                   acc[4 * q + 3]);
            }
        }
    }
}

// Anchor of a task within its CTA.
__device__ __forceinline__ int tq_of(int task, const Problem &pb) { return static_cast<int>(pb.div_G.div(task)); }

// The projected layout's kernel: fwd_kernel's decomposition, with the
// projection and the softmax in front. (Kept apart from fwd_kernel: folding
// it into that template as a compile-time branch slowed the standard
// instance by 6 % at the 6-camera training shape.)
template <typename T, int CH>
__global__ void __launch_bounds__(kThreads) fwd_proj_kernel(const FwdArgs args)
{
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;   // channels per 16-byte chunk
    constexpr int ESZ = 16 / VEC;   // bytes per feature element
    constexpr int SPP = 8 / CH;     // samples per warp-wide load
    // Samples per lane per step; a warp-wide step covers U * SPP <= 32.
    constexpr int U = DA_FWD_UNROLL * SPP <= 32 ? DA_FWD_UNROLL : 32 / SPP;
    // The steps of U*SPP samples must tile the 32 table entries exactly.
    static_assert(U % 2 == 0 && 32 % (U * SPP) == 0, "unroll must divide the 32-sample table");
    const Problem &pb = args.pb;

    __shared__ __align__(16) int2 tab[kWarps][4][kTabPitch];
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane % CH;
    const int corner = (lane / CH) & 3;
    const int slot = lane / (4 * CH);

    const int ba0 = static_cast<int>(blockIdx.x) * pb.anchors_per_cta;
    const int na = min(pb.anchors_per_cta, pb.num_ba - ba0);
    const int ntask = na * pb.G;
    const uint32_t row_bytes = static_cast<uint32_t>(pb.C) * ESZ;
    // Dynamic shared memory: the CTA's projected locations
    // [anchors_per_cta][P*K], then per warp the softmax numerators of its
    // task's P*K*S samples.
    extern __shared__ float2 proj_s[];
    float *const ebuf = reinterpret_cast<float *>(proj_s + pb.anchors_per_cta * pb.pk) + warp * pb.pks;
    {
        // Each (anchor, point, camera) is projected once for all G groups.
        for (int i = threadIdx.x; i < na * pb.pk; i += kThreads) {
            const int tq = i / pb.pk;
            const int jk = i - tq * pb.pk;
            const int ba = ba0 + tq;
            const int p = static_cast<int>(pb.div_K.div(jk));
            const int k = jk - p * pb.K;
            const int b = static_cast<int>(pb.div_A.div(ba));
            const float2 xy = project_point(pb.keypoints + (static_cast<int64_t>(ba) * pb.P + p) * 3,
                                            pb.projection + (static_cast<int64_t>(b) * pb.K + k) * 16, pb.image_w,
                                            pb.image_h);
            proj_s[i] = xy;
            if (args.loc_out) {
                float *o = args.loc_out + (static_cast<int64_t>(ba) * pb.pk + jk) * 2;
                o[0] = xy.x;
                o[1] = xy.y;
            }
        }
    }
    __syncthreads();

    for (int task = warp; task < ntask; task += kWarps) {
        const int tq = static_cast<int>(pb.div_G.div(task));
        const int g = task - tq * pb.G;
        const int ba = ba0 + tq;
        const int b = static_cast<int>(pb.div_A.div(ba));
        const char *base = static_cast<const char *>(pb.feat) +
                           (static_cast<int64_t>(b) * pb.rows * pb.C + static_cast<int64_t>(g) * pb.D) * ESZ +
                           chunk * 16;
        float acc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = 0.f;

        // Projected layout: the softmax over the task's samples. The
        // numerators exp(z - max) go to the warp's buffer; 1/sum scales them.
        float inv_sum = 1.f;
        {
            const float *z = pb.logits + static_cast<int64_t>(ba) * pb.pks * pb.G + g;
            float m = -INFINITY;
            for (int j = lane; j < pb.pks; j += 32) m = fmaxf(m, z[static_cast<int64_t>(j) * pb.G]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float sum = 0.f;
            for (int j = lane; j < pb.pks; j += 32) {
                const float e = expf(z[static_cast<int64_t>(j) * pb.G] - m);
                ebuf[j] = e;
                sum += e;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            inv_sum = 1.f / sum;
            __syncwarp();
        }

        for (int j0 = 0; j0 < pb.pks; j0 += 32) {
            const int n = min(32, pb.pks - j0);
            {
                int row[4] = {-1, -1, -1, -1};
                float tw[4] = {0.f, 0.f, 0.f, 0.f};
                if (lane < n) {
                    const int j = j0 + lane;
                    const int jk = static_cast<int>(pb.div_S.div(j));  // p*K + k
                    const int s = j - jk * pb.S;
                    const int k = jk - static_cast<int>(pb.div_K.div(jk)) * pb.K;
                    float2 xy;
                    float w;
                    xy = proj_s[tq_of(task, pb) * pb.pk + jk];
                    w = ebuf[j] * inv_sum;
                    if (args.weights_out)
                        args.weights_out[((static_cast<int64_t>(ba) * pb.pk + jk) * pb.S + s) * pb.G + g] = w;
                    Footprint f;
                    footprint(xy.x, xy.y, maps_s[k * pb.S + s], f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        row[c] = f.row[c];
                        tw[c] = w * f.cw[c];
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) tab[warp][c][lane] = make_int2(row[c], __float_as_int(tw[c]));
            }
            __syncwarp();

            for (int i0 = 0; i0 < n; i0 += U * SPP) {
                const int i = i0 + U * slot;
                int r[U];
                float cw[U];
#pragma unroll
                for (int h = 0; h < U / 2; ++h) {
                    const int4 e = *reinterpret_cast<const int4 *>(&tab[warp][corner][i + 2 * h]);
                    r[2 * h] = e.x;
                    cw[2 * h] = __int_as_float(e.y);
                    r[2 * h + 1] = e.z;
                    cw[2 * h + 1] = __int_as_float(e.w);
                }
                uint4 raw[U];
#pragma unroll
                for (int u = 0; u < U; ++u) raw[u] = ldg16_if(feat_row_ok(pb, r[u]), row_addr(base, r[u], row_bytes));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float v[VEC];
                    Ck::unpack(raw[u], v);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] = fmaf(cw[u], v[q], acc[q]);
                }
            }
            __syncwarp();
        }

        // Sum the corner and slot partials: lanes that differ only above the
        // chunk bits hold the same channels.
#pragma unroll
        for (int m = CH; m < 32; m <<= 1) {
#pragma unroll
            for (int q = 0; q < VEC; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], m);
        }
        if (lane < CH) {
            float4 *o = reinterpret_cast<float4 *>(args.out + static_cast<int64_t>(ba) * pb.C +
                                                   static_cast<int64_t>(g) * pb.D + chunk * VEC);
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q)
                o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
    }
}

// Few samples per (anchor, group), as in the DCNv4 form (9 points, one map):
// the warp-per-task mapping above would leave most lanes idle. Here one
// lane owns one 16-byte chunk of one anchor's C channels (the DCNv4 page's
// "one thread, several channels of a group", "Solving the problem: 2"). A
// warp holds APW = 32 / cpa anchors, cpa = C*elem/16 lanes each (a power of
// two). Per round of J samples, the warp first builds the footprints of its
// APW*G*J <= 32 (anchor, group, sample) items, one per lane, into a shared
// table: {row, weight * corner weight} for the four corners. Then every lane
// walks the J entries of its own (anchor, group), four at a time, with the
// 16 corner loads of a step in flight together. (A 64-entry table, two
// items per lane, measured slower: its item decode needs runtime divisions
// in the loop.)
constexpr int kSmallItems = 32;  // table entries per warp and round

template <typename T, bool FUSED>
__global__ void __launch_bounds__(kThreads) fwd_small_kernel(const FwdArgs args, int cpa_log2, int jstep)
{
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;
    constexpr int ESZ = 16 / VEC;
    const Problem &pb = args.pb;
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    __shared__ __align__(16) int4 tab[kWarps][kSmallItems][2];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int apw = 32 >> cpa_log2;
    const int aw = lane >> cpa_log2;                 // anchor slot in the warp
    const int chunk = lane & ((1 << cpa_log2) - 1);  // 16-byte chunk of the C channels
    const int c0 = chunk * VEC;
    const int g = c0 / pb.D;
    const int64_t ba0 = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * apw;
    const int64_t ba = ba0 + aw;
    const bool live = ba < pb.num_ba;
    const int b = live ? static_cast<int>(pb.div_A.div(static_cast<uint32_t>(ba))) : 0;
    const char *base = static_cast<const char *>(pb.feat) + (static_cast<int64_t>(b) * pb.rows * pb.C + c0) * ESZ;
    const uint32_t row_bytes = static_cast<uint32_t>(pb.C) * ESZ;
    // This lane's table item in a round: (anchor slot, group, sample).
    const int it_aw = lane / (pb.G * jstep);
    const int it_g = (lane / jstep) % pb.G;
    const int it_j = lane % jstep;
    const int64_t it_ba = ba0 + it_aw;
    const bool it_live = lane < apw * pb.G * jstep && it_ba < pb.num_ba;
    const int my_item0 = (aw * pb.G + g) * jstep;

    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    for (int j0 = 0; j0 < pb.pks; j0 += jstep) {
        {
            int row[4] = {-1, -1, -1, -1};
            float tw[4] = {0.f, 0.f, 0.f, 0.f};
            const int j = j0 + it_j;
            if (it_live && j < pb.pks) {
                const int jk = static_cast<int>(pb.div_S.div(j));  // p*K + k
                const int s = j - jk * pb.S;
                const int k = jk - static_cast<int>(pb.div_K.div(jk)) * pb.K;
                float2 xy;
                float w;
                sample_xyw<FUSED>(pb, it_ba, it_g, jk, s, xy, w);
                Footprint f;
                footprint(xy.x, xy.y, maps_s[k * pb.S + s], f);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    row[c] = f.row[c];
                    tw[c] = w * f.cw[c];
                }
            }
            tab[warp][lane][0] = make_int4(row[0], __float_as_int(tw[0]), row[1], __float_as_int(tw[1]));
            tab[warp][lane][1] = make_int4(row[2], __float_as_int(tw[2]), row[3], __float_as_int(tw[3]));
        }
        __syncwarp();
        const int n = min(jstep, pb.pks - j0);
        for (int jj = 0; jj < n; jj += 4) {
            uint4 raw[4][4];
            float tw[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int4 e0 = make_int4(-1, 0, -1, 0), e1 = e0;
                if (jj + u < n) {
                    e0 = tab[warp][my_item0 + jj + u][0];
                    e1 = tab[warp][my_item0 + jj + u][1];
                }
                const int r[4] = {e0.x, e0.z, e1.x, e1.z};
                tw[u][0] = __int_as_float(e0.y);
                tw[u][1] = __int_as_float(e0.w);
                tw[u][2] = __int_as_float(e1.y);
                tw[u][3] = __int_as_float(e1.w);
#pragma unroll
                for (int c = 0; c < 4; ++c) raw[u][c] = ldg16_if(live && feat_row_ok(pb, r[c]), row_addr(base, r[c], row_bytes));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[VEC];
                    Ck::unpack(raw[u][c], v);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] = fmaf(tw[u][c], v[q], acc[q]);
                }
        }
        __syncwarp();
    }
    if (!live) return;
    float4 *o = reinterpret_cast<float4 *>(args.out + ba * pb.C + c0);
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
}

// ------------------------------------------------------------ row forward
//
// The standard layout with C = 256 (one 1 KB fp32 or 512-byte 16-bit feature
// row per pixel) and at most 8 groups: a warp owns half the scales of one
// anchor (and camera part), all its groups, and lane l channels 8l..8l+7 of
// every row. A corner of a sample is then one warp-wide 256-bit (fp32) or
// 128-bit (16-bit) load of the whole feature row, the sample's footprint is
// computed once for all G groups, and each lane applies its own group's
// weight: about 110 warp instructions per sample (all groups) instead of 8
// group-warps' 20 each, for the same bytes from L2.
//
// Two samples per step (8 row loads of 32 bytes per lane in flight), 113
// registers, 2 CTAs (16 warps) per SM. The 6-camera training-shape forward
// alone: 344 us against 385 us for the group-per-warp kernel (one sample per
// step, 59 registers and 32 warps per SM: 380 us; two at 3 CTAs per SM, 80
// registers: 349 us). With one warp per (anchor, camera part) the resident
// warps spanned about 2.7 (batch item, part) slices of the maps and read
// 1.12 GB of DRAM (70.6 % L2 hits); two warps per anchor, one per half of the
// scales, halve the anchors in flight: 0.72 GB (79.1 % L2 hits), 310 against
// 314 us under ncu. A warp per anchor gives few warps on small batches: B = 1
// at 900 anchors took 87-101 us against 86 us, so the kernel serves problems
// with at least kRowTasksMin (anchor, camera part) tasks.
constexpr int kFwdRowU = 2;
constexpr int kRowAnchors = kWarps / 2;  // anchors per CTA: two warps (scale halves) each
constexpr int kRowTasksMin = 8192;

// 32 bytes (8 floats) at a 32-byte aligned address, or zeros when `pred` is
// false (then nothing is read).
__device__ __forceinline__ void ldg32_if(bool pred, const void *p, float4 &x, float4 &y)
{
    asm("{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %9, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "mov.b32 %4, 0;\n\tmov.b32 %5, 0;\n\tmov.b32 %6, 0;\n\tmov.b32 %7, 0;\n\t"
        "@q ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t}"
        : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w), "=f"(y.x), "=f"(y.y), "=f"(y.z), "=f"(y.w)
        : "l"(p), "r"(static_cast<int>(pred)));
}

// The lane's 8 channels of one feature row (fp32: 32 bytes; 16-bit: 16
// bytes), widened; zeros when `pred` is false.
template <typename T>
__device__ __forceinline__ void row_chunk_if(bool pred, const char *p, float (&v)[8])
{
    if constexpr (sizeof(T) == 4) {
        float4 x, y;
        ldg32_if(pred, p, x, y);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    } else {
        Chunk<T>::unpack(ldg16_if(pred, p), v);
    }
}

// One CTA = 8 warps = 4 anchors of one (batch item, camera part), two warps
// each: warp 2*q + h takes anchor 4*ci + q over the part's cameras and scale
// half h (scales [0, ceil(S/2)) or [ceil(S/2), S)). For even S the two
// halves have the same number of samples, so they finish together (for odd S
// the first takes one scale more; at S = 1 the second has no samples and only
// adds zeros); a CTA's resident
// anchors (about 1,200 at 16 warps per SM) keep about one (batch item,
// camera part) slice of the maps live in L2. Per round of 32 samples each
// lane computes one sample's footprint into the warp's table (rows and corner
// weights sample-major, the G weights group-major); the lanes then walk the
// round U samples at a time: four row loads per sample (zeros, and no load,
// for a corner outside its map), and acc += (w_g * cw_i) * v_i
// with the lane's group g. The second half's sums are added to the first's
// in shared memory, and the first writes the anchor's row: a plain store, or
// with SPLIT (two camera parts) a vector reduction into the zeroed output,
// as in fwd_kernel.
template <typename T, bool SPLIT, int U>
__global__ void __launch_bounds__(kThreads, 2) fwd_row_kernel(const FwdArgs args)
{
    constexpr int ESZ = sizeof(T) == 4 ? 4 : 2;
    constexpr int WP = 36;  // weight row pitch: the 8 groups' rows 4 banks apart
    const Problem &pb = args.pb;
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    __shared__ __align__(16) int4 rows_s[kWarps][32];
    __shared__ __align__(16) float4 cw_s[kWarps][32];
    __shared__ __align__(16) float w_s[kWarps][8][WP];
    __shared__ float sum_s[kWarps][8][33];  // a warp's 8 channels per lane
    stage_maps(pb, maps_s);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = warp & 1, q = warp >> 1;
    const int s0 = half ? (pb.S + 1) / 2 : 0;           // first scale of this half
    const int sh = half ? pb.S / 2 : (pb.S + 1) / 2;    // scales in this half
    const int gl = (lane * pb.G) >> 5;  // the lane's group: channels 8*lane.. of D = 256/G
    int ba, part = 0;
    bool valid;
    if constexpr (SPLIT) {
        const int c = static_cast<int>(blockIdx.x);
        const int bq = static_cast<int>(args.div_cpp.div(c));  // b * parts + part
        const int ci = c - bq * args.ctas_per_part;
        const int bb = bq / args.parts;
        part = bq - bb * args.parts;
        const int a = ci * kRowAnchors + q;
        valid = a < pb.A;
        ba = bb * pb.A + a;
    } else {
        ba = static_cast<int>(blockIdx.x) * kRowAnchors + q;
        valid = ba < pb.num_ba;
    }
    float2 acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = make_float2(0.f, 0.f);

    // Samples of this warp: (p, camera of the part, scale of the half).
    const int nsamp = valid ? pb.P * (SPLIT ? args.kpart : pb.K) * sh : 0;
    const int b = valid ? static_cast<int>(pb.div_A.div(ba)) : 0;
    const uint32_t row_bytes = 256u * ESZ;
    const char *base = static_cast<const char *>(pb.feat) + static_cast<int64_t>(b) * pb.rows * row_bytes + lane * 8 * ESZ;
    for (int j0 = 0; j0 < nsamp; j0 += 32) {
        const int n = min(32, nsamp - j0);
        {
            int4 rr = make_int4(-1, -1, -1, -1);
            float4 cw = make_float4(0.f, 0.f, 0.f, 0.f);
            float wv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (lane < n) {
                const int j = j0 + lane;
                int jk = j / sh;  // p*K + k (p*kpart + k' with parts)
                const int s = s0 + (j - jk * sh);
                int k;
                if constexpr (SPLIT) {
                    const int p = static_cast<int>(args.div_kpart.div(jk));
                    k = part * args.kpart + (jk - p * args.kpart);
                    jk = p * pb.K + k;
                } else {
                    k = jk - static_cast<int>(pb.div_K.div(jk)) * pb.K;
                }
                const int64_t locid = static_cast<int64_t>(ba) * pb.pk + jk;
                const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + locid * 2);
                Footprint f;
                footprint(xy.x, xy.y, maps_s[k * pb.S + s], f);
                rr = make_int4(feat_row_ok(pb, f.row[0]) ? f.row[0] : -1, feat_row_ok(pb, f.row[1]) ? f.row[1] : -1,
                               feat_row_ok(pb, f.row[2]) ? f.row[2] : -1, feat_row_ok(pb, f.row[3]) ? f.row[3] : -1);
                cw = make_float4(f.cw[0], f.cw[1], f.cw[2], f.cw[3]);
                const float *wp = pb.weights + (locid * pb.S + s) * pb.G;
                for (int g = 0; g < pb.G; ++g) wv[g] = wp[g];
            }
            rows_s[warp][lane] = rr;
            cw_s[warp][lane] = cw;
#pragma unroll
            for (int g = 0; g < 8; ++g) w_s[warp][g][lane] = wv[g];
        }
        __syncwarp();
        for (int i0 = 0; i0 < n; i0 += U) {
            float v[U][4][8];
            float tw[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u;
                const bool live = U == 1 || i < n;
                const int4 rr = live ? rows_s[warp][i] : make_int4(-1, -1, -1, -1);
                const float4 cw = live ? cw_s[warp][i] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float wg = live ? w_s[warp][gl][i] : 0.f;
                const int r4[4] = {rr.x, rr.y, rr.z, rr.w};
                tw[u][0] = wg * cw.x;
                tw[u][1] = wg * cw.y;
                tw[u][2] = wg * cw.z;
                tw[u][3] = wg * cw.w;
#pragma unroll
                for (int c = 0; c < 4; ++c) row_chunk_if<T>(r4[c] >= 0, row_addr(base, r4[c], row_bytes), v[u][c]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float2 t2 = make_float2(tw[u][c], tw[u][c]);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        acc[m] = __ffma2_rn(t2, make_float2(v[u][c][2 * m], v[u][c][2 * m + 1]), acc[m]);
                }
            }
        }
        __syncwarp();
    }
    // The two halves of an anchor meet in shared memory: first + second.
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        sum_s[warp][2 * m][lane] = acc[m].x;
        sum_s[warp][2 * m + 1][lane] = acc[m].y;
    }
    __syncthreads();
    if (half != 0 || !valid) return;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        acc[m].x += sum_s[warp + 1][2 * m][lane];
        acc[m].y += sum_s[warp + 1][2 * m + 1][lane];
    }
    float *o = args.out + static_cast<int64_t>(ba) * 256 + lane * 8;
    if constexpr (SPLIT) {
        red_add_v4_if(true, o, acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        red_add_v4_if(true, o + 4, acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    } else {
        reinterpret_cast<float4 *>(o)[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        reinterpret_cast<float4 *>(o)[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
}

// Camera parts of the standard forward: 2 when a batch item's feature maps
// are large next to L2 and the cameras split evenly, else 1. A CTA then
// gathers from half the cameras, so the CTAs resident at once (about one
// batch item's anchors) keep about half a batch item's maps live in L2.
inline int forward_parts(const Problem &pb, int esz)
{
    const int64_t item_bytes = pb.rows * pb.C * esz;
    return (pb.K >= 2 && pb.K % 2 == 0 && item_bytes >= (int64_t(48) << 20)) ? 2 : 1;
}

template <typename T, int CH>
cudaError_t launch(const FwdArgs &a, cudaStream_t st)
{
    constexpr int ESZ = 16 / Chunk<T>::kVec;
    const int cpa = a.pb.C * ESZ / 16;
    if (a.pb.layout != kLayoutProj && use_small_task_kernels(a.pb, ESZ) && (cpa & (cpa - 1)) == 0) {
        int cpa_log2 = 0;
        while ((1 << cpa_log2) < cpa) ++cpa_log2;
        const int apw = 32 >> cpa_log2;
        // Samples per round: the warp's apw*G*jstep items fit one per lane.
        const int per_j = apw * a.pb.G;
        if (per_j <= kSmallItems) {
            const int jstep = kSmallItems / per_j;
            const int64_t warps = (static_cast<int64_t>(a.pb.num_ba) + apw - 1) / apw;
            const int64_t grid = (warps + kWarps - 1) / kWarps;
            if (grid == 0) return cudaSuccess;
            if (a.pb.layout == kLayoutFused)
                fwd_small_kernel<T, true><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(a, cpa_log2, jstep);
            else
                fwd_small_kernel<T, false><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(a, cpa_log2, jstep);
            return cudaGetLastError();
        }
    }
    const int64_t grid = sampling_grid(a.pb);
    if (grid == 0) return cudaSuccess;
    switch (a.pb.layout) {
        case kLayoutFused: fwd_kernel<T, CH, true, false, 1><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(a); break;
        case kLayoutProj: {
            const size_t smem = projected_smem_bytes(a.pb);
            if (smem > 48 * 1024) {
                const cudaError_t e = cudaFuncSetAttribute(fwd_proj_kernel<T, CH>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           static_cast<int>(smem));
                if (e != cudaSuccess) return e;
            }
            fwd_proj_kernel<T, CH><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
            break;
        }
        default: {
            const int row_parts = forward_parts(a.pb, ESZ);
            if (a.pb.C == 256 && a.pb.G <= 8 && (sizeof(T) != 4 || aligned(a.pb.feat, 32)) &&
                static_cast<int64_t>(a.pb.num_ba) * row_parts >= kRowTasksMin) {
                FwdArgs f = a;
                f.parts = row_parts;
                const int ctas = (a.pb.A + kRowAnchors - 1) / kRowAnchors;  // per (batch item, part)
                int64_t g = (static_cast<int64_t>(a.pb.num_ba) + kRowAnchors - 1) / kRowAnchors;
                if (f.parts > 1) {
                    f.ctas_per_part = ctas;
                    f.kpart = a.pb.K / f.parts;
                    f.div_cpp = FastDiv::make(static_cast<uint32_t>(ctas));
                    f.div_kpart = FastDiv::make(static_cast<uint32_t>(f.kpart));
                    g = static_cast<int64_t>(a.pb.B) * f.parts * ctas;
                    const cudaError_t e = cudaMemsetAsync(a.out, 0, static_cast<size_t>(a.pb.num_ba) * a.pb.C * 4, st);
                    if (e != cudaSuccess) return e;
                }
                if (g == 0) return cudaSuccess;
                const dim3 gg(static_cast<unsigned>(g));
                if (f.parts > 1) fwd_row_kernel<T, true, kFwdRowU><<<gg, kThreads, 0, st>>>(f);
                else fwd_row_kernel<T, false, kFwdRowU><<<gg, kThreads, 0, st>>>(f);
                break;
            }
            FwdArgs f = a;
            // Two groups per task when a group's row slice is at most half a
            // line; a CTA then takes twice the anchors to keep its 8 warps busy.
            constexpr int GP = CH <= 4 ? 2 : 1;
            const bool pair = GP == 2 && a.pb.G % 2 == 0;
            if (pair) {
                const int tpa = a.pb.G / 2;  // tasks per anchor
                f.pb.anchors_per_cta = tpa < kWarps ? kWarps / tpa : 1;
            }
            f.parts = forward_parts(a.pb, ESZ);
            if (f.parts > 1 && (a.pb.K % f.parts) != 0) f.parts = 1;
            int64_t g = sampling_grid(f.pb);
            if (f.parts > 1) {
                f.ctas_per_part = (a.pb.A + f.pb.anchors_per_cta - 1) / f.pb.anchors_per_cta;
                f.kpart = a.pb.K / f.parts;
                f.div_cpp = FastDiv::make(static_cast<uint32_t>(f.ctas_per_part));
                f.div_kpart = FastDiv::make(static_cast<uint32_t>(f.kpart));
                g = static_cast<int64_t>(a.pb.B) * f.parts * f.ctas_per_part;
                // A plain launch after a memset: launched as a programmatic
                // dependent of a zero-fill kernel, the forward took the SMs
                // ahead of the binning that a caller runs beside it on a
                // second stream (6-camera training step 1.011 -> 1.021 ms).
                const cudaError_t e = cudaMemsetAsync(a.out, 0, static_cast<size_t>(a.pb.num_ba) * a.pb.C * 4, st);
                if (e != cudaSuccess) return e;
            }
            const dim3 gg(static_cast<unsigned>(g));
            if (f.parts > 1) {
                if (pair) fwd_kernel<T, CH, false, true, GP><<<gg, kThreads, 0, st>>>(f);
                else fwd_kernel<T, CH, false, true, 1><<<gg, kThreads, 0, st>>>(f);
            } else {
                if (pair) fwd_kernel<T, CH, false, false, GP><<<gg, kThreads, 0, st>>>(f);
                else fwd_kernel<T, CH, false, false, 1><<<gg, kThreads, 0, st>>>(f);
            }
            break;
        }
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_ch(const FwdArgs &a, int chunks, cudaStream_t st)
{
    switch (chunks) {
        case 1: return launch<T, 1>(a, st);
        case 2: return launch<T, 2>(a, st);
        case 4: return launch<T, 4>(a, st);
        case 8: return launch<T, 8>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_forward(const FwdArgs &a, int feat_dtype, int chunks, cudaStream_t st)
{
    switch (feat_dtype) {
        case DA_BF16: return dispatch_ch<Bf16Tag>(a, chunks, st);
        case DA_F16: return dispatch_ch<F16Tag>(a, chunks, st);
        default: return dispatch_ch<float>(a, chunks, st);
    }
}

}  // namespace da
