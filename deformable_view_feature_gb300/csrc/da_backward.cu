// Backward kernels of the deformable-aggregation operator: the three gradients
// of the page "Inside Sparse4D's CUDA core", §4.1. For one sample with weight
// w, corners v1..v4 and corner weights w1..w4:
//   top_grad    = grad_out * w (per channel)
//   grad_feat   += w_i * top_grad at corner i (inside the map only)
//   grad_loc[0] += W * (lh*(v4-v3) + hh*(v2-v1)) * top_grad   (x pairs with W)
//   grad_loc[1] += H * (lw*(v4-v2) + hw*(v3-v1)) * top_grad   (y pairs with H)
//   grad_weight += grad_out * (w1*v1 + w2*v2 + w3*v3 + w4*v4)
// each summed over the group's D channels.
//
// Decomposition: a warp owns one (b, k, a, g) task, i.e. the P*S samples of
// one anchor in one camera for one group. Lanes split into sample slot,
// corner and 16-byte chunk, as in the forward.
//   * d_i = sum_c grad_out[c] * v_i[c] is the only per-channel reduction the
//     three gradients need: grad_weight = sum_i w_i d_i, grad_x =
//     W*w*(lh*(d4-d3) + hh*(d2-d1)), grad_y = H*w*(lw*(d4-d2) + hw*(d3-d1)). Each
//     lane forms its chunk's part of d_i, shuffles sum it over the CH lanes of
//     the row, and the per-corner totals go to shared memory. The lane that
//     built the sample's footprint then finishes the three gradients for it.
//   * grad_feat: each lane adds (w * w_i) * grad_out for its chunk with one
//     16-byte vector reduction (red.global.add.v4.f32). The scatter is the one
//     place where samples of different anchors meet, so it must be atomic.
//   * grad_weight: every (b,a,p,k,s,g) belongs to one warp: a plain store.
//   * grad_loc[b,a,p,k] sums over s and g, all inside the CTA that owns view
//     (b, k, a). It is accumulated with shared-memory atomics and stored
//     once.
// With FUSED (per-group locations, one loc_weight tensor [B,A,G,P,K,2+S]),
// grad_loc is kept per group (summed over s only), and both gradients land
// in one grad_loc_weight tensor of the same layout.
#include "da_internal.cuh"

namespace da {
namespace {

__global__ void zero_fill_kernel(float4 *__restrict__ p, int64_t n4)
{
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Sums each of a lane's four per-sample values d[0..3] over the CH lanes of
// its corner row (the lanes that differ only in the chunk bits). Instead of
// reducing each value on its own (4*log2(CH) shuffles), the lanes split the
// work: each halving step sends half of the values still held. After the
// last step each sum sits in CH/4 lanes (CH >= 4), or 2 or 4 sums per lane
// (CH = 2 or 1). Then one lane per sum stores it to dst[u * 4], the table
// entry of sample i + u.
template <int CH>
__device__ __forceinline__ void row_sum_store(const float (&d)[4], int chunk, float *dst)
{
    if constexpr (CH >= 4) {
        const bool hA = (chunk & (CH / 2)) != 0;
        float a0 = hA ? d[2] : d[0], a1 = hA ? d[3] : d[1];
        const float s0 = hA ? d[0] : d[2], s1 = hA ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, CH / 2);
        a1 += __shfl_xor_sync(0xffffffffu, s1, CH / 2);
        const bool hB = (chunk & (CH / 4)) != 0;
        float r = hB ? a1 : a0;
        const float t = hB ? a0 : a1;
        r += __shfl_xor_sync(0xffffffffu, t, CH / 4);
#pragma unroll
        for (int m = CH / 8; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
        if ((chunk & (CH / 4 - 1)) == 0) dst[((hA ? 2 : 0) + (hB ? 1 : 0)) * 4] = r;
    } else if constexpr (CH == 2) {
        const bool h = (chunk & 1) != 0;
        float a0 = h ? d[2] : d[0], a1 = h ? d[3] : d[1];
        const float s0 = h ? d[0] : d[2], s1 = h ? d[1] : d[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        a1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        dst[(h ? 2 : 0) * 4] = a0;
        dst[(h ? 3 : 1) * 4] = a1;
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u * 4] = d[u];
    }
}

// The backward walks the problem camera-major: CTA i owns the views
// v = (b*K + k)*A + a in [i*views_per_cta, (i+1)*views_per_cta), all groups
// of each. At any moment the resident CTAs touch the maps of one or two
// cameras of one batch item (feat and grad_feat slices of NPIX*C values each).
// That working set stays in L2, so the grad_feat reductions hit lines that
// are already there. Every output element still has one owner:
//   * grad_weight and grad_loc are per camera;
//   * grad_feat rows belong to one camera's maps.
template <typename T, int CH, bool FUSED>
__global__ void __launch_bounds__(kThreads, 4) bwd_kernel(const BwdArgs args)
{
    pdl_wait();
    pdl_trigger();
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;
    constexpr int ESZ = 16 / VEC;
    constexpr int SPP = 8 / CH;
    const Problem &pb = args.pb;

    __shared__ __align__(16) int2 tab[kWarps][4][kTabPitch];  // {row, w * corner weight}
    __shared__ __align__(16) float dtab[kWarps][32][4];        // per-corner d_i of each sample
    // Epilogue coefficients per sample: grad_weight = sum cw_i d_i,
    // grad_x = sum ax_i d_i, grad_y = sum ay_i d_i.
    __shared__ __align__(16) float4 etab[kWarps][32][3];
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    extern __shared__ float gl_s[];  // [views_per_cta][P][2], or [views_per_cta][G][P][2] if FUSED

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane % CH;
    const int corner = (lane / CH) & 3;
    const int slot = lane / (4 * CH);

    const int num_views = pb.num_ba * pb.K;
    const int v0 = static_cast<int>(blockIdx.x) * pb.anchors_per_cta;
    const int nv = min(pb.anchors_per_cta, num_views - v0);
    const int ntask = nv * pb.G;
    const int ps = pb.P * pb.S;  // samples per task
    const uint32_t row_bytes = static_cast<uint32_t>(pb.C) * ESZ;
    const uint32_t grow_bytes = static_cast<uint32_t>(pb.C) * 4;  // grad_feat row pitch

    stage_maps(pb, maps_s);
    const int gl_groups = FUSED ? pb.G : 1;
    const int nloc = nv * gl_groups * pb.P * 2;
    for (int i = threadIdx.x; i < nloc; i += kThreads) gl_s[i] = 0.f;
    __syncthreads();

    for (int task = warp; task < ntask; task += kWarps) {
        const int vloc = static_cast<int>(pb.div_G.div(task));
        const int g = task - vloc * pb.G;
        const int view = v0 + vloc;
        const int bk = static_cast<int>(pb.div_A.div(view));
        const int a = view - bk * pb.A;
        const int b = static_cast<int>(pb.div_K.div(bk));
        const int k = bk - b * pb.K;
        const int64_t ba = static_cast<int64_t>(b) * pb.A + a;
        const int64_t coff = static_cast<int64_t>(g) * pb.D + chunk * VEC;  // channel offset
        const char *base = static_cast<const char *>(pb.feat) + (b * pb.rows * pb.C + coff) * ESZ;
        char *gbase = reinterpret_cast<char *>(args.grad_feat + b * pb.rows * pb.C + coff);

        float go[VEC];
        {
            const float4 *src = reinterpret_cast<const float4 *>(args.grad_out + ba * pb.C + coff);
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const float4 t = src[q];
                go[4 * q] = t.x;
                go[4 * q + 1] = t.y;
                go[4 * q + 2] = t.z;
                go[4 * q + 3] = t.w;
            }
        }

        for (int j0 = 0; j0 < ps; j0 += 32) {
            const int n = min(32, ps - j0);
            // Footprint of sample j0 + lane: the gather table, and the
            // coefficients that turn the four d_i into the three gradients
            // (page §4.1: grad_w = lh*(v4-v3) + hh*(v2-v1) times W*w, and
            // grad_h = lw*(v4-v2) + hw*(v3-v1) times H*w).
            {
                int row[4] = {-1, -1, -1, -1};
                float tw[4] = {0.f, 0.f, 0.f, 0.f};
                if (lane < n) {
                    const int j = j0 + lane;
                    const int p = static_cast<int>(pb.div_S.div(j));
                    const int s = j - p * pb.S;
                    float2 xy;
                    float w;
                    sample_xyw<FUSED ? kLayoutFused : kLayoutStd>(pb, ba, g, p * pb.K + k, s, xy, w);
                    const MapInfo m = maps_s[k * pb.S + s];
                    Footprint f;
                    footprint(xy.x, xy.y, m, f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        row[c] = f.row[c];
                        tw[c] = w * f.cw[c];
                    }
                    const float wx = static_cast<float>(m.W) * w;
                    const float wy = static_cast<float>(m.H) * w;
                    etab[warp][lane][0] = make_float4(f.cw[0], f.cw[1], f.cw[2], f.cw[3]);
                    etab[warp][lane][1] = make_float4(-wx * f.hh, wx * f.hh, -wx * f.lh, wx * f.lh);
                    etab[warp][lane][2] = make_float4(-wy * f.hw, -wy * f.lw, wy * f.hw, wy * f.lw);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) tab[warp][c][lane] = make_int2(row[c], __float_as_int(tw[c]));
            }
            __syncwarp();

            for (int i0 = 0; i0 < n; i0 += 4 * SPP) {
                const int i = i0 + 4 * slot;
                const int4 e01 = *reinterpret_cast<const int4 *>(&tab[warp][corner][i]);
                const int4 e23 = *reinterpret_cast<const int4 *>(&tab[warp][corner][i + 2]);
                const int r[4] = {e01.x, e01.z, e23.x, e23.z};
                const float tw[4] = {__int_as_float(e01.y), __int_as_float(e01.w), __int_as_float(e23.y),
                                     __int_as_float(e23.w)};
                uint4 raw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) raw[u] = ldg16_if(feat_row_ok(pb, r[u]), row_addr(base, r[u], row_bytes));
                float d[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float v[VEC];
                    Ck::unpack(raw[u], v);
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc = fmaf(go[q], v[q], acc);
                    d[u] = acc;
                    float *dst = reinterpret_cast<float *>(gbase + static_cast<uint64_t>(static_cast<uint32_t>(r[u])) *
                                                                       grow_bytes);
#pragma unroll
                    for (int q = 0; q < VEC / 4; ++q)
                        red_add_v4_if(feat_row_ok(pb, r[u]), dst + 4 * q, tw[u] * go[4 * q], tw[u] * go[4 * q + 1],
                                      tw[u] * go[4 * q + 2], tw[u] * go[4 * q + 3]);
                }
                row_sum_store<CH>(d, chunk, &dtab[warp][i][corner]);
            }
            __syncwarp();

            if (lane < n) {
                const int j = j0 + lane;
                const int p = static_cast<int>(pb.div_S.div(j));
                const int s = j - p * pb.S;
                const float4 dd = *reinterpret_cast<const float4 *>(&dtab[warp][lane][0]);
                const float4 cw = etab[warp][lane][0];
                const float4 ax = etab[warp][lane][1];
                const float4 ay = etab[warp][lane][2];
                const float gweight = cw.x * dd.x + cw.y * dd.y + cw.z * dd.z + cw.w * dd.w;
                if constexpr (FUSED)
                    args.grad_loc[((ba * pb.G + g) * pb.pk + p * pb.K + k) * (2 + pb.S) + 2 + s] = gweight;
                else
                    args.grad_weight[(((ba * pb.P + p) * pb.K + k) * pb.S + s) * pb.G + g] = gweight;
                const float gx = ax.x * dd.x + ax.y * dd.y + ax.z * dd.z + ax.w * dd.w;
                const float gy = ay.x * dd.x + ay.y * dd.y + ay.z * dd.z + ay.w * dd.w;
                const int gslot = ((vloc * gl_groups + (FUSED ? g : 0)) * pb.P + p) * 2;
                atomicAdd(&gl_s[gslot + 0], gx);
                atomicAdd(&gl_s[gslot + 1], gy);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // grad_loc[b,a,p,k,:] for the CTA's views: a stride of K pairs between p.
    // (FUSED: grad_loc_weight[b,a,g,p,k,0..1].)
    for (int i = threadIdx.x; i < nloc; i += kThreads) {
        const int vg = i / (pb.P * 2);  // vloc * gl_groups + g
        const int r = i - vg * pb.P * 2;
        const int p = r >> 1;
        const int vloc = vg / gl_groups;
        const int g = vg - vloc * gl_groups;
        const int view = v0 + vloc;
        const int bk = static_cast<int>(pb.div_A.div(view));
        const int a = view - bk * pb.A;
        const int b = static_cast<int>(pb.div_K.div(bk));
        const int k = bk - b * pb.K;
        const int64_t ba = static_cast<int64_t>(b) * pb.A + a;
        if constexpr (FUSED)
            args.grad_loc[((ba * pb.G + g) * pb.pk + p * pb.K + k) * (2 + pb.S) + (r & 1)] = gl_s[i];
        else
            args.grad_loc[((ba * pb.P + p) * pb.K + k) * 2 + (r & 1)] = gl_s[i];
    }
}

// Few samples per (anchor, group) (the DCNv4 form): one thread per 16-byte
// chunk of an anchor's C channels, as in the forward's small-task kernel.
// An anchor's cpa threads (a power of two, at most 32) are adjacent lanes;
// the CH lanes of a group sum the corner dot products d_i with xor
// shuffles, and (standard layout) the groups' grad_loc terms are summed over
// the anchor's lanes the same way. kSmallUnroll samples' loads are in
// flight together.
constexpr int kSmallUnroll = 3;

template <typename T, bool FUSED>
__global__ void __launch_bounds__(kThreads) bwd_small_kernel(const BwdArgs args, int cpa_log2, int ch)
{
    pdl_wait();
    pdl_trigger();
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;
    constexpr int ESZ = 16 / VEC;
    const Problem &pb = args.pb;
    __shared__ MapInfo maps_s[DA_MAX_MAPS];
    stage_maps(pb, maps_s);
    __syncthreads();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int cpa = 1 << cpa_log2;
    const int64_t ba_raw = t >> cpa_log2;
    // Lanes past the last anchor run along on anchor num_ba - 1 (whole
    // anchors, so the shuffles stay within live lanes) and store nothing.
    const bool live = ba_raw < pb.num_ba;
    const int64_t ba = live ? ba_raw : pb.num_ba - 1;
    const int chunk = static_cast<int>(t & (cpa - 1));
    const int c0 = chunk * VEC;
    const int g = c0 / pb.D;
    const int gsub = chunk & (ch - 1);
    const int b = static_cast<int>(pb.div_A.div(static_cast<uint32_t>(ba)));
    const char *base = static_cast<const char *>(pb.feat) + (static_cast<int64_t>(b) * pb.rows * pb.C + c0) * ESZ;
    float *gbase = args.grad_feat + static_cast<int64_t>(b) * pb.rows * pb.C + c0;
    const uint32_t row_bytes = static_cast<uint32_t>(pb.C) * ESZ;
    float go[VEC];
    {
        const float4 *src = reinterpret_cast<const float4 *>(args.grad_out + ba * pb.C + c0);
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const float4 v = src[q];
            go[4 * q] = v.x;
            go[4 * q + 1] = v.y;
            go[4 * q + 2] = v.z;
            go[4 * q + 3] = v.w;
        }
    }
    float gx = 0.f, gy = 0.f;  // the current (p, k): sums over s
    for (int j0 = 0; j0 < pb.pks; j0 += kSmallUnroll) {
        uint4 raw[kSmallUnroll][4];
        Footprint f[kSmallUnroll];
        float w[kSmallUnroll];
        int mw[kSmallUnroll], mh[kSmallUnroll];
#pragma unroll
        for (int u = 0; u < kSmallUnroll; ++u) {
            const int j = j0 + u;
            w[u] = 0.f;
            mw[u] = mh[u] = 0;
            if (j < pb.pks) {
                const int jk = static_cast<int>(pb.div_S.div(j));
                const int s = j - jk * pb.S;
                const int k = jk - static_cast<int>(pb.div_K.div(jk)) * pb.K;
                float2 xy;
                sample_xyw<FUSED ? kLayoutFused : kLayoutStd>(pb, ba, g, jk, s, xy, w[u]);
                const MapInfo m = maps_s[k * pb.S + s];
                mw[u] = m.W;
                mh[u] = m.H;
                footprint(xy.x, xy.y, m, f[u]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    f[u].row[c] = -1;
                    f[u].cw[c] = 0.f;
                }
                f[u].lh = f[u].lw = f[u].hh = f[u].hw = 0.f;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) raw[u][c] = ldg16_if(feat_row_ok(pb, f[u].row[c]), row_addr(base, f[u].row[c], row_bytes));
        }
#pragma unroll
        for (int u = 0; u < kSmallUnroll; ++u) {
            const int j = j0 + u;
            if (j >= pb.pks) break;  // uniform: every lane walks the same j
            float d[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[VEC];
                Ck::unpack(raw[u][c], v);
                float acc = 0.f;
#pragma unroll
                for (int q = 0; q < VEC; ++q) acc = fmaf(go[q], v[q], acc);
                d[c] = acc;
                const float tw = w[u] * f[u].cw[c];
                float *dst = gbase + static_cast<int64_t>(f[u].row[c]) * pb.C;
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q)
                    red_add_v4_if(live && feat_row_ok(pb, f[u].row[c]), dst + 4 * q, tw * go[4 * q], tw * go[4 * q + 1],
                                  tw * go[4 * q + 2], tw * go[4 * q + 3]);
            }
            for (int m = 1; m < ch; m <<= 1)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[c] += __shfl_xor_sync(0xffffffffu, d[c], m);
            const int jk = static_cast<int>(pb.div_S.div(j));
            const int s = j - jk * pb.S;
            const float gweight = f[u].cw[0] * d[0] + f[u].cw[1] * d[1] + f[u].cw[2] * d[2] + f[u].cw[3] * d[3];
            const float wx = static_cast<float>(mw[u]) * w[u];
            const float wy = static_cast<float>(mh[u]) * w[u];
            gx += wx * (f[u].lh * (d[3] - d[2]) + f[u].hh * (d[1] - d[0]));
            gy += wy * (f[u].lw * (d[3] - d[1]) + f[u].hw * (d[2] - d[0]));
            if constexpr (FUSED) {
                float *e = args.grad_loc + ((ba * pb.G + g) * pb.pk + jk) * (2 + pb.S);
                if (live && gsub == 0) e[2 + s] = gweight;
                if (s == pb.S - 1) {
                    if (live && gsub == 0) {
                        e[0] = gx;
                        e[1] = gy;
                    }
                    gx = gy = 0.f;
                }
            } else {
                if (live && gsub == 0) args.grad_weight[((ba * pb.pk + jk) * pb.S + s) * pb.G + g] = gweight;
                if (s == pb.S - 1) {
                    // Sum over the groups: one value per group, held by
                    // all of its lanes.
                    for (int m = ch; m < cpa; m <<= 1) {
                        gx += __shfl_xor_sync(0xffffffffu, gx, m);
                        gy += __shfl_xor_sync(0xffffffffu, gy, m);
                    }
                    if (live && chunk == 0) {
                        args.grad_loc[(ba * pb.pk + jk) * 2] = gx;
                        args.grad_loc[(ba * pb.pk + jk) * 2 + 1] = gy;
                    }
                    gx = gy = 0.f;
                }
            }
        }
    }
}

template <typename T, int CH, bool FUSED>
cudaError_t launch_layout(const BwdArgs &a, cudaStream_t st)
{
    constexpr int ESZ = 16 / Chunk<T>::kVec;
    if (use_small_task_kernels(a.pb, ESZ)) {
        const int cpa = a.pb.C * ESZ / 16;
        if ((cpa & (cpa - 1)) == 0) {
            int cpa_log2 = 0;
            while ((1 << cpa_log2) < cpa) ++cpa_log2;
            const int64_t threads = static_cast<int64_t>(a.pb.num_ba) << cpa_log2;
            const int64_t grid = (threads + kThreads - 1) / kThreads;
            if (grid == 0) return cudaSuccess;
            return launch_pdl(bwd_small_kernel<T, FUSED>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, st, a,
                              cpa_log2, CH);
        }
    }
    const int64_t views = static_cast<int64_t>(a.pb.num_ba) * a.pb.K;
    const int64_t grid = (views + a.pb.anchors_per_cta - 1) / a.pb.anchors_per_cta;
    if (grid == 0) return cudaSuccess;
    const size_t smem = scatter_smem_bytes(a.pb);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(bwd_kernel<T, CH, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(bwd_kernel<T, CH, FUSED>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, st, a);
}

template <typename T, int CH>
cudaError_t launch(const BwdArgs &a, cudaStream_t st)
{
    return a.pb.layout == kLayoutFused ? launch_layout<T, CH, true>(a, st) : launch_layout<T, CH, false>(a, st);
}

template <typename T>
cudaError_t dispatch_ch(const BwdArgs &a, int chunks, cudaStream_t st)
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

cudaError_t launch_zero_fill(float *p, int64_t n_floats, cudaStream_t st)
{
    const int64_t n4 = n_floats / 4;  // callers pass a multiple of 4
    if (n4 == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (n4 + 1023) / 1024;
    const int64_t grid = want < static_cast<int64_t>(sms) * 8 ? want : static_cast<int64_t>(sms) * 8;
    return launch_pdl(zero_fill_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st,
                      reinterpret_cast<float4 *>(p), n4);
}

cudaError_t launch_backward(const BwdArgs &a, int feat_dtype, int chunks, cudaStream_t st)
{
    switch (feat_dtype) {
        case DA_BF16: return dispatch_ch<Bf16Tag>(a, chunks, st);
        case DA_F16: return dispatch_ch<F16Tag>(a, chunks, st);
        default: return dispatch_ch<float>(a, chunks, st);
    }
}

}  // namespace da
