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
// Decomposition (same as the forward: a warp owns (b*A+a, g), lanes split
// into sample slot, corner and 16-byte chunk):
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
//   * grad_loc: sums over s and g, all inside the CTA (it owns whole
//     anchors). It is accumulated with shared-memory atomics and stored once.
#include "da_internal.cuh"

namespace da {
namespace {

__global__ void zero_fill_kernel(float4 *__restrict__ p, int64_t n4)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <typename T, int CH>
__global__ void __launch_bounds__(kThreads) bwd_kernel(const BwdArgs args)
{
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;
    constexpr int SPP = 8 / CH;
    const Problem &pb = args.pb;

    __shared__ __align__(16) int2 tab[kWarps][32][4];   // {row, w * corner weight}
    __shared__ __align__(16) float dtab[kWarps][32][4]; // per-corner d_i
    extern __shared__ float gl_s[];                      // [anchors_per_cta][P*K][2]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane % CH;
    const int corner = (lane / CH) & 3;
    const int slot = lane / (4 * CH);

    const int64_t ba0 = static_cast<int64_t>(blockIdx.x) * pb.anchors_per_cta;
    const int64_t na = min(static_cast<int64_t>(pb.anchors_per_cta), pb.num_ba - ba0);
    const int ntask = static_cast<int>(na) * pb.G;
    const int64_t row_bytes = static_cast<int64_t>(pb.C) * static_cast<int64_t>(16 / VEC);
    const int64_t grow = pb.C;  // grad_feat row stride, in floats

    const int nloc = static_cast<int>(na) * pb.pk * 2;
    for (int i = threadIdx.x; i < nloc; i += kThreads) gl_s[i] = 0.f;
    __syncthreads();

    for (int task = warp; task < ntask; task += kWarps) {
        const int64_t ba = ba0 + task / pb.G;
        const int aloc = task / pb.G;
        const int g = task % pb.G;
        const int64_t b = ba / pb.A;
        const int64_t coff = static_cast<int64_t>(g) * pb.D + chunk * VEC;  // channel offset
        const char *base = static_cast<const char *>(pb.feat) +
                           (b * pb.rows * pb.C + coff) * (16 / VEC);
        float *gbase = args.grad_feat + b * pb.rows * pb.C + coff;

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

        for (int j0 = 0; j0 < pb.pks; j0 += 32) {
            const int n = min(32, pb.pks - j0);
            // Footprint of sample j0 + lane; kept in registers for the epilogue.
            Footprint f;
            float w = 0.f;
            int jk = 0;
            MapInfo m{};
            if (lane < n) {
                const int j = j0 + lane;
                jk = j / pb.S;
                const int s = j - jk * pb.S;
                const int k = jk % pb.K;
                const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + (ba * pb.pk + jk) * 2);
                w = pb.weights[(ba * pb.pks + j) * pb.G + g];
                m = pb.maps[k * pb.S + s];
                footprint(xy.x, xy.y, m, f);
                int4 *dst = reinterpret_cast<int4 *>(&tab[warp][lane][0]);
                dst[0] = make_int4(f.row[0], __float_as_int(w * f.cw[0]),
                                   f.row[1], __float_as_int(w * f.cw[1]));
                dst[1] = make_int4(f.row[2], __float_as_int(w * f.cw[2]),
                                   f.row[3], __float_as_int(w * f.cw[3]));
            }
            __syncwarp();

            for (int i0 = 0; i0 < n; i0 += 4 * SPP) {
                int2 e[4];
                uint4 raw[4];
                float d[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + slot + u * SPP;
                    e[u] = (i < n) ? tab[warp][i][corner] : make_int2(-1, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    raw[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (e[u].x >= 0) raw[u] = ldg16(base + static_cast<int64_t>(e[u].x) * row_bytes);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float v[VEC];
                    Ck::unpack(raw[u], v);
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc = fmaf(go[q], v[q], acc);
                    d[u] = acc;
                    if (e[u].x >= 0) {
                        const float tw = __int_as_float(e[u].y);
                        float *dst = gbase + static_cast<int64_t>(e[u].x) * grow;
#pragma unroll
                        for (int q = 0; q < VEC / 4; ++q)
                            red_add_v4(dst + 4 * q, tw * go[4 * q], tw * go[4 * q + 1],
                                       tw * go[4 * q + 2], tw * go[4 * q + 3]);
                    }
                }
#pragma unroll
                for (int m2 = 1; m2 < CH; m2 <<= 1) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) d[u] += __shfl_xor_sync(0xffffffffu, d[u], m2);
                }
                if (chunk == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + slot + u * SPP;
                        if (i < n) dtab[warp][i][corner] = d[u];
                    }
                }
            }
            __syncwarp();

            if (lane < n) {
                const float4 dd = *reinterpret_cast<const float4 *>(&dtab[warp][lane][0]);
                const int j = j0 + lane;
                const float gweight = f.cw[0] * dd.x + f.cw[1] * dd.y + f.cw[2] * dd.z + f.cw[3] * dd.w;
                args.grad_weight[(ba * pb.pks + j) * pb.G + g] = gweight;
                const float gx = static_cast<float>(m.W) * w * (f.lh * (dd.w - dd.z) + f.hh * (dd.y - dd.x));
                const float gy = static_cast<float>(m.H) * w * (f.lw * (dd.w - dd.y) + f.hw * (dd.z - dd.x));
                atomicAdd(&gl_s[(aloc * pb.pk + jk) * 2 + 0], gx);
                atomicAdd(&gl_s[(aloc * pb.pk + jk) * 2 + 1], gy);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    float *gdst = args.grad_loc + ba0 * pb.pk * 2;
    for (int i = threadIdx.x; i < nloc; i += kThreads) gdst[i] = gl_s[i];
}

template <typename T, int CH>
cudaError_t launch(const BwdArgs &a, cudaStream_t st)
{
    const int64_t grid = sampling_grid(a.pb);
    if (grid == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(a.pb.anchors_per_cta) * a.pb.pk * 2 * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(bwd_kernel<T, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    bwd_kernel<T, CH><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
    return cudaGetLastError();
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
    zero_fill_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(reinterpret_cast<float4 *>(p), n4);
    return cudaGetLastError();
}

cudaError_t launch_backward(const BwdArgs &a, int feat_dtype, int chunks, cudaStream_t st)
{
    return feat_dtype == DA_BF16 ? dispatch_ch<Bf16Tag>(a, chunks, st)
                                 : dispatch_ch<float>(a, chunks, st);
}

}  // namespace da
