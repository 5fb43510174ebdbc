// Forward sampling kernel of the deformable-aggregation operator.
//
// out[b,a,c] = sum_{p,k,s} weights[b,a,p,k,s,g] * bilinear(map (b,k,s), loc[b,a,p,k], c)
// (page "Inside Sparse4D's CUDA core", §3.2 for the sample and §5.1 for the
// dimensions summed over).
//
// Work decomposition (the page's kernel uses one thread per sample; here a
// warp owns one (b*A+a, g) task and its P*K*S samples):
//   * A CTA of 8 warps owns `anchors_per_cta` whole anchors: all their groups.
//   * Footprints: 32 samples at a time, one per lane. Each lane writes its
//     sample's four {row, weight * corner weight} pairs to a per-warp table in
//     shared memory.
//   * Gather: the D channels of one corner row are D*sizeof(T) bytes, i.e.
//     CH 16-byte chunks. Lane l reads chunk l % CH of corner (l / CH) % 4 of
//     sample slot l / (4*CH). So one warp-wide 16-byte load reads the four
//     corner rows of 8/CH samples, every row as one coalesced segment (the
//     vectorised channel-last access of the DCNv4 page, "Solving the problem:
//     2. let the GPU move less data").
//   * Each lane accumulates its chunk in fp32 registers. At the end, shuffles
//     sum over corners and slots, and the CH lanes of slot 0 write the group's
//     D outputs with 16-byte stores.
#include "da_internal.cuh"

namespace da {
namespace {

template <typename T, int CH>
__global__ void __launch_bounds__(kThreads) fwd_kernel(const FwdArgs args)
{
    using Ck = Chunk<T>;
    constexpr int VEC = Ck::kVec;   // channels per 16-byte chunk
    constexpr int SPP = 8 / CH;     // samples per warp-wide load
    const Problem &pb = args.pb;

    __shared__ __align__(16) int2 tab[kWarps][32][4];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane % CH;
    const int corner = (lane / CH) & 3;
    const int slot = lane / (4 * CH);

    const int64_t ba0 = static_cast<int64_t>(blockIdx.x) * pb.anchors_per_cta;
    const int64_t na = min(static_cast<int64_t>(pb.anchors_per_cta), pb.num_ba - ba0);
    const int ntask = static_cast<int>(na) * pb.G;
    const int64_t row_bytes = static_cast<int64_t>(pb.C) * static_cast<int64_t>(16 / VEC);

    for (int task = warp; task < ntask; task += kWarps) {
        const int64_t ba = ba0 + task / pb.G;
        const int g = task % pb.G;
        const int64_t b = ba / pb.A;
        const char *base = static_cast<const char *>(pb.feat) +
                           (b * pb.rows * pb.C + static_cast<int64_t>(g) * pb.D) * (16 / VEC) +
                           chunk * 16;
        float acc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = 0.f;

        for (int j0 = 0; j0 < pb.pks; j0 += 32) {
            const int n = min(32, pb.pks - j0);
            if (lane < n) {
                const int j = j0 + lane;
                const int jk = j / pb.S;  // p*K + k
                const int s = j - jk * pb.S;
                const int k = jk % pb.K;
                const float2 xy = *reinterpret_cast<const float2 *>(pb.loc + (ba * pb.pk + jk) * 2);
                const float w = pb.weights[(ba * pb.pks + j) * pb.G + g];
                Footprint f;
                footprint(xy.x, xy.y, pb.maps[k * pb.S + s], f);
                int4 *dst = reinterpret_cast<int4 *>(&tab[warp][lane][0]);
                dst[0] = make_int4(f.row[0], __float_as_int(w * f.cw[0]),
                                   f.row[1], __float_as_int(w * f.cw[1]));
                dst[1] = make_int4(f.row[2], __float_as_int(w * f.cw[2]),
                                   f.row[3], __float_as_int(w * f.cw[3]));
            }
            __syncwarp();

            int i = slot;
            for (; i + 3 * SPP < n; i += 4 * SPP) {
                int2 e[4];
                uint4 raw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) e[u] = tab[warp][i + u * SPP][corner];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    raw[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (e[u].x >= 0) raw[u] = ldg16(base + static_cast<int64_t>(e[u].x) * row_bytes);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float v[VEC];
                    Ck::unpack(raw[u], v);
                    const float cw = __int_as_float(e[u].y);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] = fmaf(cw, v[q], acc[q]);
                }
            }
            for (; i < n; i += SPP) {
                const int2 e = tab[warp][i][corner];
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (e.x >= 0) raw = ldg16(base + static_cast<int64_t>(e.x) * row_bytes);
                float v[VEC];
                Ck::unpack(raw, v);
                const float cw = __int_as_float(e.y);
#pragma unroll
                for (int q = 0; q < VEC; ++q) acc[q] = fmaf(cw, v[q], acc[q]);
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
            float4 *o = reinterpret_cast<float4 *>(args.out + ba * pb.C + static_cast<int64_t>(g) * pb.D +
                                                   chunk * VEC);
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q)
                o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
    }
}

template <typename T, int CH>
cudaError_t launch(const FwdArgs &a, cudaStream_t st)
{
    const int64_t grid = sampling_grid(a.pb);
    if (grid == 0) return cudaSuccess;
    fwd_kernel<T, CH><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(a);
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
    return feat_dtype == DA_BF16 ? dispatch_ch<Bf16Tag>(a, chunks, st)
                                 : dispatch_ch<float>(a, chunks, st);
}

}  // namespace da
