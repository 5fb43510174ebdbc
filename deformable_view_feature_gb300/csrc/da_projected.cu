// Backward of the upstream step (the projected layout): the chain rule from
// the operator's grad_loc and grad_weight back to the anchors' key points and
// the weight logits.
//
// The forward (da_forward.cu, kLayoutProj) projects key point p of anchor
// (b, a) into camera k and takes a softmax of the logits over the P*K*S
// samples of each (b, a, g). Its derivatives:
//   grad_logits = w * (grad_weight - sum over (p,k,s) of w * grad_weight),
//     per (b, a, g): one warp per anchor (all groups, coalesced) when G
//     divides 32, else one warp per (anchor, group); shuffle sums;
//   grad_keypoints[b,a,p,:] = sum over k of J_k^T grad_loc[b,a,p,k,:], with
//     x = (ud/d)/image_w, y = (vd/d)/image_h and u = ud/d, v = vd/d:
//     dx/dX_i = (m0i - u*m2i) / (d*image_w), dy/dX_i = (m1i - v*m2i) / (d*image_h),
//     0 for a camera the point is behind (the forward's fp32 test d <= 1e-5);
//     one thread per (b, a, p), summing its K cameras.
#include "da_internal.cuh"

namespace da {
namespace {

__global__ void __launch_bounds__(256) logits_grad_kernel(const Problem pb, const float *w, const float *gw,
                                                          float *glog)
{
    pdl_wait();
    pdl_trigger();
    const int64_t task = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (task >= static_cast<int64_t>(pb.num_ba) * pb.G) return;  // whole warps leave together
    const int ba = static_cast<int>(pb.div_G.div(static_cast<uint32_t>(task)));
    const int g = static_cast<int>(task - static_cast<int64_t>(ba) * pb.G);
    const int64_t base = static_cast<int64_t>(ba) * pb.pks * pb.G + g;
    float dot = 0.f;
    for (int j = lane; j < pb.pks; j += 32) {
        const int64_t e = base + static_cast<int64_t>(j) * pb.G;
        dot = fmaf(w[e], gw[e], dot);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    for (int j = lane; j < pb.pks; j += 32) {
        const int64_t e = base + static_cast<int64_t>(j) * pb.G;
        glog[e] = w[e] * (gw[e] - dot);
    }
}

// The same for G dividing 32, coalesced: one warp per anchor reads its
// P*K*S*G contiguous weights as whole 128-byte lines. Lane l only ever sees
// group l % G, so the per-group sums are lane partials summed over the lanes
// of that group (xor shuffles over the bits above log2(G)).
__global__ void __launch_bounds__(256) logits_grad_anchor_kernel(const Problem pb, const float *w, const float *gw,
                                                                 float *glog)
{
    pdl_wait();
    pdl_trigger();
    const int64_t ba = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (ba >= pb.num_ba) return;  // whole warps leave together
    const int64_t n = static_cast<int64_t>(pb.pks) * pb.G;
    const int64_t base = ba * n;
    float dot = 0.f;
    for (int64_t e = lane; e < n; e += 32) dot = fmaf(w[base + e], gw[base + e], dot);
    for (int o = pb.G; o < 32; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    for (int64_t e = lane; e < n; e += 32) glog[base + e] = w[base + e] * (gw[base + e] - dot);
}

__global__ void __launch_bounds__(256) keypoint_grad_kernel(const Problem pb, const float *grad_loc, float *gkp)
{
    pdl_wait();
    pdl_trigger();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (b*A + a)*P + p
    if (i >= static_cast<int64_t>(pb.num_ba) * pb.P) return;
    const int ba = static_cast<int>(pb.div_P.div(static_cast<uint32_t>(i)));
    const int b = static_cast<int>(pb.div_A.div(static_cast<uint32_t>(ba)));
    const float X = pb.keypoints[i * 3], Y = pb.keypoints[i * 3 + 1], Z = pb.keypoints[i * 3 + 2];
    float acc[3] = {0.f, 0.f, 0.f};
    for (int k = 0; k < pb.K; ++k) {
        const float *m = pb.projection + (static_cast<int64_t>(b) * pb.K + k) * 16;
        // The forward's fp32 steps, for the same visibility decision.
        const float ud = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[0], X), __fmul_rn(m[1], Y)), __fmul_rn(m[2], Z)), m[3]);
        const float vd = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[4], X), __fmul_rn(m[5], Y)), __fmul_rn(m[6], Z)), m[7]);
        const float d = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[8], X), __fmul_rn(m[9], Y)), __fmul_rn(m[10], Z)), m[11]);
        if (!(d > 1e-5f)) continue;
        const float gx = grad_loc[(i * pb.K + k) * 2] / (d * pb.image_w);
        const float gy = grad_loc[(i * pb.K + k) * 2 + 1] / (d * pb.image_h);
        const float u = ud / d, v = vd / d;
#pragma unroll
        for (int c = 0; c < 3; ++c) acc[c] += gx * (m[c] - u * m[8 + c]) + gy * (m[4 + c] - v * m[8 + c]);
    }
    gkp[i * 3] = acc[0];
    gkp[i * 3 + 1] = acc[1];
    gkp[i * 3 + 2] = acc[2];
}

}  // namespace

cudaError_t launch_projected_chain(const Problem &pb, const float *weights, const float *grad_loc,
                                   const float *grad_weight, float *grad_keypoints, float *grad_logits,
                                   cudaStream_t st)
{
    const int64_t tasks = static_cast<int64_t>(pb.num_ba) * pb.G;
    if (tasks > 0 && pb.pks > 0) {
        const cudaError_t e =
            32 % pb.G == 0
                ? launch_pdl(logits_grad_anchor_kernel,
                             dim3(static_cast<unsigned>((static_cast<int64_t>(pb.num_ba) * 32 + 255) / 256)), dim3(256),
                             0, st, pb, weights, grad_weight, grad_logits)
                : launch_pdl(logits_grad_kernel, dim3(static_cast<unsigned>((tasks * 32 + 255) / 256)), dim3(256), 0,
                             st, pb, weights, grad_weight, grad_logits);
        if (e != cudaSuccess) return e;
    }
    const int64_t pts = static_cast<int64_t>(pb.num_ba) * pb.P;
    if (pts > 0) {
        const cudaError_t e = launch_pdl(keypoint_grad_kernel, dim3(static_cast<unsigned>((pts + 255) / 256)), dim3(256),
                                         0, st, pb, grad_loc, grad_keypoints);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace da
