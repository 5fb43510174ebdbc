// Warpaffine preprocessing kernels (include/wa.h): the page "Hand-written
// warpaffine kernel", §2-§4.
//
// One thread per destination pixel (three channels), 32x8 blocks (the
// page's suggestion for recent architectures, §5.2), one grid z-slice per
// frame. The source coordinates, the corner weights and the four-term sum
// are fp32 operations in the order wa.h fixes, so the uint8 truncation
// decides the same integer as any other implementation of those steps.
#include <cmath>

#include "da_internal.cuh"
#include "wa.h"

namespace da {
namespace {

constexpr int kWaBx = 32, kWaBy = 8;

struct WaArgs {
    const uint8_t *src;
    const float *d2i;
    int H, W, Hd, Wd;
    float fill;
    float mean[3], inv_std[3];
    uint32_t *dbg_err;  // bounds-checking builds: the device error word
};

// Interpolated channel values of destination pixel (dx, dy) of frame b, or
// the fill value.
__device__ __forceinline__ void wa_sample(const WaArgs &a, int b, int dx, int dy, float (&v)[3])
{
    const float *m = a.d2i + static_cast<int64_t>(b) * 6;
    const float fx = static_cast<float>(dx), fy = static_cast<float>(dy);
    const float sx = __fadd_rn(__fadd_rn(__fmul_rn(m[0], fx), __fmul_rn(m[1], fy)), m[2]);
    const float sy = __fadd_rn(__fadd_rn(__fmul_rn(m[3], fx), __fmul_rn(m[4], fy)), m[5]);
    if (!(sx >= 0.f && sy >= 0.f && sx < static_cast<float>(a.W) && sy < static_cast<float>(a.H))) {
        v[0] = v[1] = v[2] = a.fill;
        return;
    }
    const int x0 = static_cast<int>(floorf(sx)), y0 = static_cast<int>(floorf(sy));
    if (!(DA_CHECK(a.dbg_err, x0, a.W, kBoundsPixel) && DA_CHECK(a.dbg_err, y0, a.H, kBoundsPixel))) {
        v[0] = v[1] = v[2] = a.fill;
        return;
    }
    const float wx = __fsub_rn(sx, static_cast<float>(x0)), wy = __fsub_rn(sy, static_cast<float>(y0));
    const float ux = __fsub_rn(1.f, wx), uy = __fsub_rn(1.f, wy);
    const float w00 = __fmul_rn(ux, uy), w10 = __fmul_rn(wx, uy), w01 = __fmul_rn(ux, wy), w11 = __fmul_rn(wx, wy);
    const bool in_x1 = x0 + 1 < a.W, in_y1 = y0 + 1 < a.H;
    const uint8_t *f = a.src + static_cast<int64_t>(b) * a.H * a.W * 3;
    const uint8_t *r0 = f + (static_cast<int64_t>(y0) * a.W + x0) * 3;
    const uint8_t *r1 = r0 + static_cast<int64_t>(a.W) * 3;
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const float p00 = static_cast<float>(__ldg(r0 + c));
        const float p10 = in_x1 ? static_cast<float>(__ldg(r0 + 3 + c)) : a.fill;
        const float p01 = in_y1 ? static_cast<float>(__ldg(r1 + c)) : a.fill;
        const float p11 = (in_x1 && in_y1) ? static_cast<float>(__ldg(r1 + 3 + c)) : a.fill;
        v[c] = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(w00, p00), __fmul_rn(w10, p10)), __fmul_rn(w01, p01)),
                         __fmul_rn(w11, p11));
    }
}

__global__ void __launch_bounds__(kWaBx *kWaBy) wa_u8_kernel(const WaArgs a, uint8_t *dst)
{
    const int dx = blockIdx.x * kWaBx + threadIdx.x;
    const int dy = blockIdx.y * kWaBy + threadIdx.y;
    const int b = blockIdx.z;
    if (dx >= a.Wd || dy >= a.Hd) return;
    float v[3];
    wa_sample(a, b, dx, dy, v);
    uint8_t *o = dst + ((static_cast<int64_t>(b) * a.Hd + dy) * a.Wd + dx) * 3;
#pragma unroll
    for (int c = 0; c < 3; ++c) o[c] = static_cast<uint8_t>(__float2uint_rz(v[c]));
}

__global__ void __launch_bounds__(kWaBx *kWaBy) wa_preprocess_kernel(const WaArgs a, float *dst)
{
    const int dx = blockIdx.x * kWaBx + threadIdx.x;
    const int dy = blockIdx.y * kWaBy + threadIdx.y;
    const int b = blockIdx.z;
    if (dx >= a.Wd || dy >= a.Hd) return;
    float v[3];
    wa_sample(a, b, dx, dy, v);
    const int64_t plane = static_cast<int64_t>(a.Hd) * a.Wd;
    float *o = dst + static_cast<int64_t>(b) * 3 * plane + static_cast<int64_t>(dy) * a.Wd + dx;
#pragma unroll
    for (int p = 0; p < 3; ++p) {
        const int c = 2 - p;  // RGB planes from BGR channels
        o[p * plane] = (v[c] / 255.f - a.mean[c]) * a.inv_std[c];
    }
}

da_status wa_prepare(const wa_dims *dims, const uint8_t *src, const float *d2i, const void *dst, WaArgs &a,
                     int64_t &npix)
{
    if (!dims) return fail(DA_ERR_NULL, "dims is NULL");
    const wa_dims d = *dims;
    if (d.batch < 0 || d.src_h < 1 || d.src_w < 1 || d.dst_h < 0 || d.dst_w < 0)
        return fail(DA_ERR_SHAPE, "wa_dims: batch %d, source %d x %d, destination %d x %d", d.batch, d.src_h,
                    d.src_w, d.dst_h, d.dst_w);
    if (d.batch > 65535) return fail(DA_ERR_UNSUPPORTED, "batch %d exceeds 65535 frames per call", d.batch);
    npix = static_cast<int64_t>(d.batch) * d.dst_h * d.dst_w;
    if (npix > 0 && (!src || !d2i || !dst)) return fail(DA_ERR_NULL, "src, d2i or dst is NULL");
    if (!aligned(d2i, 4)) return fail(DA_ERR_ALIGN, "d2i must be 4-byte aligned");
    a.src = src;
    a.d2i = d2i;
    a.H = d.src_h;
    a.W = d.src_w;
    a.Hd = d.dst_h;
    a.Wd = d.dst_w;
    a.dbg_err = bounds_word();
    return DA_OK;
}

dim3 wa_grid(const WaArgs &a, int batch)
{
    return dim3(static_cast<unsigned>((a.Wd + kWaBx - 1) / kWaBx), static_cast<unsigned>((a.Hd + kWaBy - 1) / kWaBy),
                static_cast<unsigned>(batch));
}

}  // namespace
}  // namespace da

extern "C" {

da_status wa_warpaffine_u8(const wa_dims *dims, const uint8_t *src, const float *d2i, uint8_t fill, uint8_t *dst,
                           da_stream_t stream)
{
    da::WaArgs a{};
    int64_t npix = 0;
    const da_status st = da::wa_prepare(dims, src, d2i, dst, a, npix);
    if (st != DA_OK) return st;
    if (npix == 0) return DA_OK;
    a.fill = static_cast<float>(fill);
    da::wa_u8_kernel<<<da::wa_grid(a, dims->batch), dim3(da::kWaBx, da::kWaBy), 0,
                       reinterpret_cast<cudaStream_t>(stream)>>>(a, dst);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return da::cuda_fail(e, "warpaffine launch");
    return da::bounds_report(reinterpret_cast<cudaStream_t>(stream));
}

da_status wa_preprocess(const wa_dims *dims, const uint8_t *src, const float *d2i, uint8_t fill, const float *mean,
                        const float *stdev, float *dst, da_stream_t stream)
{
    da::WaArgs a{};
    int64_t npix = 0;
    da_status st = da::wa_prepare(dims, src, d2i, dst, a, npix);
    if (st != DA_OK) return st;
    if (!da::aligned(dst, 4)) return da::fail(DA_ERR_ALIGN, "dst must be 4-byte aligned");
    if (!mean || !stdev) return da::fail(DA_ERR_NULL, "mean / stdev is NULL");
    for (int c = 0; c < 3; ++c) {
        if (!(stdev[c] > 0.f) || !std::isfinite(stdev[c]) || !std::isfinite(mean[c]))
            return da::fail(DA_ERR_SHAPE, "stdev[%d] = %g must be positive and finite (mean finite)", c, stdev[c]);
        a.mean[c] = mean[c];
        a.inv_std[c] = 1.f / stdev[c];
    }
    if (npix == 0) return DA_OK;
    a.fill = static_cast<float>(fill);
    da::wa_preprocess_kernel<<<da::wa_grid(a, dims->batch), dim3(da::kWaBx, da::kWaBy), 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(a, dst);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return da::cuda_fail(e, "preprocess launch");
    return da::bounds_report(reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
