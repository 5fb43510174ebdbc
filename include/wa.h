/*
 * wa.h: warpaffine preprocessing kernels of libda.so (C ABI).
 *
 * The page "Hand-written warpaffine kernel" (手写warpaffine核函数) describes a
 * second bilinear workload next to the deformable aggregation: resizing and
 * warping 8-bit camera frames on the GPU before inference.
 *   - §2.1: the affine map is a 2x3 matrix; the kernel uses the inverse map
 *     d2i from a destination pixel (dx, dy) to source coordinates
 *       src_x = m0*dx + m1*dy + m2,   src_y = m3*dx + m4*dy + m5;
 *   - §2.2: bilinear interpolation of the four integer neighbours of
 *     (src_x, src_y), each weighted by its distance;
 *   - §3.2: one thread per output pixel of three channels; a pixel whose
 *     source point is outside the source image gets the fill value; the
 *     uint8 result is the interpolated value converted to uint8;
 *   - §4.1/§4.2: the fused variant also reverses the channel order (BGR to
 *     RGB), normalises (v/255 - mean)/std and writes planar CHW floats.
 *
 * Conventions are those of da.h (device/host pointers, stream, validation,
 * da_last_error). Readings of the page:
 *   - a destination pixel is interpolated iff 0 <= src_x < W and
 *     0 <= src_y < H (the printed test lost its operators);
 *   - a neighbour outside the image (the column x0+1 = W or the row
 *     y0+1 = H) reads the fill value: a constant border. The printed listing
 *     reads past the image there;
 *   - each corner gets its own distance weight: (x0, y0) (1-wx)(1-wy),
 *     (x0+1, y0) wx(1-wy), (x0, y0+1) (1-wx)wy, (x0+1, y0+1) wx*wy, with
 *     wx = src_x - x0, wy = src_y - y0 (the printed listing swaps the two
 *     off-diagonal weights);
 *   - the uint8 output truncates, so floating point decides the integer:
 *     src_x = ((m0*dx) + (m1*dy)) + m2 (likewise src_y), the weights and
 *     v = ((w00*p00 + w10*p10) + w01*p01) + w11*p11 are fp32 operations in
 *     this order, each product and sum rounded (no fused multiply-add).
 */
#ifndef WA_H_
#define WA_H_

#include "da.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct wa_dims {
    int32_t batch;  /* B >= 0 frames */
    int32_t src_h;  /* H >= 1 */
    int32_t src_w;  /* W >= 1 */
    int32_t dst_h;  /* Hd >= 0 */
    int32_t dst_w;  /* Wd >= 0 */
} wa_dims;

/*
 * wa_warpaffine_u8
 *   src  device [B, H, W, 3] uint8 (HWC, rows of W*3 bytes), any alignment.
 *   d2i  device [B, 6] fp32, 4-byte aligned: frame b's destination -> source
 *        matrix (m0..m5 above).
 *   fill the value of every channel of an outside pixel.
 *   dst  device [B, Hd, Wd, 3] uint8; overwritten.
 */
da_status wa_warpaffine_u8(const wa_dims *dims, const uint8_t *src, const float *d2i, uint8_t fill, uint8_t *dst,
                           da_stream_t stream);

/*
 * wa_preprocess: the fused preprocessing.
 *   src, d2i, fill as above.
 *   mean, stdev host [3] fp32, in the source's channel order (B, G, R);
 *        stdev > 0.
 *   dst  device [B, 3, Hd, Wd] fp32, 4-byte aligned; plane o holds source
 *        channel 2 - o (R, G, B), each value (v/255 - mean[c]) / stdev[c] with v
 *        the interpolated value (or the fill value), not truncated, and
 *        (v/255 - mean[c]) * (1/stdev[c]) computed in fp32.
 */
da_status wa_preprocess(const wa_dims *dims, const uint8_t *src, const float *d2i, uint8_t fill, const float *mean,
                        const float *stdev, float *dst, da_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WA_H_ */
