/*
 * CPU oracle for the warpaffine preprocessing kernels.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library. The CUDA path shares no code,
 * header or table with it.
 *
 * It follows the page "Hand-written warpaffine kernel" (手写warpaffine核函数):
 *   - §2.1: an affine map is a 2x3 matrix; preprocessing uses the inverse
 *     map d2i from destination pixel (dx, dy) to source coordinates
 *     src_x = m0*dx + m1*dy + m2, src_y = m3*dx + m4*dy + m5;
 *   - §2.2: bilinear interpolation of the four integer neighbours of
 *     (src_x, src_y), each weighted by its distance;
 *   - §3.2: one output pixel of three channels; a destination pixel whose
 *     source point lies outside the source image gets the fill value; the
 *     uint8 output is the interpolated value converted to uint8 (truncation);
 *   - §4.1/§4.2: the fused preprocessing writes float CHW planes, channel
 *     order reversed (BGR in, RGB out), each value v normalised as
 *     (v/255 - mean)/std with the source channel's mean and std.
 *
 * Readings where the page's listing is garbled or inconsistent:
 *   - the bounds test prints without its operators; here a destination pixel
 *     is interpolated iff 0 <= src_x < W and 0 <= src_y < H;
 *   - the listing reads the neighbours at x0+1 and y0+1 without a bounds
 *     check, so at the right and bottom edges it reads past the image. Here a
 *     neighbour outside the image reads the fill value (a constant border);
 *   - the listing pairs the weight (1-wx)*wy with the neighbour (x0+1, y0)
 *     and wx*(1-wy) with (x0, y0+1): the two off-diagonal corners swapped,
 *     which is not the distance weighting §2.2 describes. Here each corner
 *     gets its own weight: (x0, y0) (1-wx)(1-wy), (x0+1, y0) wx(1-wy),
 *     (x0, y0+1) (1-wx)wy, (x0+1, y0+1) wx*wy;
 *   - in the fused preprocessing, v is the interpolated value before any
 *     uint8 conversion (the output is float), and the fill value for outside
 *     pixels.
 *
 * Precision: the uint8 output truncates a float, so floating point decides
 * an integer. The source coordinates, the weights and the four-term sum are
 * fp32 operations in a fixed order, every product and sum rounded (build
 * with -ffp-contract=off), the same steps as the kernel's:
 *   src_x = ((m0*dx) + (m1*dy)) + m2, likewise src_y;
 *   wx = src_x - x0, wy = src_y - y0;
 *   v = ((w00*p00 + w10*p10) + w01*p01) + w11*p11.
 * The normalisation of the fused output is done in double.
 */
#include <math.h>
#include <stdint.h>

#define WAO_OK 0
#define WAO_ERR_ARGS 1

static float corner(const uint8_t *img, int H, int W, int x, int y, int c, uint8_t fill)
{
    if (x < 0 || y < 0 || x >= W || y >= H) return (float)fill;
    return (float)img[((int64_t)y * W + x) * 3 + c];
}

/* The interpolated value of channel c at destination pixel (dx, dy), or the
 * fill value; *inside says which. */
static float sample(const uint8_t *img, int H, int W, const float *m, int dx, int dy, int c, uint8_t fill,
                    int *inside)
{
    float fx = (float)dx, fy = (float)dy;
    float src_x = (m[0] * fx + m[1] * fy) + m[2];
    float src_y = (m[3] * fx + m[4] * fy) + m[5];
    if (!(src_x >= 0.0f && src_y >= 0.0f && src_x < (float)W && src_y < (float)H)) {
        *inside = 0;
        return (float)fill;
    }
    *inside = 1;
    int x0 = (int)floorf(src_x), y0 = (int)floorf(src_y);
    float wx = src_x - (float)x0, wy = src_y - (float)y0;
    float w00 = (1.0f - wx) * (1.0f - wy);
    float w10 = wx * (1.0f - wy);
    float w01 = (1.0f - wx) * wy;
    float w11 = wx * wy;
    float p00 = corner(img, H, W, x0, y0, c, fill);
    float p10 = corner(img, H, W, x0 + 1, y0, c, fill);
    float p01 = corner(img, H, W, x0, y0 + 1, c, fill);
    float p11 = corner(img, H, W, x0 + 1, y0 + 1, c, fill);
    return ((w00 * p00 + w10 * p10) + w01 * p01) + w11 * p11;
}

/* src [B, H, W, 3] uint8, d2i [B, 6], dst [B, Hd, Wd, 3] uint8. */
int wao_warpaffine_u8(int B, int H, int W, int Hd, int Wd, const uint8_t *src, const float *d2i, uint8_t fill,
                      uint8_t *dst)
{
    if (B < 0 || H <= 0 || W <= 0 || Hd < 0 || Wd < 0) return WAO_ERR_ARGS;
    int b, y, x, c, inside;
    for (b = 0; b < B; ++b)
        for (y = 0; y < Hd; ++y)
            for (x = 0; x < Wd; ++x)
                for (c = 0; c < 3; ++c) {
                    float v = sample(src + (int64_t)b * H * W * 3, H, W, d2i + b * 6, x, y, c, fill, &inside);
                    dst[(((int64_t)b * Hd + y) * Wd + x) * 3 + c] = (uint8_t)v;
                }
    return WAO_OK;
}

/* dst [B, 3, Hd, Wd] float: plane o holds source channel 2 - o. */
int wao_warpaffine_preprocess(int B, int H, int W, int Hd, int Wd, const uint8_t *src, const float *d2i,
                              uint8_t fill, const float *mean, const float *stdev, float *dst)
{
    if (B < 0 || H <= 0 || W <= 0 || Hd < 0 || Wd < 0) return WAO_ERR_ARGS;
    int b, y, x, o, inside;
    for (b = 0; b < B; ++b)
        for (o = 0; o < 3; ++o) {
            const int c = 2 - o;
            for (y = 0; y < Hd; ++y)
                for (x = 0; x < Wd; ++x) {
                    double v = sample(src + (int64_t)b * H * W * 3, H, W, d2i + b * 6, x, y, c, fill, &inside);
                    dst[(((int64_t)b * 3 + o) * Hd + y) * Wd + x] =
                        (float)((v / 255.0 - (double)mean[c]) / (double)stdev[c]);
                }
        }
    return WAO_OK;
}
