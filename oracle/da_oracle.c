/*
 * CPU oracle for the Sparse4D deformable-aggregation operator.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library. The CUDA path shares no code,
 * header or table with it.
 *
 * The code is plain, single-threaded C11. It is slow and written to be easy
 * to check by eye against the page "Inside Sparse4D's CUDA core:
 * deformable_aggregation bilinear interpolation and gradient
 * back-propagation" (深入Sparse4D的CUDA核心：图解deformable_aggregation算子的双线性插值与梯度回传):
 *   - §3.1: HWC layout; the pixel (i, j) of a map starts at i*W*C + j*C;
 *   - §3.2: bilinear interpolation: floor gives the four corners, lh/lw/hh/hw
 *     give their weights, corners outside the map read 0, and the value is
 *     w1*v1 + w2*v2 + w3*v3 + w4*v4;
 *   - §4.1: the three gradients. top_grad = grad_output * weight is
 *     scattered to the corners with the corner weights;
 *     grad_w = lh*(v4-v3) + hh*(v2-v1) scaled by the width feeds
 *     sampling_location[0]; grad_h = lw*(v4-v2) + hw*(v3-v1) scaled by the
 *     height feeds sampling_location[1]; grad_weights += grad_output * val;
 *   - §5.1: the sum runs over the six dimensions batch, pts, embeds,
 *     anchors, cams and scales.
 *
 * Precision (the page's own listing declares h_im, lh, hh, lw, hw as float):
 *   - the sampling coordinate h_im = y*H - 0.5 and the fractional weights
 *     lh, hh, lw, hw are computed in fp32, with two roundings and no fused
 *     multiply-add (build with -ffp-contract=off). They decide which integer
 *     corners are read, so both implementations must take that decision in
 *     the same precision;
 *   - everything after that is accumulated in double and rounded to fp32 once,
 *     at the end.
 *
 * Readings where the page is garbled or silent:
 *   - §3.2 prints only part of the bounds test. Here a corner is read iff
 *     0 <= row <= H-1 and 0 <= col <= W-1, with all four inequalities for
 *     every corner; otherwise it reads 0;
 *   - a sample whose h_im or w_im is not finite reads nothing and gets zero
 *     gradients;
 *   - every output is overwritten, never accumulated into.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DAO_OK 0
#define DAO_ERR_ARGS 1
#define DAO_ERR_NOMEM 2

/* The four corners of one bilinear sample, in the page's order:
 * 1 = (h_low, w_low), 2 = (h_low, w_high), 3 = (h_high, w_low),
 * 4 = (h_high, w_high). row[i] is the feature row, or -1 outside the map. */
typedef struct {
    int64_t row[4];
    float lh, lw, hh, hw;
} footprint;

static void make_footprint(float x, float y, int32_t H, int32_t W, int64_t start,
                           footprint *f)
{
    /* §3.2: the normalised location times the map size, shifted half a pixel. */
    float yh = y * (float)H;
    float h_im = yh - 0.5f;
    float xw = x * (float)W;
    float w_im = xw - 0.5f;
    int i;
    for (i = 0; i < 4; ++i) f->row[i] = -1;
    f->lh = f->lw = f->hh = f->hw = 0.0f;
    if (!isfinite(h_im) || !isfinite(w_im)) return;

    float h_low = floorf(h_im);
    float w_low = floorf(w_im);
    f->lh = h_im - h_low;
    f->lw = w_im - w_low;
    f->hh = 1.0f - f->lh;
    f->hw = 1.0f - f->lw;

    double rows[4] = {h_low, h_low, (double)h_low + 1.0, (double)h_low + 1.0};
    double cols[4] = {w_low, (double)w_low + 1.0, w_low, (double)w_low + 1.0};
    for (i = 0; i < 4; ++i) {
        if (rows[i] >= 0.0 && rows[i] <= (double)(H - 1) &&
            cols[i] >= 0.0 && cols[i] <= (double)(W - 1)) {
            f->row[i] = start + (int64_t)rows[i] * W + (int64_t)cols[i];
        }
    }
}

/* w1..w4 of §3.2, formed in double from the fp32 fractional weights. */
static void corner_weights(const footprint *f, double cw[4])
{
    cw[0] = (double)f->hh * (double)f->hw;
    cw[1] = (double)f->hh * (double)f->lw;
    cw[2] = (double)f->lh * (double)f->hw;
    cw[3] = (double)f->lh * (double)f->lw;
}

/* IEEE binary16 bits to double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 holds zero and the
 * subnormals (fraction * 2^-24), exponent 31 infinity and NaN. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* feat_kind: 0 = fp32, 1 = bf16 bits, 2 = fp16 bits. */
static double feat_value(const void *feat, int feat_kind, int64_t index)
{
    if (feat_kind == 1) {
        /* bf16 is the top half of an fp32 bit pattern: widening is exact. */
        uint32_t bits = (uint32_t)((const uint16_t *)feat)[index] << 16;
        float v;
        memcpy(&v, &bits, sizeof v);
        return (double)v;
    }
    if (feat_kind == 2) return f16_bits_to_double(((const uint16_t *)feat)[index]);
    return (double)((const float *)feat)[index];
}

static int check_dims(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                      const int32_t *shape, const int32_t *start)
{
    int k, s;
    if (B < 0 || K < 0 || S < 0 || A < 0 || P < 0 || C <= 0 || G <= 0 || C % G) return 0;
    if (rows < 0) return 0;
    for (k = 0; k < K; ++k)
        for (s = 0; s < S; ++s) {
            int32_t H = shape[(k * S + s) * 2], W = shape[(k * S + s) * 2 + 1];
            int64_t st = start[k * S + s];
            if (H <= 0 || W <= 0 || st < 0 || st + (int64_t)H * W > rows) return 0;
        }
    return 1;
}

/*
 * Forward (§3.2 and §5.1):
 *   out[b,a,c] = sum over p,k,s of
 *                weights[b,a,p,k,s,g(c)] * bilinear(map (b,k,s), loc[b,a,p,k], c),
 * with g(c) = c / (C/G). Only anchors with flat index b*A+a in
 * [ba_begin, ba_end) are computed; out holds their rows only, starting at
 * ba_begin.
 */
int dao_forward(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                const int32_t *shape, const int32_t *start,
                const void *feat, int feat_kind,
                const float *loc, const float *weights,
                int64_t ba_begin, int64_t ba_end, float *out)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    if (ba_begin < 0 || ba_end < ba_begin || ba_end > (int64_t)B * A) return DAO_ERR_ARGS;
    const int D = C / G;
    double *acc = (double *)malloc(sizeof(double) * (size_t)C);
    double *val = (double *)malloc(sizeof(double) * (size_t)D);
    if (!acc || !val) { free(acc); free(val); return DAO_ERR_NOMEM; }

    int64_t ba;
    for (ba = ba_begin; ba < ba_end; ++ba) {
        const int64_t b = ba / A;
        memset(acc, 0, sizeof(double) * (size_t)C);
        int p, k, s, g, c, i;
        for (p = 0; p < P; ++p)
            for (k = 0; k < K; ++k) {
                const float *xy = loc + ((ba * P + p) * K + k) * 2;
                for (s = 0; s < S; ++s) {
                    const int32_t H = shape[(k * S + s) * 2];
                    const int32_t W = shape[(k * S + s) * 2 + 1];
                    footprint f;
                    double cw[4];
                    make_footprint(xy[0], xy[1], H, W, start[k * S + s], &f);
                    corner_weights(&f, cw);
                    for (g = 0; g < G; ++g) {
                        const double w = weights[(((ba * P + p) * K + k) * S + s) * G + g];
                        for (c = 0; c < D; ++c) val[c] = 0.0;
                        for (i = 0; i < 4; ++i) {
                            if (f.row[i] < 0) continue;
                            const int64_t base = (b * rows + f.row[i]) * C + (int64_t)g * D;
                            for (c = 0; c < D; ++c)
                                val[c] += cw[i] * feat_value(feat, feat_kind, base + c);
                        }
                        for (c = 0; c < D; ++c) acc[g * D + c] += w * val[c];
                    }
                }
            }
        for (int c2 = 0; c2 < C; ++c2) out[(ba - ba_begin) * C + c2] = (float)acc[c2];
    }
    free(acc);
    free(val);
    return DAO_OK;
}

/*
 * Backward (§4.1), for the anchors with flat index in [ba_begin, ba_end):
 *   grad_feat   [B, rows, C]      : every element is written; it holds the
 *                                   contributions of the selected anchors;
 *   grad_loc    [ba_end-ba_begin, P, K, 2];
 *   grad_weight [ba_end-ba_begin, P, K, S, G].
 */
int dao_backward(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                 const int32_t *shape, const int32_t *start,
                 const void *feat, int feat_kind,
                 const float *loc, const float *weights, const float *grad_out,
                 int64_t ba_begin, int64_t ba_end,
                 float *grad_feat, float *grad_loc, float *grad_weight)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    if (ba_begin < 0 || ba_end < ba_begin || ba_end > (int64_t)B * A) return DAO_ERR_ARGS;
    const int D = C / G;
    const int64_t nfeat = (int64_t)B * rows * C;
    double *gf = (double *)calloc((size_t)(nfeat > 0 ? nfeat : 1), sizeof(double));
    double *gl = (double *)calloc((size_t)(P * K * 2 > 0 ? P * K * 2 : 1), sizeof(double));
    if (!gf || !gl) { free(gf); free(gl); return DAO_ERR_NOMEM; }

    int64_t ba;
    for (ba = ba_begin; ba < ba_end; ++ba) {
        const int64_t b = ba / A;
        const int64_t lba = ba - ba_begin;
        memset(gl, 0, sizeof(double) * (size_t)(P * K * 2));
        int p, k, s, g, c, i;
        for (p = 0; p < P; ++p)
            for (k = 0; k < K; ++k) {
                const float *xy = loc + ((ba * P + p) * K + k) * 2;
                for (s = 0; s < S; ++s) {
                    const int32_t H = shape[(k * S + s) * 2];
                    const int32_t W = shape[(k * S + s) * 2 + 1];
                    footprint f;
                    double cw[4];
                    make_footprint(xy[0], xy[1], H, W, start[k * S + s], &f);
                    corner_weights(&f, cw);
                    const double lh = f.lh, lw = f.lw, hh = f.hh, hw = f.hw;
                    for (g = 0; g < G; ++g) {
                        const int64_t widx = (((ba * P + p) * K + k) * S + s) * G + g;
                        const double w = weights[widx];
                        double gw_sum = 0.0, gh_sum = 0.0, gweight = 0.0;
                        for (c = 0; c < D; ++c) {
                            const double go = grad_out[ba * C + (int64_t)g * D + c];
                            const double top_grad = go * w;
                            double v[4] = {0.0, 0.0, 0.0, 0.0};
                            for (i = 0; i < 4; ++i) {
                                if (f.row[i] < 0) continue;
                                const int64_t idx = (b * rows + f.row[i]) * C + (int64_t)g * D + c;
                                v[i] = feat_value(feat, feat_kind, idx);
                                gf[idx] += cw[i] * top_grad;
                            }
                            const double grad_w = lh * (v[3] - v[2]) + hh * (v[1] - v[0]);
                            const double grad_h = lw * (v[3] - v[1]) + hw * (v[2] - v[0]);
                            gw_sum += (double)W * grad_w * top_grad;
                            gh_sum += (double)H * grad_h * top_grad;
                            const double val = cw[0] * v[0] + cw[1] * v[1] + cw[2] * v[2] + cw[3] * v[3];
                            gweight += go * val;
                        }
                        gl[(p * K + k) * 2 + 0] += gw_sum;
                        gl[(p * K + k) * 2 + 1] += gh_sum;
                        grad_weight[widx - ba_begin * (int64_t)P * K * S * G] = (float)gweight;
                    }
                }
            }
        for (i = 0; i < P * K * 2; ++i) grad_loc[lba * P * K * 2 + i] = (float)gl[i];
    }
    int64_t e;
    for (e = 0; e < nfeat; ++e) grad_feat[e] = (float)gf[e];
    free(gf);
    free(gl);
    return DAO_OK;
}

/*
 * The DCNv4 form (page "DCNv4", "Defining the problem" and "Solving the
 * problem: 1"): every group g has its own sampling points and weights,
 *   y_g(p0) = sum_k m_gk x_g(p0 + p_k + dp_gk),
 * here with the points given as normalised locations, one per camera, valid
 * at every scale, and one weight per scale. The locations and weights share
 * one tensor lw [B, A, G, P, K, 2 + S] = (x, y, w_0 .. w_{S-1}).
 *   out[b,a,c] = sum over p,k,s of lw[b,a,g,p,k,2+s] *
 *                bilinear(map (b,k,s), lw[b,a,g,p,k,0..1], c),  g = c / (C/G).
 * The bilinear step and its precision are those of dao_forward.
 */
int dao_forward_fused(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                      const int32_t *shape, const int32_t *start,
                      const void *feat, int feat_kind, const float *lw, float *out)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    const int D = C / G;
    const int E = 2 + S;
    int64_t ba;
    for (ba = 0; ba < (int64_t)B * A; ++ba) {
        const int64_t b = ba / A;
        int g, p, k, s, c, i;
        for (g = 0; g < G; ++g) {
            double *acc = (double *)calloc((size_t)D, sizeof(double));
            if (!acc) return DAO_ERR_NOMEM;
            for (p = 0; p < P; ++p)
                for (k = 0; k < K; ++k) {
                    const float *e = lw + (((ba * G + g) * P + p) * K + k) * E;
                    for (s = 0; s < S; ++s) {
                        footprint f;
                        double cw[4];
                        make_footprint(e[0], e[1], shape[(k * S + s) * 2], shape[(k * S + s) * 2 + 1],
                                       start[k * S + s], &f);
                        corner_weights(&f, cw);
                        const double m = e[2 + s];
                        for (c = 0; c < D; ++c) {
                            double val = 0.0;
                            for (i = 0; i < 4; ++i)
                                if (f.row[i] >= 0)
                                    val += cw[i] * feat_value(feat, feat_kind,
                                                              (b * rows + f.row[i]) * C + (int64_t)g * D + c);
                            acc[c] += m * val;
                        }
                    }
                }
            for (c = 0; c < D; ++c) out[ba * C + (int64_t)g * D + c] = (float)acc[c];
            free(acc);
        }
    }
    return DAO_OK;
}

/*
 * Backward of the DCNv4 form: the gradients of §4.1 of the Sparse4D page,
 * kept per group. grad_lw has lw's layout: entries 0 and 1 hold dL/dx and
 * dL/dy (scaled by W and H, summed over the scales and the group's
 * channels), entry 2 + s holds dL/dw_s. grad_feat [B, rows, C] is written
 * in full.
 */
int dao_backward_fused(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                       const int32_t *shape, const int32_t *start,
                       const void *feat, int feat_kind, const float *lw, const float *grad_out,
                       float *grad_feat, float *grad_lw)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    const int D = C / G;
    const int E = 2 + S;
    const int64_t nfeat = (int64_t)B * rows * C;
    double *gf = (double *)calloc((size_t)(nfeat > 0 ? nfeat : 1), sizeof(double));
    if (!gf) return DAO_ERR_NOMEM;
    int64_t ba;
    for (ba = 0; ba < (int64_t)B * A; ++ba) {
        const int64_t b = ba / A;
        int g, p, k, s, c, i;
        for (g = 0; g < G; ++g)
            for (p = 0; p < P; ++p)
                for (k = 0; k < K; ++k) {
                    const int64_t eoff = (((ba * G + g) * P + p) * K + k) * E;
                    const float *e = lw + eoff;
                    double gx = 0.0, gy = 0.0;
                    for (s = 0; s < S; ++s) {
                        const int32_t H = shape[(k * S + s) * 2];
                        const int32_t W = shape[(k * S + s) * 2 + 1];
                        footprint f;
                        double cw[4];
                        make_footprint(e[0], e[1], H, W, start[k * S + s], &f);
                        corner_weights(&f, cw);
                        const double m = e[2 + s];
                        double gm = 0.0;
                        for (c = 0; c < D; ++c) {
                            const double go = grad_out[ba * C + (int64_t)g * D + c];
                            const double top_grad = go * m;
                            double v[4] = {0.0, 0.0, 0.0, 0.0};
                            for (i = 0; i < 4; ++i) {
                                if (f.row[i] < 0) continue;
                                const int64_t idx = (b * rows + f.row[i]) * C + (int64_t)g * D + c;
                                v[i] = feat_value(feat, feat_kind, idx);
                                gf[idx] += cw[i] * top_grad;
                            }
                            gx += (double)W * (f.lh * (v[3] - v[2]) + f.hh * (v[1] - v[0])) * top_grad;
                            gy += (double)H * (f.lw * (v[3] - v[1]) + f.hw * (v[2] - v[0])) * top_grad;
                            gm += go * (cw[0] * v[0] + cw[1] * v[1] + cw[2] * v[2] + cw[3] * v[3]);
                        }
                        grad_lw[eoff + 2 + s] = (float)gm;
                    }
                    grad_lw[eoff + 0] = (float)gx;
                    grad_lw[eoff + 1] = (float)gy;
                }
    }
    int64_t j;
    for (j = 0; j < nfeat; ++j) grad_feat[j] = (float)gf[j];
    free(gf);
    return DAO_OK;
}

/*
 * The step before the operator in Sparse4D (the Sparse4D page, §1 and §6:
 * each 3D anchor's key points are projected into every camera view). The
 * page prints no formula; the reading here is the pinhole projection by a
 * 4x4 matrix whose first three rows map a homogeneous point (X, Y, Z, 1) to
 * (u*d, v*d, d) in pixels, then a division by the image size:
 *   ud = ((m00*X + m01*Y) + m02*Z) + m03   (fp32: every product and sum
 *   vd, d likewise with rows 1 and 2        rounded, in this order)
 *   x = (ud / d) / image_w,  y = (vd / d) / image_h   (fp32 divisions)
 * A point with d <= 1e-5 (behind or on the camera plane) gets the location
 * (NaN, NaN), which reads nothing. The location decides which pixels are
 * read, so the kernel computes it with the same fp32 operations.
 * kp [B, A, P, 3], proj [B, K, 4, 4] row-major, loc [B, A, P, K, 2].
 */
static void project_point(const float *kp, const float *m, float image_w, float image_h, float *xy)
{
    float ud = ((m[0] * kp[0] + m[1] * kp[1]) + m[2] * kp[2]) + m[3];
    float vd = ((m[4] * kp[0] + m[5] * kp[1]) + m[6] * kp[2]) + m[7];
    float d = ((m[8] * kp[0] + m[9] * kp[1]) + m[10] * kp[2]) + m[11];
    if (!(d > 1e-5f)) {
        xy[0] = NAN;
        xy[1] = NAN;
        return;
    }
    float u = ud / d, v = vd / d;
    xy[0] = u / image_w;
    xy[1] = v / image_h;
}

int dao_project(int B, int K, int A, int P, const float *kp, const float *proj, float image_w, float image_h,
                float *loc)
{
    if (B < 0 || K < 0 || A < 0 || P < 0) return DAO_ERR_ARGS;
    int64_t b, a, p, k;
    for (b = 0; b < B; ++b)
        for (a = 0; a < A; ++a)
            for (p = 0; p < P; ++p)
                for (k = 0; k < K; ++k)
                    project_point(kp + ((b * A + a) * P + p) * 3, proj + (b * K + k) * 16, image_w, image_h,
                                  loc + (((b * A + a) * P + p) * K + k) * 2);
    return DAO_OK;
}

/*
 * Weights from logits: a softmax over the P*K*S samples of every (b, a, g),
 * the normalisation the Sparse4D head applies before the operator. In double,
 * rounded to fp32 at the end. logits and w are [B, A, P, K, S, G].
 */
int dao_softmax_weights(int B, int A, int P, int K, int S, int G, const float *logits, float *w)
{
    if (B < 0 || A < 0 || P < 0 || K < 0 || S < 0 || G <= 0) return DAO_ERR_ARGS;
    const int64_t n = (int64_t)P * K * S;
    int64_t ba, j;
    int g;
    for (ba = 0; ba < (int64_t)B * A; ++ba)
        for (g = 0; g < G; ++g) {
            double mx = -INFINITY, sum = 0.0;
            for (j = 0; j < n; ++j) {
                const double z = logits[(ba * n + j) * G + g];
                if (z > mx) mx = z;
            }
            for (j = 0; j < n; ++j) sum += exp((double)logits[(ba * n + j) * G + g] - mx);
            for (j = 0; j < n; ++j)
                w[(ba * n + j) * G + g] = (float)(exp((double)logits[(ba * n + j) * G + g] - mx) / sum);
        }
    return DAO_OK;
}

/*
 * Chain rule from the operator's gradients back to the key points and the
 * logits (double):
 *   grad_logits[b,a,p,k,s,g] = w * (grad_weight - sum over (p,k,s) of w * grad_weight),
 *     per (b, a, g), the derivative of the softmax;
 *   grad_kp[b,a,p,:] = sum over k of J_k^T grad_loc[b,a,p,k,:], with J_k the
 *     derivative of (x, y) above with respect to (X, Y, Z):
 *     dx/dX_i = (m0i * d - ud * m2i) / (d^2 * image_w),
 *     dy/dX_i = (m1i * d - vd * m2i) / (d^2 * image_h),
 *     and 0 for a point with d <= 1e-5.
 */
int dao_projected_chain(int B, int K, int S, int G, int A, int P, const float *kp, const float *proj,
                        float image_w, float image_h, const float *w, const float *grad_loc,
                        const float *grad_weight, float *grad_kp, float *grad_logits)
{
    if (B < 0 || K < 0 || S < 0 || G <= 0 || A < 0 || P < 0) return DAO_ERR_ARGS;
    const int64_t n = (int64_t)P * K * S;
    int64_t ba, j;
    int g, p, k, i;
    for (ba = 0; ba < (int64_t)B * A; ++ba) {
        for (g = 0; g < G; ++g) {
            double dot = 0.0;
            for (j = 0; j < n; ++j) dot += (double)w[(ba * n + j) * G + g] * grad_weight[(ba * n + j) * G + g];
            for (j = 0; j < n; ++j) {
                const int64_t e = (ba * n + j) * G + g;
                grad_logits[e] = (float)((double)w[e] * ((double)grad_weight[e] - dot));
            }
        }
        const int64_t b = ba / A;
        for (p = 0; p < P; ++p) {
            const float *x = kp + (ba * P + p) * 3;
            double acc[3] = {0.0, 0.0, 0.0};
            for (k = 0; k < K; ++k) {
                const float *m = proj + (b * K + k) * 16;
                const double ud = (double)m[0] * x[0] + (double)m[1] * x[1] + (double)m[2] * x[2] + m[3];
                const double vd = (double)m[4] * x[0] + (double)m[5] * x[1] + (double)m[6] * x[2] + m[7];
                const double d = (double)m[8] * x[0] + (double)m[9] * x[1] + (double)m[10] * x[2] + m[11];
                /* the validity test is the forward's fp32 one */
                const float d32 = (((m[8] * x[0] + m[9] * x[1]) + m[10] * x[2]) + m[11]);
                if (!(d32 > 1e-5f)) continue;
                const double gx = grad_loc[((ba * P + p) * K + k) * 2];
                const double gy = grad_loc[((ba * P + p) * K + k) * 2 + 1];
                for (i = 0; i < 3; ++i) {
                    const double dxd = (m[i] * d - ud * m[8 + i]) / (d * d * image_w);
                    const double dyd = (m[4 + i] * d - vd * m[8 + i]) / (d * d * image_h);
                    acc[i] += gx * dxd + gy * dyd;
                }
            }
            for (i = 0; i < 3; ++i) grad_kp[(ba * P + p) * 3 + i] = (float)acc[i];
        }
    }
    return DAO_OK;
}

/* Bilinear value of one channel at one location, for pin tests. */
double dao_bilinear(const float *map, int32_t H, int32_t W, int32_t C, int32_t c,
                    float x, float y)
{
    footprint f;
    double cw[4], v = 0.0;
    int i;
    make_footprint(x, y, H, W, 0, &f);
    corner_weights(&f, cw);
    for (i = 0; i < 4; ++i)
        if (f.row[i] >= 0) v += cw[i] * (double)map[f.row[i] * C + c];
    return v;
}

/*
 * Error-bound helper for the parity tests, not part of the operator.
 *
 * For each location (b,a,p,k) it returns the sum, over s, g and the group's
 * channels, of the absolute values of the products that make up grad_loc in
 * §4.1. mag[..,0] is that sum for the width component, mag[..,1] for the
 * height component:
 *   mag[..,0] = sum W * |top_grad| * (lh*(|v4|+|v3|) + hh*(|v2|+|v1|))
 *   mag[..,1] = sum H * |top_grad| * (lw*(|v4|+|v2|) + hw*(|v3|+|v1|))
 * A floating-point sum of these terms cannot be off by more than (number of
 * sequential roundings) * unit roundoff * mag.
 */
int dao_grad_loc_magnitude(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                           const int32_t *shape, const int32_t *start,
                           const void *feat, int feat_kind,
                           const float *loc, const float *weights, const float *grad_out,
                           int64_t ba_begin, int64_t ba_end, float *mag)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    if (ba_begin < 0 || ba_end < ba_begin || ba_end > (int64_t)B * A) return DAO_ERR_ARGS;
    const int D = C / G;
    int64_t ba;
    for (ba = ba_begin; ba < ba_end; ++ba) {
        const int64_t b = ba / A;
        int p, k, s, g, c, i;
        for (p = 0; p < P; ++p)
            for (k = 0; k < K; ++k) {
                const float *xy = loc + ((ba * P + p) * K + k) * 2;
                double mx = 0.0, my = 0.0;
                for (s = 0; s < S; ++s) {
                    const int32_t H = shape[(k * S + s) * 2];
                    const int32_t W = shape[(k * S + s) * 2 + 1];
                    footprint f;
                    make_footprint(xy[0], xy[1], H, W, start[k * S + s], &f);
                    for (g = 0; g < G; ++g) {
                        const double w = fabs((double)weights[(((ba * P + p) * K + k) * S + s) * G + g]);
                        for (c = 0; c < D; ++c) {
                            const double tg = fabs((double)grad_out[ba * C + (int64_t)g * D + c]) * w;
                            double v[4] = {0.0, 0.0, 0.0, 0.0};
                            for (i = 0; i < 4; ++i)
                                if (f.row[i] >= 0)
                                    v[i] = fabs(feat_value(feat, feat_kind,
                                                           (b * rows + f.row[i]) * C + (int64_t)g * D + c));
                            mx += (double)W * tg * (f.lh * (v[3] + v[2]) + f.hh * (v[1] + v[0]));
                            my += (double)H * tg * (f.lw * (v[3] + v[1]) + f.hw * (v[2] + v[0]));
                        }
                    }
                }
                mag[(((ba - ba_begin) * P + p) * K + k) * 2 + 0] = (float)mx;
                mag[(((ba - ba_begin) * P + p) * K + k) * 2 + 1] = (float)my;
            }
    }
    return DAO_OK;
}

/*
 * Records per feature row, an error-bound helper for the parity tests (not
 * a step of the operator).
 *
 * §4.1 scatters one product to each in-map corner of every sample; a row's
 * grad_feat entry is the sum of the products its row receives, one per
 * (anchor, point, camera, scale, corner) that lands there. count[b*rows + r]
 * is that number for feature row r of batch item b. Corners are decided by
 * the same fp32 footprint as the operator itself.
 */
int dao_row_counts(int B, int K, int S, int C, int G, int A, int P, int64_t rows,
                   const int32_t *shape, const int32_t *start, const float *loc, int32_t *count)
{
    if (!check_dims(B, K, S, C, G, A, P, rows, shape, start)) return DAO_ERR_ARGS;
    memset(count, 0, sizeof(int32_t) * (size_t)B * (size_t)rows);
    int64_t ba;
    for (ba = 0; ba < (int64_t)B * A; ++ba) {
        const int64_t b = ba / A;
        int p, k, s, i;
        for (p = 0; p < P; ++p)
            for (k = 0; k < K; ++k) {
                const float *xy = loc + ((ba * P + p) * K + k) * 2;
                for (s = 0; s < S; ++s) {
                    footprint f;
                    make_footprint(xy[0], xy[1], shape[(k * S + s) * 2], shape[(k * S + s) * 2 + 1],
                                   start[k * S + s], &f);
                    for (i = 0; i < 4; ++i)
                        if (f.row[i] >= 0) count[b * rows + f.row[i]] += 1;
                }
            }
    }
    return DAO_OK;
}
