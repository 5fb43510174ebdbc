/*
 * da.h: C ABI of the GB300 deformable-aggregation library (libda.so).
 *
 * The operator is Sparse4D's deformable aggregation. The page "Inside
 * Sparse4D's CUDA core: deformable_aggregation bilinear interpolation and
 * gradient back-propagation" (深入Sparse4D的CUDA核心：图解deformable_aggregation算子的双线性插值与梯度回传)
 * defines it:
 *   - §3.1: HWC feature layout;
 *   - §3.2: bilinear sampling with per-corner zeroing outside the map;
 *   - §4.1: the three gradients;
 *   - §5.1: the six-dimensional decomposition;
 *   - §6: the inputs of DeformableAggregationFunction and the packing done
 *     by feature_maps_format.
 *
 * Notation: B batch, K cameras, S scales, C channels (num_embeds),
 * G groups, D = C / G channels per group, A anchors, P points per anchor.
 * Map (k, s) has H x W pixels and starts at feature row level_start_index[k, s].
 *
 *   out[b,a,c] = sum_{p,k,s} weights[b,a,p,k,s,c/D] *
 *                bilinear(map (b,k,s), h = y*H - 0.5, w = x*W - 0.5, channel c)
 *
 * with (x, y) = sampling_location[b,a,p,k,0..1]; x is scaled by the width and
 * y by the height. A corner outside the map reads 0. No softmax or other
 * normalisation is applied to the weights: the DCNv4 page ("Solving the
 * problem: 1. remove softmax") treats them as unbounded reals.
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" point to memory the calling CUDA context can
 *     read or write from kernels. Pointers marked "host" point to ordinary
 *     host memory, read during the call only.
 *   - The caller owns every buffer; the library allocates nothing. The one
 *     exception is a da_pipeline (below): it owns the device buffers it
 *     allocates when it is created.
 *   - Work is enqueued on `stream`, or on the legacy default stream when it is
 *     NULL. The call returns without synchronising. Outputs are valid once the
 *     stream reaches that point.
 *   - Outputs are overwritten, never accumulated into.
 *   - Sizes may be 0 (B, A, P, K or S). An empty sum leaves zeros in the
 *     outputs. A pointer may be NULL only when its tensor has no elements.
 *   - Arguments are validated on the host before anything is enqueued. On any
 *     error nothing is enqueued and a non-zero da_status is returned;
 *     da_last_error() gives a one-line reason. The only exception is
 *     DA_ERR_CUDA, which a failed launch can return after part of the work was
 *     enqueued.
 *   - The library keeps no state between calls. Calls on different streams
 *     may run concurrently, provided they write to different buffers.
 */
#ifndef DA_H_
#define DA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here without the CUDA headers. */
typedef struct CUstream_st *da_stream_t;

typedef enum da_status {
    DA_OK = 0,
    DA_ERR_NULL = 1,        /* a required pointer is NULL */
    DA_ERR_SHAPE = 2,       /* sizes negative, inconsistent, or a map outside the feature rows */
    DA_ERR_ALIGN = 3,       /* a pointer is not aligned as required below */
    DA_ERR_UNSUPPORTED = 4, /* valid sizes this build has no kernel for (see da_forward) */
    DA_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed */
    DA_ERR_WORKSPACE = 6,   /* workspace too small or not 256-byte aligned */
    DA_ERR_DEVICE_BOUNDS = 7 /* bounds-checking builds only: see below */
} da_status;

/*
 * Bounds-checking builds (compiled with DA_DEBUG_BOUNDS; libda_debug.so).
 * Every index a kernel computes before it reads or writes device memory
 * (feature rows from the sampling locations, record slots from the binning,
 * anchors and sample ids decoded from records, d entries, output elements,
 * source pixels of the warpaffine kernels) is checked against the extent of
 * its tensor first. An index outside it is not used: the access is skipped,
 * and the kernel sets a bit for the kind of index in a device error word.
 * Nothing traps, so the context stays usable. After enqueueing its work,
 * each entry point of such a build waits for its stream, reads the word
 * (then clears it) and returns DA_ERR_DEVICE_BOUNDS if a bit was set;
 * da_last_error() names the kinds. A call made while its stream is being
 * captured into a CUDA graph skips that wait; the next call outside a
 * capture reports what it set. Release builds contain none of this.
 */

typedef enum da_dtype {
    DA_F32 = 0,  /* IEEE binary32 features */
    DA_BF16 = 1, /* bfloat16 features; all arithmetic and every other tensor stay fp32 */
    DA_F16 = 2   /* IEEE binary16 features (the half precision of the DCNv4 page,
                    "Solving the problem: 2"); arithmetic and other tensors fp32 */
} da_dtype;

typedef struct da_dims {
    int32_t batch;        /* B >= 0 */
    int32_t num_cams;     /* K >= 0 */
    int32_t num_scales;   /* S >= 0; K*S <= DA_MAX_MAPS */
    int32_t num_embeds;   /* C >= 1 */
    int32_t num_groups;   /* G >= 1, C % G == 0 */
    int32_t num_anchors;  /* A >= 0 */
    int32_t num_pts;      /* P >= 0 */
    int32_t feat_dtype;   /* a da_dtype */
    int64_t num_feat_rows;/* feature rows per batch item, 0 <= rows <= DA_MAX_ROWS */
} da_dims;

#define DA_MAX_MAPS 64              /* largest K*S */
#define DA_MAX_MAP_SIDE (1 << 24)   /* largest H or W */
#define DA_MAX_ROWS (1 << 30)       /* largest num_feat_rows; row indices stay in int32 */

/*
 * Forward pass: the sampling and weighting of page §3.2, summed over the
 * dimensions of page §5.1.
 *
 *   mc_ms_feat        device [B, num_feat_rows, C], feat_dtype, 16-byte aligned.
 *                     Row level_start_index[k,s] + i*W + j holds pixel (i, j)
 *                     of map (k, s) (HWC, page §3.1).
 *   spatial_shape     host   [K, S, 2] int32: (H, W) of each map, 1..DA_MAX_MAP_SIDE.
 *   level_start_index host   [K, S] int32: first row of each map. The map must
 *                     fit: start + H*W <= num_feat_rows. Maps may overlap.
 *   sampling_location device [B, A, P, K, 2] fp32, (x, y) normalised to the
 *                     image, 8-byte aligned. The same (x, y) serves every scale.
 *   weights           device [B, A, P, K, S, G] fp32, 4-byte aligned.
 *   out               device [B, A, C] fp32, 16-byte aligned; overwritten.
 *
 * Supported: D * sizeof(feature) in {16, 32, 64, 128} bytes. That is D in
 * {4, 8, 16, 32} for fp32 and D in {8, 16, 32, 64} for bf16 and fp16. Other D return
 * DA_ERR_UNSUPPORTED.
 * Arithmetic: h = y*H - 0.5 and w = x*W - 0.5 are each rounded twice (a
 * product, then a difference; no fused multiply-add). Corner weights and sums
 * are fp32.
 */
da_status da_forward(const da_dims *dims,
                     const void *mc_ms_feat,
                     const int32_t *spatial_shape,
                     const int32_t *level_start_index,
                     const float *sampling_location,
                     const float *weights,
                     float *out,
                     da_stream_t stream);

/*
 * Size in bytes of the device workspace that the binned path of da_backward
 * needs for `dims` (stored in *bytes). It depends on the sizes only:
 * about 4*B*A*P*K*S*(8.5 + 4*G) bytes plus 4 bytes per feature row. This
 * is about 277 MB for B=6, A=900, P=13, K=6, S=4, G=8. The same workspace
 * serves both modes of da_backward_ex.
 * Returns DA_ERR_UNSUPPORTED when 4*B*A*P*K*S or B*num_feat_rows does not
 * fit in int32. It also returns DA_ERR_UNSUPPORTED unless C is a power of
 * two in [8, 256] and D is a multiple of 8. The scatter path (no workspace)
 * still serves such sizes.
 */
da_status da_backward_workspace_size(const da_dims *dims, size_t *bytes);

/*
 * Backward pass: the three gradients of page §4.1, for a loss L with
 * dL/d out = grad_out.
 *
 *   inputs as for da_forward, plus
 *   grad_out    device [B, A, C] fp32, 16-byte aligned.
 *   grad_feat   device [B, num_feat_rows, C] fp32 for both feature types,
 *               16-byte aligned; overwritten. Rows outside every map get 0.
 *               Contributions are summed in an unspecified order, so the
 *               bits may differ from run to run (see da_backward_ex for a
 *               deterministic mode).
 *   grad_loc    device [B, A, P, K, 2] fp32, 4-byte aligned; overwritten.
 *               [...,0] is dL/dx (scaled by W), [...,1] is dL/dy (scaled by H).
 *   grad_weight device [B, A, P, K, S, G] fp32, 4-byte aligned; overwritten.
 *   workspace   device scratch of at least da_backward_workspace_size bytes,
 *               256-byte aligned, owned by the caller and not read
 *               afterwards; or NULL with workspace_bytes = 0.
 *
 * With a workspace (the binned path), the corner contributions are sorted by
 * feature row, and every grad_feat row is computed once by the lanes that
 * own it. There is no zero-fill and no atomic scatter.
 * Without one (the scatter path), grad_feat is zero-filled and then scattered
 * into with 16-byte vector reductions. That path is slower at large sizes
 * but needs no scratch.
 * Both paths write grad_loc and grad_weight exactly once per element.
 * Calls that share one workspace must not overlap on the GPU.
 */
da_status da_backward(const da_dims *dims,
                      const void *mc_ms_feat,
                      const int32_t *spatial_shape,
                      const int32_t *level_start_index,
                      const float *sampling_location,
                      const float *weights,
                      const float *grad_out,
                      float *grad_feat,
                      float *grad_loc,
                      float *grad_weight,
                      void *workspace,
                      size_t workspace_bytes,
                      da_stream_t stream);

/*
 * da_backward_ex: da_backward with option flags.
 *
 *   DA_BACKWARD_DETERMINISTIC  grad_feat, grad_loc and grad_weight are the
 *       same bit for bit on every run with the same inputs and sizes. Needs
 *       the binned path (a workspace); without one the call returns
 *       DA_ERR_WORKSPACE. The corner contributions of every feature row are
 *       put in a fixed order (by sample and corner) before they are summed.
 *       This costs four more kernels: about a sixth more backward time
 *       at the 6-camera Sparse4D training shape, more when many samples
 *       crowd a few pixels.
 *
 * Other arguments are those of da_backward. Unknown flags give
 * DA_ERR_SHAPE. da_backward(...) is da_backward_ex(..., 0, stream). With
 * DA_BACKWARD_BINNED_READY, DA_BACKWARD_DETERMINISTIC has no further effect
 * (the order was fixed, or not, by da_backward_bin).
 */
#define DA_BACKWARD_DETERMINISTIC 1u
/*
 *   DA_BACKWARD_BINNED_READY  the workspace already holds the binning of
 *       these sampling locations, made by da_backward_bin (with the same
 *       dims, map tables and locations, and DA_BACKWARD_DETERMINISTIC there
 *       if a fixed order is wanted); only the steps that need grad_out run.
 *       The call must be ordered after that da_backward_bin on the GPU.
 */
#define DA_BACKWARD_BINNED_READY 2u
da_status da_backward_ex(const da_dims *dims,
                         const void *mc_ms_feat,
                         const int32_t *spatial_shape,
                         const int32_t *level_start_index,
                         const float *sampling_location,
                         const float *weights,
                         const float *grad_out,
                         float *grad_feat,
                         float *grad_loc,
                         float *grad_weight,
                         void *workspace,
                         size_t workspace_bytes,
                         uint32_t flags,
                         da_stream_t stream);

/*
 * The DCNv4 form: per-group locations, fused with the weights in one tensor.
 *
 * The DCNv4 page ("Defining the problem") writes the operator as
 * y_g(p0) = sum_k m_gk x_g(p0 + p_k + dp_gk): every group g of channels has
 * its own sampling points and weights. Its step "Solving the problem: 1"
 * produces offsets and weights with one linear layer, so they arrive in one
 * tensor. Here, in the dimensions above:
 *
 *   loc_weight  device [B, A, G, P, K, 2 + S] fp32, 4-byte aligned. The entry
 *               of (b, a, g, p, k) is (x, y, w_0, ..., w_{S-1}): the
 *               normalised location of point p in camera k for group g (the
 *               same at every scale), and its weight at each scale.
 *   out[b,a,c]  = sum_{p,k,s} w_s(b,a,g,p,k) *
 *                 bilinear(map (b,k,s), (x, y)(b,a,g,p,k), channel c),
 *               with g = c / D; the bilinear step is da_forward's.
 *
 * Turning DCNv4's pixel offsets p0 + p_k + dp_gk into normalised locations
 * is the caller's step: (x, y) = ((j + 0.5) / W, (i + 0.5) / H) for pixel
 * (i, j), so a location on a pixel centre reads that pixel exactly.
 *
 * da_forward_fused: arguments and rules of da_forward, with loc_weight in
 * place of sampling_location and weights.
 *
 * da_backward_fused: arguments and rules of da_backward, with
 * grad_loc_weight [B, A, G, P, K, 2 + S] fp32 (4-byte aligned, overwritten)
 * in place of grad_loc and grad_weight: entries 0, 1 hold dL/dx, dL/dy
 * (scaled by W and H, summed over the scales and the group's channels) and
 * entry 2 + s holds dL/dw_s. With a workspace of at least
 * da_backward_fused_workspace_size bytes it takes the binned path, which
 * treats the D channels of each (pixel, group) as a row of their own and
 * each (anchor, group) as an anchor; it needs D a power of two in [8, 256]
 * (else DA_ERR_UNSUPPORTED). Without one, the scatter path.
 *
 * da_backward_fused_workspace_size: the binned path's workspace for dims,
 * about 4*B*A*G*P*K*S*12.5 bytes plus 4*G bytes per feature row.
 */
da_status da_backward_fused_workspace_size(const da_dims *dims, size_t *bytes);
da_status da_forward_fused(const da_dims *dims,
                           const void *mc_ms_feat,
                           const int32_t *spatial_shape,
                           const int32_t *level_start_index,
                           const float *loc_weight,
                           float *out,
                           da_stream_t stream);

da_status da_backward_fused(const da_dims *dims,
                            const void *mc_ms_feat,
                            const int32_t *spatial_shape,
                            const int32_t *level_start_index,
                            const float *loc_weight,
                            const float *grad_out,
                            float *grad_feat,
                            float *grad_loc_weight,
                            void *workspace,
                            size_t workspace_bytes,
                            da_stream_t stream);

/*
 * The step before the operator, fused into it (the projected layout).
 *
 * The Sparse4D page (§1, §6) projects each 3D anchor's key points into every
 * camera view before the aggregation, and the Sparse4D head normalises the
 * weights with a softmax. Here the forward kernel does both while it builds
 * the samples, so no location or weight tensor has to be written and read
 * back in between:
 *   keypoints     device [B, A, P, 3] fp32 (X, Y, Z), 4-byte aligned.
 *   projection    device [B, K, 4, 4] fp32 row-major: rows 0..2 map
 *                 (X, Y, Z, 1) to (u*d, v*d, d) in pixels; row 3 is unused.
 *   image_w, image_h  the image size in pixels (> 0).
 *   weight_logits device [B, A, P, K, S, G] fp32, 4-byte aligned.
 * The page gives no formula; the reading is the pinhole projection:
 *   ud = ((m00*X + m01*Y) + m02*Z) + m03, vd and d likewise (rows 1, 2),
 *   x = (ud / d) / image_w, y = (vd / d) / image_h,
 * every step an fp32 operation rounded in this order (no fused
 * multiply-add), because the location decides which pixels are read. A key
 * point with d <= 1e-5 (behind the camera) gets the location (NaN, NaN) and
 * reads nothing. weights = softmax of the logits over the P*K*S samples of
 * each (b, a, g). Then out is da_forward's.
 *
 * da_forward_projected also writes the locations [B, A, P, K, 2] and the
 * weights [B, A, P, K, S, G] it used when sampling_location / weights are
 * not NULL (the backward needs them).
 *
 * da_backward_projected takes those two tensors, runs da_backward_ex on
 * them (grad_feat, grad_loc, grad_weight, workspace and flags as there), and
 * then the chain rule:
 *   grad_logits    [B, A, P, K, S, G]: w * (grad_weight - sum over
 *                  (p, k, s) of w * grad_weight), per (b, a, g);
 *   grad_keypoints [B, A, P, 3]: sum over k of J_k^T grad_loc[b,a,p,k,:],
 *                  J_k the derivative of (x, y) above; 0 for cameras the
 *                  point is behind.
 * grad_loc and grad_weight are outputs too (the chain rule reads them).
 */
da_status da_forward_projected(const da_dims *dims,
                               const void *mc_ms_feat,
                               const int32_t *spatial_shape,
                               const int32_t *level_start_index,
                               const float *keypoints,
                               const float *projection,
                               float image_w,
                               float image_h,
                               const float *weight_logits,
                               float *out,
                               float *sampling_location,
                               float *weights,
                               da_stream_t stream);

da_status da_backward_projected(const da_dims *dims,
                                const void *mc_ms_feat,
                                const int32_t *spatial_shape,
                                const int32_t *level_start_index,
                                const float *keypoints,
                                const float *projection,
                                float image_w,
                                float image_h,
                                const float *sampling_location,
                                const float *weights,
                                const float *grad_out,
                                float *grad_feat,
                                float *grad_loc,
                                float *grad_weight,
                                float *grad_keypoints,
                                float *grad_logits,
                                void *workspace,
                                size_t workspace_bytes,
                                uint32_t flags,
                                da_stream_t stream);

/*
 * da_backward_bin: the first half of the binned backward, the part that
 * depends on the sampling locations only: it sorts the corner contributions
 * by feature row into the workspace (counts, prefix sums, records, and with
 * DA_BACKWARD_DETERMINISTIC the fixed order inside each row). A later
 * da_backward_ex with DA_BACKWARD_BINNED_READY and the same workspace does
 * the rest. The pages have no counterpart: it lets a training step run the
 * binning on another stream while da_forward runs, since neither needs the
 * other's results.
 *   dims, spatial_shape, level_start_index, sampling_location: as for
 *   da_backward (mc_ms_feat, weights and grad_out are not read).
 *   workspace, workspace_bytes: as for da_backward's binned path.
 * The workspace must not be in use by another call on the GPU meanwhile.
 */
da_status da_backward_bin(const da_dims *dims,
                          const int32_t *spatial_shape,
                          const int32_t *level_start_index,
                          const float *sampling_location,
                          void *workspace,
                          size_t workspace_bytes,
                          uint32_t flags,
                          da_stream_t stream);

/*
 * da_backward_noalloc: the binned backward, with its scratch in a fixed
 * array of DA_NOALLOC_SCRATCH_BYTES that the library carries in device
 * memory. No call allocates anything.
 *
 * The pages have no counterpart to this entry point. It exists for callers
 * that cannot call cudaMalloc. Examples: a runtime that fixes its device
 * memory at start-up and forbids later allocation; a plug-in whose host
 * framework owns all device memory and hands it no allocator; code that
 * cannot accept the device-wide synchronisation an allocation may cause.
 * They still pass their own inputs and outputs, exactly as for da_backward.
 *
 * Arguments, layouts and results are those of da_backward. Rules:
 *   - The scratch array exists once per device that loads the library and is
 *     held until the process exits.
 *   - Every call looks up the array's device address in the current
 *     context. The first call on a device may also load the library's device
 *     code there (a one-time set-up per device): make that first call before
 *     any stream capture. Because the address is not cached, a device reset
 *     between calls is safe: the next call finds the array where the new
 *     context put it (its contents start over).
 *   - Problems whose workspace (da_backward_workspace_size) exceeds
 *     DA_NOALLOC_SCRATCH_BYTES are rejected with DA_ERR_WORKSPACE. The limit
 *     fits e.g. the 6-camera Sparse4D shape at B = 1 (about 46 MB); the
 *     B = 6 training shape needs about 277 MB and must use da_backward.
 *   - Every call uses the same array. Each call clears what must start at
 *     zero, so a call does not depend on what the last one left there.
 *   - Calls that overlap on the GPU (on different streams, or from
 *     different threads without ordering) race on the array and give wrong
 *     results. Order them on one stream.
 */
#define DA_NOALLOC_SCRATCH_BYTES (64u << 20)
da_status da_backward_noalloc(const da_dims *dims,
                              const void *mc_ms_feat,
                              const int32_t *spatial_shape,
                              const int32_t *level_start_index,
                              const float *sampling_location,
                              const float *weights,
                              const float *grad_out,
                              float *grad_feat,
                              float *grad_loc,
                              float *grad_weight,
                              da_stream_t stream);

/*
 * Host pipeline: the forward (and backward) of a sequence of problems of one
 * shape whose tensors live in HOST memory.
 *
 * The pages do not describe this part. It is the path for callers whose data
 * sits in host memory: every step copies its inputs to the device, runs
 * da_forward (and da_backward), and copies the outputs back. The pipeline
 * keeps `depth` sets of device buffers and three CUDA streams (copy in,
 * compute, copy out). Step n uses buffer set n % depth, so step n's input
 * copy and step n-1's output copy run while a third step computes, and the
 * two copy directions share the host link at once.
 *
 * da_pipeline_create
 *   dims, spatial_shape, level_start_index: as for da_forward (host arrays,
 *     copied; the caller may free them afterwards).
 *   with_backward: 0 = forward only; 1 = forward, then backward.
 *   depth: buffer sets, 1 to 4. depth 1 serialises copies and compute; 2 is
 *     enough to overlap them.
 *   *pipeline receives the new pipeline.
 *   Works on the CUDA device that is current when it is called. It allocates
 *   depth * (inputs + outputs + backward workspace) bytes of device memory
 *   with cudaMalloc. With a backward, the binned path of da_backward is used
 *   when the sizes allow it (see da_backward_workspace_size), and the scatter
 *   path otherwise. Sizes are validated before any CUDA call.
 *
 * da_pipeline_submit
 *   Host pointers with the layouts of da_forward and da_backward:
 *   mc_ms_feat, sampling_location, weights, grad_out (inputs) and out,
 *   grad_feat, grad_loc, grad_weight (outputs). Without a backward, grad_out
 *   and the three gradients are ignored and may be NULL. A pointer may be
 *   NULL only when its tensor has no elements.
 *   Enqueues one step and returns. It does not wait when every host buffer
 *   is page-locked (cudaHostAlloc, cudaHostRegister); with pageable memory
 *   the copies may block the caller. Do not change the step's input buffers
 *   or read its output buffers until da_pipeline_sync returns.
 *
 * da_pipeline_sync
 *   Waits until every submitted step has finished and its outputs are in host
 *   memory.
 *
 * da_pipeline_destroy
 *   Waits like da_pipeline_sync, then frees the device buffers, streams and
 *   events. NULL is accepted and ignored.
 *
 * A pipeline is not thread-safe: one thread at a time. After DA_ERR_CUDA
 * from submit or sync, the pipeline refuses further steps with DA_ERR_CUDA;
 * destroy it.
 */
typedef struct da_pipeline da_pipeline;

da_status da_pipeline_create(const da_dims *dims,
                             const int32_t *spatial_shape,
                             const int32_t *level_start_index,
                             int32_t with_backward,
                             int32_t depth,
                             da_pipeline **pipeline);

da_status da_pipeline_submit(da_pipeline *pipeline,
                             const void *mc_ms_feat,
                             const float *sampling_location,
                             const float *weights,
                             const float *grad_out,
                             float *out,
                             float *grad_feat,
                             float *grad_loc,
                             float *grad_weight);

da_status da_pipeline_sync(da_pipeline *pipeline);

da_status da_pipeline_destroy(da_pipeline *pipeline);

/* Static name of a status code. */
const char *da_status_string(da_status status);

/* One-line reason for the last non-OK status returned on this thread. The
 * pointer stays valid until the next call on this thread. */
const char *da_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int32_t da_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DA_H_ */
