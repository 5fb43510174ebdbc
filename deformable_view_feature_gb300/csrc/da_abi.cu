// extern "C" entry points of libda.so (declared in include/da.h): host-side
// argument validation, then kernel launches on the caller's stream.
//
// The interface mirrors the autograd function DeformableAggregationFunction of
// the page "Inside Sparse4D's CUDA core", §6:
// (mc_ms_feat, spatial_shape, scale_start_index, sampling_location, weights).
// Here the start index is called level_start_index, the two small map tables
// are host arrays (so the host can check every map against the feature rows
// without a device round trip), and the sizes travel in da_dims.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "da_internal.cuh"

// Scratch of da_backward_noalloc: a fixed array in device memory, present
// on every device that loads the library. In host code its name only stands
// in for it; the device address comes from cudaGetSymbolAddress, called
// with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DA_NOALLOC_SCRATCH_BYTES];

#ifdef DA_DEBUG_BOUNDS
// Error word of the bounds-checking build: one bit per kind of index that a
// kernel found outside its tensor (da_bounds.h).
static __device__ uint32_t g_bounds_word;
#endif

namespace da {

namespace {
thread_local char g_err[256] = "";
}  // namespace

da_status fail(da_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

const char *last_error() { return g_err; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

da_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(DA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#ifdef DA_DEBUG_BOUNDS
uint32_t *bounds_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_bounds_word) == cudaSuccess ? static_cast<uint32_t *>(p) : nullptr;
}

da_status bounds_report(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "bounds check: cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone) return DA_OK;  // reported by the next call outside the capture
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "bounds check: stream synchronize");
    uint32_t v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_bounds_word, sizeof v)) != cudaSuccess)
        return cuda_fail(e, "bounds check: read of the error word");
    if (v == 0) return DA_OK;
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof zero)) != cudaSuccess)
        return cuda_fail(e, "bounds check: clear of the error word");
    static const char *names[] = {"feature row", "output element", "record slot", "anchor",
                                  "sample id", "row counter", "shared table entry", "source pixel"};
    char buf[200] = "";
    for (int i = 0; i < 8; ++i)
        if (v & (1u << i)) {
            std::strncat(buf, buf[0] ? ", " : "", sizeof buf - std::strlen(buf) - 1);
            std::strncat(buf, names[i], sizeof buf - std::strlen(buf) - 1);
        }
    return fail(DA_ERR_DEVICE_BOUNDS, "a kernel computed an index outside its tensor (%s); the accesses were skipped",
                buf);
}
#else
uint32_t *bounds_word() { return nullptr; }
da_status bounds_report(cudaStream_t) { return DA_OK; }
#endif

da_status prepare_shape(const da_dims *dims, const int32_t *spatial_shape, const int32_t *level_start_index,
                        Problem &pb, int &chunks)
{
    if (!dims) return fail(DA_ERR_NULL, "dims is NULL");
    const da_dims d = *dims;
    if (d.batch < 0 || d.num_cams < 0 || d.num_scales < 0 || d.num_anchors < 0 || d.num_pts < 0)
        return fail(DA_ERR_SHAPE, "negative size in dims");
    if (d.num_embeds < 1 || d.num_groups < 1 || d.num_embeds % d.num_groups != 0)
        return fail(DA_ERR_SHAPE, "num_embeds (%d) must be a positive multiple of num_groups (%d)",
                    d.num_embeds, d.num_groups);
    if (d.feat_dtype != DA_F32 && d.feat_dtype != DA_BF16 && d.feat_dtype != DA_F16)
        return fail(DA_ERR_SHAPE, "unknown feat_dtype %d", d.feat_dtype);
    if (d.num_feat_rows < 0 || d.num_feat_rows > DA_MAX_ROWS)
        return fail(DA_ERR_SHAPE, "num_feat_rows %lld outside [0, %d]",
                    static_cast<long long>(d.num_feat_rows), DA_MAX_ROWS);
    const int64_t nmaps = static_cast<int64_t>(d.num_cams) * d.num_scales;
    if (nmaps > DA_MAX_MAPS)
        return fail(DA_ERR_UNSUPPORTED, "num_cams*num_scales = %lld exceeds %d",
                    static_cast<long long>(nmaps), DA_MAX_MAPS);
    const int D = d.num_embeds / d.num_groups;
    const int elem = d.feat_dtype == DA_F32 ? 4 : 2;
    const int row_bytes = D * elem;
    if (row_bytes != 16 && row_bytes != 32 && row_bytes != 64 && row_bytes != 128)
        return fail(DA_ERR_UNSUPPORTED, "group width D*elem = %d bytes; supported: 16, 32, 64, 128",
                    row_bytes);
    chunks = row_bytes / 16;

    const int64_t num_ba = static_cast<int64_t>(d.batch) * d.num_anchors;
    const int64_t pks = static_cast<int64_t>(d.num_pts) * nmaps;
    if (num_ba > INT32_MAX || pks > INT32_MAX || num_ba * d.num_cams > INT32_MAX ||
        static_cast<int64_t>(d.num_pts) * d.num_cams > INT32_MAX)
        return fail(DA_ERR_UNSUPPORTED, "batch*anchors*cams or pts*cams*scales exceeds int32");

    if (nmaps > 0 && (!spatial_shape || !level_start_index))
        return fail(DA_ERR_NULL, "spatial_shape / level_start_index is NULL");
    for (int64_t i = 0; i < nmaps; ++i) {
        const int32_t H = spatial_shape[2 * i], W = spatial_shape[2 * i + 1];
        const int32_t st = level_start_index[i];
        if (H < 1 || W < 1 || H > DA_MAX_MAP_SIDE || W > DA_MAX_MAP_SIDE)
            return fail(DA_ERR_SHAPE, "map %lld has shape %d x %d", static_cast<long long>(i), H, W);
        if (st < 0 || static_cast<int64_t>(st) + static_cast<int64_t>(H) * W > d.num_feat_rows)
            return fail(DA_ERR_SHAPE, "map %lld (start %d, %d x %d) does not fit in %lld feature rows",
                        static_cast<long long>(i), st, H, W, static_cast<long long>(d.num_feat_rows));
        pb.maps[i] = da::MapInfo{H, W, st, 0};
    }
    pb.rows = d.num_feat_rows;
    pb.B = d.batch;
    pb.A = d.num_anchors;
    pb.P = d.num_pts;
    pb.K = d.num_cams;
    pb.S = d.num_scales;
    pb.C = d.num_embeds;
    pb.G = d.num_groups;
    pb.D = D;
    pb.pks = static_cast<int32_t>(pks);
    pb.pk = d.num_pts * d.num_cams;
    pb.num_ba = static_cast<int32_t>(num_ba);
    pb.anchors_per_cta = d.num_groups < da::kWarps ? da::kWarps / d.num_groups : 1;
    pb.nmaps = static_cast<int32_t>(nmaps);
    pb.gsplit = 1;
    pb.div_S = da::FastDiv::make(d.num_scales > 0 ? d.num_scales : 1);
    pb.div_K = da::FastDiv::make(d.num_cams > 0 ? d.num_cams : 1);
    pb.div_G = da::FastDiv::make(d.num_groups);
    pb.div_A = da::FastDiv::make(d.num_anchors > 0 ? d.num_anchors : 1);
    pb.div_P = da::FastDiv::make(d.num_pts > 0 ? d.num_pts : 1);
    pb.div_PKS = da::FastDiv::make(pks > 0 ? static_cast<uint32_t>(pks) : 1);
    pb.div_rows = da::FastDiv::make(d.num_feat_rows > 0 ? static_cast<uint32_t>(d.num_feat_rows) : 1);
    pb.dbg_err = bounds_word();
    return DA_OK;
}

}  // namespace da

namespace {

using da::aligned;
using da::cuda_fail;
using da::fail;

// Checks shared by both passes; fills the kernel's Problem and the chunk count.
da_status prepare(const da_dims *dims, const void *feat, const int32_t *spatial_shape,
                  const int32_t *level_start_index, const float *loc, const float *weights,
                  da::Problem &pb, int &chunks)
{
    da_status st = da::prepare_shape(dims, spatial_shape, level_start_index, pb, chunks);
    if (st != DA_OK) return st;
    const da_dims d = *dims;
    const int64_t num_ba = pb.num_ba;
    const int64_t pks = pb.pks;
    const int64_t n_feat = static_cast<int64_t>(d.batch) * d.num_feat_rows * d.num_embeds;
    const int64_t n_samp = num_ba * pks;
    if (n_feat > 0 && !feat) return fail(DA_ERR_NULL, "mc_ms_feat is NULL");
    if (n_samp > 0 && (!loc || !weights)) return fail(DA_ERR_NULL, "sampling_location / weights is NULL");
    if (!aligned(feat, 16)) return fail(DA_ERR_ALIGN, "mc_ms_feat must be 16-byte aligned");
    if (!aligned(loc, 8)) return fail(DA_ERR_ALIGN, "sampling_location must be 8-byte aligned");
    if (!aligned(weights, 4)) return fail(DA_ERR_ALIGN, "weights must be 4-byte aligned");

    pb.feat = feat;
    pb.loc = loc;
    pb.weights = weights;
    return DA_OK;
}

// Layout of the binned backward's workspace; DA_ERR_UNSUPPORTED when its
// record indices would not fit in int32.
da_status binned_layout(const da_dims &d, da::BinLayout &L)
{
    L = da::bin_layout(d.batch, d.num_feat_rows, d.num_anchors, d.num_pts, d.num_cams, d.num_scales,
                       d.num_groups);
    if (L.ncap > INT32_MAX || L.rows_total + da::kScanTile > INT32_MAX)
        return fail(DA_ERR_UNSUPPORTED, "binned backward: 4*B*A*P*K*S = %lld or B*rows = %lld exceeds int32",
                    static_cast<long long>(L.ncap), static_cast<long long>(L.rows_total));
    if (!da::binned_supported(d.num_embeds, d.num_embeds / d.num_groups))
        return fail(DA_ERR_UNSUPPORTED,
                    "binned backward: needs num_embeds a power of two in [8, 256] and num_embeds/num_groups "
                    "a multiple of 8 (got %d, %d)",
                    d.num_embeds, d.num_embeds / d.num_groups);
    return DA_OK;
}

// The part of both forward entry points after the layout-specific checks.
da_status forward_impl(const da_dims &d, da::FwdArgs &a, int chunks, float *out, da_stream_t stream)
{
    const int64_t n_out = static_cast<int64_t>(a.pb.num_ba) * a.pb.C;
    if (n_out > 0 && !out) return fail(DA_ERR_NULL, "out is NULL");
    if (!aligned(out, 16)) return fail(DA_ERR_ALIGN, "out must be 16-byte aligned");
    a.out = out;
    if (n_out == 0) return DA_OK;
    const cudaError_t e = da::launch_forward(a, d.feat_dtype, chunks, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return da::bounds_report(reinterpret_cast<cudaStream_t>(stream));
}

// The part of every backward entry point after the layout-specific checks
// (a.grad_loc and a.grad_weight are set and checked).
da_status backward_impl(const da_dims &d, da::BwdArgs &a, int chunks, const float *grad_out, float *grad_feat,
                        void *workspace, size_t workspace_bytes, uint32_t flags, da_stream_t stream)
{
    if (flags & ~static_cast<uint32_t>(DA_BACKWARD_DETERMINISTIC | DA_BACKWARD_BINNED_READY))
        return fail(DA_ERR_SHAPE, "unknown flags 0x%x", flags);
    const bool deterministic = (flags & DA_BACKWARD_DETERMINISTIC) != 0;
    const bool ready = (flags & DA_BACKWARD_BINNED_READY) != 0;
    if ((deterministic || ready) && !workspace && !workspace_bytes)
        return fail(DA_ERR_WORKSPACE, "DA_BACKWARD_DETERMINISTIC / DA_BACKWARD_BINNED_READY need the binned "
                                      "path's workspace");
    const da::Problem &pb = a.pb;
    const int64_t n_out = static_cast<int64_t>(pb.num_ba) * pb.C;
    const int64_t n_gf = static_cast<int64_t>(pb.B) * pb.rows * pb.C;
    if (n_out > 0 && !grad_out) return fail(DA_ERR_NULL, "grad_out is NULL");
    if (n_gf > 0 && !grad_feat) return fail(DA_ERR_NULL, "grad_feat is NULL");
    if (!aligned(grad_out, 16)) return fail(DA_ERR_ALIGN, "grad_out must be 16-byte aligned");
    if (!aligned(grad_feat, 16)) return fail(DA_ERR_ALIGN, "grad_feat must be 16-byte aligned");
    // The per-CTA grad_loc staging area of the scatter path must fit in
    // shared memory.
    const size_t smem = da::scatter_smem_bytes(pb);
    if (smem > 200 * 1024)
        return fail(DA_ERR_UNSUPPORTED, "num_pts = %d too large for the grad_loc staging area", pb.P);
    a.grad_out = grad_out;
    a.grad_feat = grad_feat;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (workspace || workspace_bytes) {
        da::BinLayout L;
        da_status st = binned_layout(d, L);
        if (st != DA_OK) return st;
        if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.bytes)
            return fail(DA_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes (got %zu)",
                        L.bytes, workspace_bytes);
        char *ws = static_cast<char *>(workspace);
        da::BinArgs w{};
        w.row_off = reinterpret_cast<int32_t *>(ws + L.off_row_off);
        w.tile_sum = reinterpret_cast<int32_t *>(ws + L.off_tile_sum);
        w.rec = reinterpret_cast<int2 *>(ws + L.off_rec);
        w.dpix = reinterpret_cast<float *>(ws + L.off_dpix);
        w.left = reinterpret_cast<int32_t *>(ws + L.off_left);
        w.left_count = w.row_off + L.ntiles * da::kScanTile + 1;
        w.rows_total = L.rows_total;
        w.nsid = L.nsid;
        w.ncap = L.ncap;
        w.ntiles = L.ntiles;
        if (deterministic) {
            w.sort_lists = reinterpret_cast<int32_t *>(ws + L.off_lists);
            w.sort_counts = w.row_off + L.ntiles * da::kScanTile + 4;
            w.cap_m = L.cap_m;
            w.cap_s = L.cap_s;
            w.cap_g = L.cap_g;
        }
        const cudaError_t e =
            da::launch_backward_binned(a, w, d.feat_dtype, s, ready ? da::kStagePull : da::kStageAll);
        if (e != cudaSuccess) return cuda_fail(e, "binned backward launch");
        return da::bounds_report(s);
    }
    cudaError_t e = da::launch_zero_fill(grad_feat, n_gf, s);
    if (e != cudaSuccess) return cuda_fail(e, "grad_feat zero-fill");
    if (n_out == 0) return DA_OK;
    if (pb.pks == 0) {
        // No samples, but with S = 0 scales the location entries still exist:
        // their gradients are 0. (The sampling kernels write grad_loc only
        // while walking samples.)
        const int64_t n_loc =
            static_cast<int64_t>(pb.num_ba) * pb.pk * (pb.layout == da::kLayoutFused ? 2 * pb.G : 2);
        if (n_loc > 0) e = cudaMemsetAsync(a.grad_loc, 0, static_cast<size_t>(n_loc) * sizeof(float), s);
        return e == cudaSuccess ? DA_OK : cuda_fail(e, "grad_loc zero-fill");
    }
    e = da::launch_backward(a, d.feat_dtype, chunks, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return da::bounds_report(s);
}

// Checks of the fused per-group layout: loc_weight [B,A,G,P,K,2+S] fp32.
da_status prepare_fused(const da_dims *dims, const void *feat, const int32_t *spatial_shape,
                        const int32_t *level_start_index, const float *loc_weight, da::Problem &pb, int &chunks)
{
    da_status st = da::prepare_shape(dims, spatial_shape, level_start_index, pb, chunks);
    if (st != DA_OK) return st;
    const int64_t n_feat = static_cast<int64_t>(dims->batch) * dims->num_feat_rows * dims->num_embeds;
    const int64_t n_lw = static_cast<int64_t>(pb.num_ba) * pb.G * pb.pk * (2 + pb.S);
    if (static_cast<int64_t>(pb.num_ba) * pb.G * pb.pk > INT32_MAX)
        return fail(DA_ERR_UNSUPPORTED, "batch*anchors*groups*pts*cams exceeds int32");
    if (n_feat > 0 && !feat) return fail(DA_ERR_NULL, "mc_ms_feat is NULL");
    if (n_lw > 0 && pb.pks > 0 && !loc_weight) return fail(DA_ERR_NULL, "loc_weight is NULL");
    if (!aligned(feat, 16)) return fail(DA_ERR_ALIGN, "mc_ms_feat must be 16-byte aligned");
    if (!aligned(loc_weight, 4)) return fail(DA_ERR_ALIGN, "loc_weight must be 4-byte aligned");
    pb.feat = feat;
    pb.loc = loc_weight;
    pb.weights = nullptr;
    pb.layout = da::kLayoutFused;
    return DA_OK;
}

// Checks of the projected layout's inputs; fills pb's projection fields.
da_status prepare_projected(const da_dims *dims, const void *feat, const int32_t *spatial_shape,
                            const int32_t *level_start_index, const float *keypoints, const float *projection,
                            float image_w, float image_h, da::Problem &pb, int &chunks)
{
    da_status st = da::prepare_shape(dims, spatial_shape, level_start_index, pb, chunks);
    if (st != DA_OK) return st;
    const int64_t n_feat = static_cast<int64_t>(dims->batch) * dims->num_feat_rows * dims->num_embeds;
    const int64_t n_kp = static_cast<int64_t>(pb.num_ba) * pb.P;
    const int64_t n_cam = static_cast<int64_t>(pb.B) * pb.K;
    if (n_kp > INT32_MAX) return fail(DA_ERR_UNSUPPORTED, "batch*anchors*pts exceeds int32");
    if (n_feat > 0 && !feat) return fail(DA_ERR_NULL, "mc_ms_feat is NULL");
    if (n_kp > 0 && !keypoints) return fail(DA_ERR_NULL, "keypoints is NULL");
    if (n_cam > 0 && !projection) return fail(DA_ERR_NULL, "projection is NULL");
    if (!aligned(feat, 16)) return fail(DA_ERR_ALIGN, "mc_ms_feat must be 16-byte aligned");
    if (!aligned(keypoints, 4) || !aligned(projection, 4))
        return fail(DA_ERR_ALIGN, "keypoints and projection must be 4-byte aligned");
    if (!(image_w > 0.f) || !(image_h > 0.f) || !std::isfinite(image_w) || !std::isfinite(image_h))
        return fail(DA_ERR_SHAPE, "image size %g x %g must be positive and finite", image_w, image_h);
    pb.feat = feat;
    pb.keypoints = keypoints;
    pb.projection = projection;
    pb.image_w = image_w;
    pb.image_h = image_h;
    return DA_OK;
}

// The binned backward of the fused layout runs on a rewrite of the problem:
// one group of D channels, A*G anchors (a' = a*G + g) and rows*G virtual
// rows (pixel row r of group g is virtual row r*G + g, at feat + (r*G + g)*D;
// anchor a' reads grad_out at a'*D). Every address stays the same.
da_status fused_binned_problem(const da_dims &d, const da::Problem &pb, da_dims &vd, da::Problem &pv)
{
    const int64_t A2 = static_cast<int64_t>(d.num_anchors) * d.num_groups;
    const int64_t rows2 = d.num_feat_rows * d.num_groups;
    if (A2 > INT32_MAX || rows2 > INT32_MAX)
        return fail(DA_ERR_UNSUPPORTED, "binned fused backward: anchors*groups or rows*groups exceeds int32");
    vd = d;
    vd.num_anchors = static_cast<int32_t>(A2);
    vd.num_groups = 1;
    vd.num_embeds = d.num_embeds / d.num_groups;
    vd.num_feat_rows = rows2;
    pv = pb;
    pv.A = static_cast<int32_t>(A2);
    pv.G = 1;
    pv.C = pb.D;
    pv.rows = rows2;
    pv.num_ba = static_cast<int32_t>(static_cast<int64_t>(d.batch) * A2);
    pv.gsplit = d.num_groups;
    pv.div_A = da::FastDiv::make(A2 > 0 ? static_cast<uint32_t>(A2) : 1);
    pv.div_G = da::FastDiv::make(1);
    pv.div_rows = da::FastDiv::make(rows2 > 0 ? static_cast<uint32_t>(rows2) : 1);
    return DA_OK;
}

// Device address of g_noalloc_scratch in the current device's context. It is
// looked up on every call rather than cached: a cached address would dangle
// after cudaDeviceReset or any other teardown and re-creation of the
// device's primary context, which loads the module (and the array) again at
// a possibly different address. After the first call on a device the lookup
// is a host-side table query.
da_status noalloc_scratch(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
    *out = p;
    return DA_OK;
}

}  // namespace

extern "C" {

da_status da_forward(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                     const int32_t *level_start_index, const float *sampling_location,
                     const float *weights, float *out, da_stream_t stream)
{
    da::FwdArgs a{};
    int chunks = 0;
    da_status st = prepare(dims, mc_ms_feat, spatial_shape, level_start_index, sampling_location,
                           weights, a.pb, chunks);
    if (st != DA_OK) return st;
    return forward_impl(*dims, a, chunks, out, stream);
}

da_status da_backward_workspace_size(const da_dims *dims, size_t *bytes)
{
    if (!dims || !bytes) return fail(DA_ERR_NULL, "dims / bytes is NULL");
    const da_dims d = *dims;
    if (d.batch < 0 || d.num_cams < 0 || d.num_scales < 0 || d.num_anchors < 0 || d.num_pts < 0 ||
        d.num_embeds < 1 || d.num_groups < 1 || d.num_embeds % d.num_groups != 0 || d.num_feat_rows < 0 ||
        d.num_feat_rows > DA_MAX_ROWS)
        return fail(DA_ERR_SHAPE, "invalid dims");
    da::BinLayout L;
    const da_status st = binned_layout(d, L);
    if (st != DA_OK) return st;
    *bytes = L.bytes;
    return DA_OK;
}

da_status da_backward_fused_workspace_size(const da_dims *dims, size_t *bytes)
{
    if (!dims || !bytes) return fail(DA_ERR_NULL, "dims / bytes is NULL");
    const da_dims d = *dims;
    if (d.batch < 0 || d.num_cams < 0 || d.num_scales < 0 || d.num_anchors < 0 || d.num_pts < 0 ||
        d.num_embeds < 1 || d.num_groups < 1 || d.num_embeds % d.num_groups != 0 || d.num_feat_rows < 0 ||
        d.num_feat_rows > DA_MAX_ROWS)
        return fail(DA_ERR_SHAPE, "invalid dims");
    da::Problem pb{}, pv{};
    pb.D = d.num_embeds / d.num_groups;
    da_dims vd;
    da_status st = fused_binned_problem(d, pb, vd, pv);
    if (st != DA_OK) return st;
    da::BinLayout L;
    st = binned_layout(vd, L);
    if (st != DA_OK) return st;
    *bytes = L.bytes;
    return DA_OK;
}

da_status da_backward(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                      const int32_t *level_start_index, const float *sampling_location,
                      const float *weights, const float *grad_out, float *grad_feat, float *grad_loc,
                      float *grad_weight, void *workspace, size_t workspace_bytes, da_stream_t stream)
{
    return da_backward_ex(dims, mc_ms_feat, spatial_shape, level_start_index, sampling_location, weights,
                          grad_out, grad_feat, grad_loc, grad_weight, workspace, workspace_bytes, 0u, stream);
}

da_status da_backward_ex(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                         const int32_t *level_start_index, const float *sampling_location,
                         const float *weights, const float *grad_out, float *grad_feat, float *grad_loc,
                         float *grad_weight, void *workspace, size_t workspace_bytes, uint32_t flags,
                         da_stream_t stream)
{
    da::BwdArgs a{};
    int chunks = 0;
    da_status st = prepare(dims, mc_ms_feat, spatial_shape, level_start_index, sampling_location,
                           weights, a.pb, chunks);
    if (st != DA_OK) return st;
    const da::Problem &pb = a.pb;
    const int64_t n_gl = static_cast<int64_t>(pb.num_ba) * pb.pk * 2;
    const int64_t n_gw = static_cast<int64_t>(pb.num_ba) * pb.pks * pb.G;
    if (n_gl > 0 && !grad_loc) return fail(DA_ERR_NULL, "grad_loc is NULL");
    if (n_gw > 0 && !grad_weight) return fail(DA_ERR_NULL, "grad_weight is NULL");
    if (!aligned(grad_loc, 4)) return fail(DA_ERR_ALIGN, "grad_loc must be 4-byte aligned");
    if (!aligned(grad_weight, 4)) return fail(DA_ERR_ALIGN, "grad_weight must be 4-byte aligned");
    a.grad_loc = grad_loc;
    a.grad_weight = grad_weight;
    return backward_impl(*dims, a, chunks, grad_out, grad_feat, workspace, workspace_bytes, flags, stream);
}

da_status da_backward_bin(const da_dims *dims, const int32_t *spatial_shape, const int32_t *level_start_index,
                          const float *sampling_location, void *workspace, size_t workspace_bytes, uint32_t flags,
                          da_stream_t stream)
{
    if (flags & ~static_cast<uint32_t>(DA_BACKWARD_DETERMINISTIC))
        return fail(DA_ERR_SHAPE, "da_backward_bin takes DA_BACKWARD_DETERMINISTIC only (flags 0x%x)", flags);
    da::BwdArgs a{};
    int chunks = 0;
    da_status st = da::prepare_shape(dims, spatial_shape, level_start_index, a.pb, chunks);
    if (st != DA_OK) return st;
    const int64_t n_loc = static_cast<int64_t>(a.pb.num_ba) * a.pb.pk;
    if (n_loc > 0 && !sampling_location) return fail(DA_ERR_NULL, "sampling_location is NULL");
    if (!aligned(sampling_location, 8)) return fail(DA_ERR_ALIGN, "sampling_location must be 8-byte aligned");
    a.pb.loc = sampling_location;
    da::BinLayout L;
    st = binned_layout(*dims, L);
    if (st != DA_OK) return st;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.bytes)
        return fail(DA_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes (got %zu)", L.bytes,
                    workspace_bytes);
    char *ws = static_cast<char *>(workspace);
    da::BinArgs w{};
    w.row_off = reinterpret_cast<int32_t *>(ws + L.off_row_off);
    w.tile_sum = reinterpret_cast<int32_t *>(ws + L.off_tile_sum);
    w.rec = reinterpret_cast<int2 *>(ws + L.off_rec);
    w.dpix = reinterpret_cast<float *>(ws + L.off_dpix);
    w.left = reinterpret_cast<int32_t *>(ws + L.off_left);
    w.left_count = w.row_off + L.ntiles * da::kScanTile + 1;
    w.rows_total = L.rows_total;
    w.nsid = L.nsid;
    w.ncap = L.ncap;
    w.ntiles = L.ntiles;
    if (flags & DA_BACKWARD_DETERMINISTIC) {
        w.sort_lists = reinterpret_cast<int32_t *>(ws + L.off_lists);
        w.sort_counts = w.row_off + L.ntiles * da::kScanTile + 4;
        w.cap_m = L.cap_m;
        w.cap_s = L.cap_s;
        w.cap_g = L.cap_g;
    }
    const cudaError_t e = da::launch_backward_binned(a, w, dims->feat_dtype, reinterpret_cast<cudaStream_t>(stream),
                                                     da::kStageBin);
    if (e != cudaSuccess) return cuda_fail(e, "binning launch");
    return da::bounds_report(reinterpret_cast<cudaStream_t>(stream));
}

da_status da_forward_fused(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                           const int32_t *level_start_index, const float *loc_weight, float *out,
                           da_stream_t stream)
{
    da::FwdArgs a{};
    int chunks = 0;
    const da_status st = prepare_fused(dims, mc_ms_feat, spatial_shape, level_start_index, loc_weight, a.pb, chunks);
    if (st != DA_OK) return st;
    return forward_impl(*dims, a, chunks, out, stream);
}

da_status da_backward_fused(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                            const int32_t *level_start_index, const float *loc_weight, const float *grad_out,
                            float *grad_feat, float *grad_loc_weight, void *workspace, size_t workspace_bytes,
                            da_stream_t stream)
{
    da::BwdArgs a{};
    int chunks = 0;
    const da_status st = prepare_fused(dims, mc_ms_feat, spatial_shape, level_start_index, loc_weight, a.pb, chunks);
    if (st != DA_OK) return st;
    const da::Problem &pb = a.pb;
    const int64_t n_glw = static_cast<int64_t>(pb.num_ba) * pb.G * pb.pk * (2 + pb.S);
    if (n_glw > 0 && !grad_loc_weight) return fail(DA_ERR_NULL, "grad_loc_weight is NULL");
    if (!aligned(grad_loc_weight, 4)) return fail(DA_ERR_ALIGN, "grad_loc_weight must be 4-byte aligned");
    a.grad_loc = grad_loc_weight;
    a.grad_weight = nullptr;
    if (workspace || workspace_bytes) {
        da_dims vd;
        da::BwdArgs av = a;
        const da_status sv = fused_binned_problem(*dims, a.pb, vd, av.pb);
        if (sv != DA_OK) return sv;
        return backward_impl(vd, av, chunks, grad_out, grad_feat, workspace, workspace_bytes, 0u, stream);
    }
    return backward_impl(*dims, a, chunks, grad_out, grad_feat, nullptr, 0, 0u, stream);
}

da_status da_forward_projected(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                               const int32_t *level_start_index, const float *keypoints, const float *projection,
                               float image_w, float image_h, const float *weight_logits, float *out,
                               float *sampling_location, float *weights, da_stream_t stream)
{
    da::FwdArgs a{};
    int chunks = 0;
    const da_status st = prepare_projected(dims, mc_ms_feat, spatial_shape, level_start_index, keypoints, projection,
                                           image_w, image_h, a.pb, chunks);
    if (st != DA_OK) return st;
    const int64_t n_w = static_cast<int64_t>(a.pb.num_ba) * a.pb.pks * a.pb.G;
    if (n_w > 0 && !weight_logits) return fail(DA_ERR_NULL, "weight_logits is NULL");
    if (!aligned(weight_logits, 4) || !aligned(sampling_location, 4) || !aligned(weights, 4))
        return fail(DA_ERR_ALIGN, "weight_logits, sampling_location and weights must be 4-byte aligned");
    a.pb.logits = weight_logits;
    a.pb.layout = da::kLayoutProj;
    if (da::projected_smem_bytes(a.pb) > da::kProjectedSmemMax)
        return fail(DA_ERR_UNSUPPORTED, "projected layout: pts*cams*scales = %d too large for the shared staging",
                    a.pb.pks);
    a.loc_out = sampling_location;
    a.weights_out = weights;
    return forward_impl(*dims, a, chunks, out, stream);
}

da_status da_backward_projected(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                                const int32_t *level_start_index, const float *keypoints, const float *projection,
                                float image_w, float image_h, const float *sampling_location, const float *weights,
                                const float *grad_out, float *grad_feat, float *grad_loc, float *grad_weight,
                                float *grad_keypoints, float *grad_logits, void *workspace, size_t workspace_bytes,
                                uint32_t flags, da_stream_t stream)
{
    da::Problem pp{};
    int chunks = 0;
    da_status st = prepare_projected(dims, mc_ms_feat, spatial_shape, level_start_index, keypoints, projection,
                                     image_w, image_h, pp, chunks);
    if (st != DA_OK) return st;
    const int64_t n_kp = static_cast<int64_t>(pp.num_ba) * pp.P;
    const int64_t n_w = static_cast<int64_t>(pp.num_ba) * pp.pks * pp.G;
    if (n_kp > 0 && !grad_keypoints) return fail(DA_ERR_NULL, "grad_keypoints is NULL");
    if (n_w > 0 && !grad_logits) return fail(DA_ERR_NULL, "grad_logits is NULL");
    if (!aligned(grad_keypoints, 4) || !aligned(grad_logits, 4))
        return fail(DA_ERR_ALIGN, "grad_keypoints and grad_logits must be 4-byte aligned");
    // The operator's backward on the forward's locations and weights.
    st = da_backward_ex(dims, mc_ms_feat, spatial_shape, level_start_index, sampling_location, weights, grad_out,
                        grad_feat, grad_loc, grad_weight, workspace, workspace_bytes, flags, stream);
    if (st != DA_OK) return st;
    const cudaError_t e = da::launch_projected_chain(pp, weights, grad_loc, grad_weight, grad_keypoints, grad_logits,
                                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projected chain-rule launch");
    return da::bounds_report(reinterpret_cast<cudaStream_t>(stream));
}

da_status da_backward_noalloc(const da_dims *dims, const void *mc_ms_feat, const int32_t *spatial_shape,
                              const int32_t *level_start_index, const float *sampling_location,
                              const float *weights, const float *grad_out, float *grad_feat, float *grad_loc,
                              float *grad_weight, da_stream_t stream)
{
    size_t need = 0;
    da_status st = da_backward_workspace_size(dims, &need);
    if (st != DA_OK) return st;
    if (need > DA_NOALLOC_SCRATCH_BYTES)
        return fail(DA_ERR_WORKSPACE,
                    "da_backward_noalloc: this problem needs %zu bytes of scratch; the built-in array holds %u "
                    "(use da_backward with a workspace)",
                    need, DA_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != DA_OK) return st;
    return da_backward(dims, mc_ms_feat, spatial_shape, level_start_index, sampling_location, weights, grad_out,
                       grad_feat, grad_loc, grad_weight, scratch, DA_NOALLOC_SCRATCH_BYTES, stream);
}

const char *da_status_string(da_status status)
{
    switch (status) {
        case DA_OK: return "DA_OK";
        case DA_ERR_NULL: return "DA_ERR_NULL";
        case DA_ERR_SHAPE: return "DA_ERR_SHAPE";
        case DA_ERR_ALIGN: return "DA_ERR_ALIGN";
        case DA_ERR_UNSUPPORTED: return "DA_ERR_UNSUPPORTED";
        case DA_ERR_CUDA: return "DA_ERR_CUDA";
        case DA_ERR_WORKSPACE: return "DA_ERR_WORKSPACE";
        case DA_ERR_DEVICE_BOUNDS: return "DA_ERR_DEVICE_BOUNDS";
    }
    return "DA_ERR_UNKNOWN";
}

const char *da_last_error(void) { return da::last_error(); }

int32_t da_version(void) { return 100; }

}  // extern "C"
