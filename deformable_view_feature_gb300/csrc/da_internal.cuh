// Internal declarations shared by the CUDA translation units of libda.so.
// The public C ABI is include/da.h. Nothing here is exported.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "da.h"
#include "da_bounds.h"

namespace da {

constexpr int kWarps = 8;            // warps per CTA in the sampling kernels
constexpr int kThreads = kWarps * 32;

// One feature map (k, s): H x W pixels starting at feature row `start`.
struct MapInfo {
    int32_t H, W, start, pad;
};

// Division by a runtime divisor d >= 1 through a multiply and a shift:
// n / d == (n * m) >> sh for every 0 <= n < 2^31, with l = ceil(log2 d),
// m = ceil(2^(31+l) / d) < 2^32 and sh = 31 + l. It holds because
// m*d - 2^(31+l) < d <= 2^l, so n*(m*d - 2^(31+l)) < 2^(31+l) and the
// error term stays below 1/d.
struct FastDiv {
    uint32_t d, m, sh;
    static FastDiv make(uint32_t divisor)
    {
        uint32_t l = 0;
        while ((1ull << l) < divisor) ++l;
        const uint64_t num = (1ull << (31 + l)) + divisor - 1;
        return FastDiv{divisor, static_cast<uint32_t>(num / divisor), 31 + l};
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        return static_cast<uint32_t>((static_cast<uint64_t>(n) * m) >> sh);
    }
};

// Everything a sampling kernel needs about the problem. It is passed by value
// as a kernel parameter; the kernels copy the map table to shared memory.
constexpr int kLayoutStd = 0;    // loc + weights
constexpr int kLayoutFused = 1;  // per-group loc_weight (the DCNv4 form)
constexpr int kLayoutProj = 2;   // key points + cameras + logits

struct Problem {
    const void *feat;
    // Standard layout: loc [B,A,P,K,2] and weights [B,A,P,K,S,G].
    // Fused per-group layout (the DCNv4 form): loc points to
    // loc_weight [B,A,G,P,K,2+S] = (x, y, w_0 .. w_{S-1}) and weights is NULL.
    // Projected layout (forward only): loc and weights are NULL; the
    // locations come from keypoints [B,A,P,3] through projection [B,K,4,4]
    // and the weights are a softmax of logits [B,A,P,K,S,G].
    const float *loc;
    const float *weights;
    int64_t rows;             // feature rows per batch item
    int32_t B, A, P, K, S, C, G, D;
    int32_t pks;              // P*K*S samples per (b, a, g)
    int32_t pk;               // P*K locations per (b, a)
    int32_t num_ba;           // B*A
    int32_t anchors_per_cta;  // anchors (or views) owned by one CTA, all groups
    int32_t nmaps;            // K*S
    int32_t layout;           // kLayoutStd, kLayoutFused or kLayoutProj
    // Binned backward of the fused layout: the problem is rewritten with one
    // group (G = 1, C = D), A*G anchors (a' = a*G + g) and rows*G virtual
    // rows; pixel row r of group g is virtual row r*gsplit + g, whose D
    // channels sit at feat + (virtual row)*D. gsplit is 1 otherwise.
    int32_t gsplit;
    FastDiv div_S, div_K, div_G, div_A, div_P, div_PKS, div_rows;
    MapInfo maps[DA_MAX_MAPS];
    // Bounds-checking builds: the device error word (see da_bounds.h);
    // NULL in release builds.
    uint32_t *dbg_err;
    // Projected layout only (after the fields every kernel reads).
    const float *keypoints;
    const float *projection;
    const float *logits;
    float image_w, image_h;
};

struct FwdArgs {
    Problem pb;
    float *out;
    // Camera parts of the standard forward (1 = all cameras in one CTA).
    // With parts > 1, CTA c takes anchors of batch item b for the cameras of
    // part q, in the order (b, q, anchors), and adds its partial sums into
    // `out`, which the launch zeroes first.
    int parts;
    int ctas_per_part;    // CTAs per (batch item, part)
    int kpart;            // cameras per part (K / parts)
    FastDiv div_cpp;      // by ctas_per_part
    FastDiv div_kpart;    // by kpart
    // Projected layout only: where to write the computed locations
    // [B,A,P,K,2] and weights [B,A,P,K,S,G]; NULL = do not write.
    float *loc_out;
    float *weights_out;
};

struct BwdArgs {
    Problem pb;
    const float *grad_out;
    float *grad_feat;
    float *grad_loc;
    float *grad_weight;
};

// Device scratch of the binned backward, carved out of one caller-provided
// buffer. Every region starts on a 256-byte boundary.
//   row_off  [ntiles*kScanTile + kRowOffTail] int32: per feature row (over
//            all B*rows rows): the corner count, then its exclusive prefix
//            sum, then (after the fill) the end of the row's record range.
//            The tail holds the scan's total and the sort's list counters.
//   tile_sum [ntiles + 4] int32: per-tile totals of the scan
//   rec      [ncap] int2: {key = sample id * 4 + corner, corner weight bits},
//            grouped by feature row; in deterministic mode sorted by key
//            within each row
//   dpix     [ncap * G] fp32: d = grad_out . feat of each (record, group),
//            at row `key` of the record: the four corners of a sample are
//            adjacent, in sample order. Entries of corners outside their
//            map are never written (no record) and never read.
//   left     [rows_total] int32: rows the pull hands from a warp's pixel run
//            to one warp each (runs of more than kRunMaxRecs records); their
//            count is row_off's tail word 1, reset by the epilogue
//   lists    [cap_m + cap_s + cap_g] int32: rows the deterministic sort
//            hands to a warp (9..128 records), a CTA with shared memory
//            (129..2048) or a CTA working in global memory (more)
// A sample id here is ((b*A + a)*P + p)*K + k)*S + s: a sample of all groups.
constexpr int kScanTile = 4096;
constexpr int kRowOffTail = 8;  // [0] scan total, [1] pull's leftover rows, [4..6] sort list counters

struct BinLayout {
    int64_t rows_total;  // B * rows
    int64_t nsid;        // B*A*P*K*S
    int64_t ncap;        // 4 * nsid
    int64_t ntiles;
    size_t off_row_off, off_tile_sum, off_rec, off_dpix, off_left, off_lists, bytes;
    // Capacities of the three row lists of the deterministic sort (rows
    // with more than 8, 128 and 2048 records).
    int64_t cap_m, cap_s, cap_g;
};
BinLayout bin_layout(int64_t B, int64_t rows, int64_t A, int64_t P, int64_t K, int64_t S, int64_t G);

// Whether the binned backward has a kernel for these channel counts: C in
// {8, 16, ..., 256} (a power of two times 8, at most one warp per row) and
// D a multiple of 8.
inline bool binned_supported(int C, int D)
{
    return C >= 8 && C <= 256 && (C & (C - 1)) == 0 && D % 8 == 0;
}

struct BinArgs {
    int32_t *row_off;
    int32_t *tile_sum;
    int2 *rec;
    float *dpix;
    int64_t rows_total, nsid, ncap, ntiles;
    // Deterministic mode: the row lists of the per-row sort, and their three
    // counters (zeroed with row_off; NULL sort_lists = no sort).
    int32_t *sort_lists;
    int32_t *sort_counts;
    int64_t cap_m, cap_s, cap_g;
    // Rows the pull hands over to one warp each, and their count.
    int32_t *left;
    int32_t *left_count;
};

// `chunks` = D * sizeof(feature) / 16, one of 1, 2, 4, 8.
cudaError_t launch_forward(const FwdArgs &a, int feat_dtype, int chunks, cudaStream_t st);
cudaError_t launch_backward(const BwdArgs &a, int feat_dtype, int chunks, cudaStream_t st);
// Stages of the binned backward: the binning (count, scan, fill, and the
// deterministic sort when asked for) depends on the locations only; the pull
// and epilogue need grad_out.
constexpr int kStageBin = 1, kStagePull = 2, kStageAll = 3;
cudaError_t launch_backward_binned(const BwdArgs &a, const BinArgs &w, int feat_dtype, cudaStream_t st,
                                   int stages = kStageAll);
cudaError_t launch_zero_fill(float *p, int64_t n_floats, cudaStream_t st);
// The pull step of the binned backward (da_pull.cu): grad_feat, and d of
// every record and group in dpix.
cudaError_t launch_pull(const BwdArgs &a, const BinArgs &w, int feat_dtype, cudaStream_t st);
// Chain rule of the projected layout: grad_logits and grad_keypoints from the
// operator's grad_loc and grad_weight (pb holds keypoints, projection, image
// size).
cudaError_t launch_projected_chain(const Problem &pb, const float *weights, const float *grad_loc,
                                   const float *grad_weight, float *grad_keypoints, float *grad_logits,
                                   cudaStream_t st);

// Host-side helpers of the entry points (da_abi.cu).
// fail: records a one-line reason for da_last_error() and returns st.
da_status fail(da_status st, const char *fmt, ...);
const char *last_error();
da_status cuda_fail(cudaError_t e, const char *what);
bool aligned(const void *p, uintptr_t a);
// Bounds-checking builds (DA_DEBUG_BOUNDS): the device address of the error
// word the kernels set bits in (NULL in release builds, and if the lookup
// fails), and the check an entry point makes after enqueueing its work: wait
// for the stream, read and clear the word, DA_ERR_DEVICE_BOUNDS if a bit
// was set. Release builds: returns DA_OK without a CUDA call.
uint32_t *bounds_word();
da_status bounds_report(cudaStream_t st);
// Validates dims and the two host map tables and fills every field of pb
// except the tensor pointers. Makes no CUDA call (but a bounds-checking
// build looks up its error word).
da_status prepare_shape(const da_dims *dims, const int32_t *spatial_shape, const int32_t *level_start_index,
                        Problem &pb, int &chunks);

// Dynamic shared memory of the scatter backward: the grad_loc staging area
// of one CTA's views (per group in the fused layout).
inline size_t scatter_smem_bytes(const Problem &pb)
{
    return static_cast<size_t>(pb.anchors_per_cta) * (pb.layout == kLayoutFused ? pb.G : 1) * pb.P * 2 *
           sizeof(float);
}

// Whether the forward and the scatter backward take the thread-per-chunk
// kernels: few samples per (anchor, group) (the DCNv4 form has 9), and an
// anchor's C channels in at most 32 chunks of 16 bytes.
inline bool use_small_task_kernels(const Problem &pb, int elem_bytes)
{
    const int cpa = pb.C * elem_bytes / 16;
    return pb.pks <= 16 && cpa <= 32 && (pb.C * elem_bytes) % 16 == 0;
}

// Dynamic shared memory of the projected forward: the CTA's projected
// locations and one buffer of softmax numerators per warp.
inline size_t projected_smem_bytes(const Problem &pb)
{
    return static_cast<size_t>(pb.anchors_per_cta) * pb.pk * 8 + static_cast<size_t>(kWarps) * pb.pks * 4;
}
constexpr size_t kProjectedSmemMax = 160 * 1024;

// Grid size that covers num_ba anchors, anchors_per_cta at a time.
inline int64_t sampling_grid(const Problem &pb)
{
    return (static_cast<int64_t>(pb.num_ba) + pb.anchors_per_cta - 1) / pb.anchors_per_cta;
}

// ------------------------------------------------------------------ device helpers

// Normalised location of key point kp seen through camera matrix m: the
// pinhole reading of the Sparse4D page's projection step (§1, §6), in fp32
// with every product, sum and quotient rounded in this order (the location
// decides which pixels are read):
//   ud = ((m00*X + m01*Y) + m02*Z) + m03, vd and d likewise with rows 1, 2;
//   x = (ud / d) / image_w, y = (vd / d) / image_h;
// (NaN, NaN) when d <= 1e-5 (behind the camera), which reads nothing.
__device__ __forceinline__ float2 project_point(const float *kp, const float *m, float image_w, float image_h)
{
    const float X = kp[0], Y = kp[1], Z = kp[2];
    const float ud = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[0], X), __fmul_rn(m[1], Y)), __fmul_rn(m[2], Z)), m[3]);
    const float vd = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[4], X), __fmul_rn(m[5], Y)), __fmul_rn(m[6], Z)), m[7]);
    const float d = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(m[8], X), __fmul_rn(m[9], Y)), __fmul_rn(m[10], Z)), m[11]);
    if (!(d > 1e-5f)) return make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    return make_float2(__fdiv_rn(__fdiv_rn(ud, d), image_w), __fdiv_rn(__fdiv_rn(vd, d), image_h));
}

// Location (x, y) and weight of the sample (b*A + a = ba, group g,
// jk = p*K + k, scale s) in the standard or the fused layout (see Problem). In the fused layout
// the entry of (ba, g, jk) holds 2 + S floats, so (x, y) need not be 8-byte
// aligned and is read as two floats. (The projected layout computes both in
// the forward kernel itself.)
template <int LAYOUT>
__device__ __forceinline__ void sample_xyw(const Problem &pb, int64_t ba, int g, int jk, int s, float2 &xy,
                                           float &w)
{
    if constexpr (LAYOUT == kLayoutFused) {
        const float *e = pb.loc + ((ba * pb.G + g) * pb.pk + jk) * (2 + pb.S);
        xy = make_float2(e[0], e[1]);
        w = e[2 + s];
    } else {
        const int64_t locid = ba * pb.pk + jk;
        xy = *reinterpret_cast<const float2 *>(pb.loc + locid * 2);
        w = pb.weights[(locid * pb.S + s) * pb.G + g];
    }
}

// Weight of sample sid (a sample of all groups) for group g in the binned
// backward: weights[sid, g], or in the fused layout's rewrite (G = 1) the
// entry 2 + s of the sample's location.
template <bool FUSED>
__device__ __forceinline__ float bin_weight(const Problem &pb, int sid, int g)
{
    if constexpr (FUSED) {
        const int pk = static_cast<int>(pb.div_S.div(sid));
        return __ldg(&pb.loc[static_cast<int64_t>(pk) * (2 + pb.S) + 2 + (sid - pk * pb.S)]);
    }
    return __ldg(&pb.weights[static_cast<int64_t>(sid) * pb.G + g]);
}

// Bilinear footprint of one sample. The steps are those of the page "Inside
// Sparse4D's CUDA core", §3.2:
//   h_im = y*H - 0.5 and w_im = x*W - 0.5, each rounded twice (a product,
//   then a difference; no fused multiply-add), because floor() of them picks
//   the integer corners;
//   corners 1..4 = (h_low, w_low), (h_low, w_low+1), (h_low+1, w_low),
//   (h_low+1, w_low+1) with weights hh*hw, hh*lw, lh*hw, lh*lw;
//   a corner is read only if 0 <= row <= H-1 and 0 <= col <= W-1.
// row[i] is the feature row of corner i within its batch item, or -1 when the
// corner is outside the map. A sample whose coordinates are not finite has
// no corners and zero weights.
struct Footprint {
    int32_t row[4];
    float cw[4];
    float lh, lw, hh, hw;
};

__device__ __forceinline__ void footprint(float x, float y, const MapInfo &m, Footprint &f)
{
    const float h_im = __fsub_rn(__fmul_rn(y, static_cast<float>(m.H)), 0.5f);
    const float w_im = __fsub_rn(__fmul_rn(x, static_cast<float>(m.W)), 0.5f);
    if (!(isfinite(h_im) && isfinite(w_im))) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f.row[i] = -1;
            f.cw[i] = 0.f;
        }
        f.lh = f.lw = f.hh = f.hw = 0.f;
        return;
    }
    const float hl = floorf(h_im);
    const float wl = floorf(w_im);
    f.lh = h_im - hl;
    f.lw = w_im - wl;
    f.hh = 1.f - f.lh;
    f.hw = 1.f - f.lw;
    // Clamp before converting: any h_low outside [-2, H] has both rows outside
    // the map, and so does its clamped value.
    const int ih = static_cast<int>(fminf(fmaxf(hl, -2.f), static_cast<float>(m.H)));
    const int iw = static_cast<int>(fminf(fmaxf(wl, -2.f), static_cast<float>(m.W)));
    const bool r0 = ih >= 0 && ih < m.H;
    const bool r1 = ih >= -1 && ih < m.H - 1;
    const bool c0 = iw >= 0 && iw < m.W;
    const bool c1 = iw >= -1 && iw < m.W - 1;
    const int base = m.start + ih * m.W + iw;
    f.row[0] = (r0 && c0) ? base : -1;
    f.row[1] = (r0 && c1) ? base + 1 : -1;
    f.row[2] = (r1 && c0) ? base + m.W : -1;
    f.row[3] = (r1 && c1) ? base + m.W + 1 : -1;
    f.cw[0] = f.hh * f.hw;
    f.cw[1] = f.hh * f.lw;
    f.cw[2] = f.lh * f.hw;
    f.cw[3] = f.lh * f.lw;
}

// Whether feature row r (of one batch item) is read or written: r >= 0 is a
// corner inside its map; a bounds-checking build also checks r < rows.
__device__ __forceinline__ bool feat_row_ok(const Problem &pb, int32_t r)
{
    return r >= 0 && DA_CHECK(pb.dbg_err, r, pb.rows, kBoundsFeatRow);
}

// 16-byte read-only load of one chunk of a feature row, or zeros when `pred`
// is false (then nothing is read, whatever the address).
__device__ __forceinline__ uint4 ldg16_if(bool pred, const void *p)
{
    uint4 r;
    asm("{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "r"(static_cast<int>(pred)));
    return r;
}

// Address of feature row `row` (>= 0 when used): one 32x32->64 multiply-add.
__device__ __forceinline__ const char *row_addr(const char *base, int32_t row, uint32_t row_bytes)
{
    return base + static_cast<uint64_t>(static_cast<uint32_t>(row)) * row_bytes;
}

// The 16 bytes as floats: 4 fp32 values, or 8 bf16 or fp16 values widened
// exactly.
template <typename T>
struct Chunk;

template <>
struct Chunk<float> {
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&v)[4])
    {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z);
        v[3] = __uint_as_float(r.w);
    }
};

struct Bf16Tag {};

template <>
struct Chunk<Bf16Tag> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&v)[8])
    {
        v[0] = __uint_as_float(r.x << 16);
        v[1] = __uint_as_float(r.x & 0xffff0000u);
        v[2] = __uint_as_float(r.y << 16);
        v[3] = __uint_as_float(r.y & 0xffff0000u);
        v[4] = __uint_as_float(r.z << 16);
        v[5] = __uint_as_float(r.z & 0xffff0000u);
        v[6] = __uint_as_float(r.w << 16);
        v[7] = __uint_as_float(r.w & 0xffff0000u);
    }
};

struct F16Tag {};

// 8 fp16 values widened exactly (every binary16 value is a binary32 value).
template <>
struct Chunk<F16Tag> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&v)[8])
    {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
};

// Vector reduction of four floats into global memory (sm_90+), issued only
// when `pred` holds (no branch; the address is not touched otherwise).
__device__ __forceinline__ void red_add_v4_if(bool pred, float *p, float a, float b, float c, float d)
{
    asm volatile("{\n\t.reg .pred q;\n\t"
                 "setp.ne.b32 q, %5, 0;\n\t"
                 "@q red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n\t}"
                 :
                 : "l"(p), "f"(a), "f"(b), "f"(c), "f"(d), "r"(static_cast<int>(pred))
                 : "memory");
}

// Per-warp table of the four corners of 32 samples: tab[corner][sample] =
// {feature row or -1, weight}. Corner-major, so a lane reads the entries of
// its corner for four consecutive samples with two 16-byte loads. The row
// pitch of 36 entries (288 B) staggers the four corners by 8 banks, so the
// four corner groups of a warp read conflict-free.
constexpr int kTabPitch = 36;

// Programmatic dependent launch for the kernels of one call that follow one
// another on a stream (the binned backward's chain): such a kernel may be
// scheduled while its predecessor drains, so its launch and CTA start-up
// overlap the predecessor's last wave. Every kernel launched this way calls
// pdl_wait() before any global memory access: it returns once the preceding
// kernels of the stream have completed and their writes are visible (at
// once when there is no programmatic dependency). pdl_trigger() lets the
// next kernel launch once every CTA of this one has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Stage the map table of the kernel parameters in shared memory: lanes index
// it with divergent (k, s), which the constant bank would serialise.
__device__ __forceinline__ void stage_maps(const Problem &pb, MapInfo *maps_s)
{
    for (int i = threadIdx.x; i < pb.nmaps; i += blockDim.x) maps_s[i] = pb.maps[i];
}

}  // namespace da
