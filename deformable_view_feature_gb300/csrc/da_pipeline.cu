// Host pipeline (da_pipeline_* in include/da.h): streams problems whose
// tensors live in host memory through the device kernels.
//
// Three streams per pipeline:
//   s_in   host -> device copies of a step's inputs
//   s_run  da_forward, then da_backward
//   s_out  device -> host copies of a step's outputs
// and `depth` buffer sets (slots). Step n uses slot n % depth. Per slot,
// three events order the streams:
//   in_ready  recorded on s_in after the input copies;   s_run waits on it.
//   computed  recorded on s_run after the kernels;       s_out waits on it, and
//             s_in waits on it before it overwrites the slot's inputs again.
//   out_done  recorded on s_out after the output copies; s_run waits on it
//             before it overwrites the slot's outputs again.
// A wait on an event that was never recorded is a no-op, so the first
// `depth` steps start at once.
#include <cstring>
#include <new>
#include <vector>

#include "da_internal.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

struct Slot {
    void *feat = nullptr;
    float *loc = nullptr, *w = nullptr, *go = nullptr;
    float *out = nullptr, *gf = nullptr, *gl = nullptr, *gw = nullptr;
    void *ws = nullptr;
    cudaEvent_t in_ready = nullptr, computed = nullptr, out_done = nullptr;
};

// Makes `dev` current for the scope and restores the previous device.
struct DeviceScope {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceScope(int dev)
    {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
    }
    ~DeviceScope()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

struct da_pipeline {
    int device = 0;
    da_dims dims{};
    std::vector<int32_t> ss, ls;
    bool backward = false;
    bool binned = false;
    bool broken = false;
    int depth = 0;
    uint64_t next = 0;
    // Bytes of each tensor of one step.
    size_t b_feat = 0, b_loc = 0, b_w = 0, b_go = 0, b_gf = 0, b_ws = 0;
    void *arena = nullptr;
    cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
    std::vector<Slot> slots;

    // Frees whatever exists; safe on a partly built pipeline.
    void release()
    {
        for (Slot &s : slots) {
            if (s.in_ready) cudaEventDestroy(s.in_ready);
            if (s.computed) cudaEventDestroy(s.computed);
            if (s.out_done) cudaEventDestroy(s.out_done);
            s.in_ready = s.computed = s.out_done = nullptr;
        }
        if (s_in) cudaStreamDestroy(s_in);
        if (s_run) cudaStreamDestroy(s_run);
        if (s_out) cudaStreamDestroy(s_out);
        s_in = s_run = s_out = nullptr;
        if (arena) cudaFree(arena);
        arena = nullptr;
    }
};

namespace {

da_status h2d(void *dst, const void *src, size_t n, cudaStream_t st)
{
    if (n == 0) return DA_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st);
    return e == cudaSuccess ? DA_OK : da::cuda_fail(e, "pipeline input copy");
}

da_status d2h(void *dst, const void *src, size_t n, cudaStream_t st)
{
    if (n == 0) return DA_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? DA_OK : da::cuda_fail(e, "pipeline output copy");
}

da_status wait_on(cudaStream_t st, cudaEvent_t ev)
{
    const cudaError_t e = cudaStreamWaitEvent(st, ev, 0);
    return e == cudaSuccess ? DA_OK : da::cuda_fail(e, "cudaStreamWaitEvent");
}

da_status record(cudaEvent_t ev, cudaStream_t st)
{
    const cudaError_t e = cudaEventRecord(ev, st);
    return e == cudaSuccess ? DA_OK : da::cuda_fail(e, "cudaEventRecord");
}

da_status sync_all(da_pipeline *p)
{
    for (cudaStream_t st : {p->s_in, p->s_run, p->s_out}) {
        const cudaError_t e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) {
            p->broken = true;
            return da::cuda_fail(e, "pipeline synchronise");
        }
    }
    return DA_OK;
}

da_status submit_step(da_pipeline *p, const void *feat, const float *loc, const float *w, const float *go,
                      float *out, float *gf, float *gl, float *gw)
{
    Slot &s = p->slots[p->next % static_cast<uint64_t>(p->depth)];
    da_status st;
    // Inputs: wait until the slot's last step has finished reading them.
    if ((st = wait_on(p->s_in, s.computed)) != DA_OK) return st;
    if ((st = h2d(s.feat, feat, p->b_feat, p->s_in)) != DA_OK) return st;
    if ((st = h2d(s.loc, loc, p->b_loc, p->s_in)) != DA_OK) return st;
    if ((st = h2d(s.w, w, p->b_w, p->s_in)) != DA_OK) return st;
    if (p->backward && (st = h2d(s.go, go, p->b_go, p->s_in)) != DA_OK) return st;
    if ((st = record(s.in_ready, p->s_in)) != DA_OK) return st;

    // Kernels: wait for the inputs, and for the slot's last outputs to be
    // copied out before they are overwritten.
    if ((st = wait_on(p->s_run, s.in_ready)) != DA_OK) return st;
    if ((st = wait_on(p->s_run, s.out_done)) != DA_OK) return st;
    const da_stream_t run = reinterpret_cast<da_stream_t>(p->s_run);
    const int32_t *ss = p->ss.empty() ? nullptr : p->ss.data();
    const int32_t *ls = p->ls.empty() ? nullptr : p->ls.data();
    if ((st = da_forward(&p->dims, s.feat, ss, ls, s.loc, s.w, s.out, run)) != DA_OK) return st;
    if (p->backward &&
        (st = da_backward(&p->dims, s.feat, ss, ls, s.loc, s.w, s.go, s.gf, s.gl, s.gw, p->binned ? s.ws : nullptr,
                          p->binned ? p->b_ws : 0, run)) != DA_OK)
        return st;
    if ((st = record(s.computed, p->s_run)) != DA_OK) return st;

    // Outputs.
    if ((st = wait_on(p->s_out, s.computed)) != DA_OK) return st;
    if ((st = d2h(out, s.out, p->b_go, p->s_out)) != DA_OK) return st;
    if (p->backward) {
        if ((st = d2h(gf, s.gf, p->b_gf, p->s_out)) != DA_OK) return st;
        if ((st = d2h(gl, s.gl, p->b_loc, p->s_out)) != DA_OK) return st;
        if ((st = d2h(gw, s.gw, p->b_w, p->s_out)) != DA_OK) return st;
    }
    return record(s.out_done, p->s_out);
}

}  // namespace

extern "C" {

da_status da_pipeline_create(const da_dims *dims, const int32_t *spatial_shape, const int32_t *level_start_index,
                             int32_t with_backward, int32_t depth, da_pipeline **pipeline)
{
    if (!pipeline) return da::fail(DA_ERR_NULL, "pipeline is NULL");
    *pipeline = nullptr;
    if (depth < 1 || depth > 4) return da::fail(DA_ERR_SHAPE, "depth %d outside [1, 4]", depth);
    if (with_backward != 0 && with_backward != 1)
        return da::fail(DA_ERR_SHAPE, "with_backward must be 0 or 1 (got %d)", with_backward);
    da::Problem pb{};
    int chunks = 0;
    da_status st = da::prepare_shape(dims, spatial_shape, level_start_index, pb, chunks);
    if (st != DA_OK) return st;
    const da_dims d = *dims;
    const size_t elem = d.feat_dtype == DA_F32 ? 4 : 2;
    const size_t n_rows = static_cast<size_t>(d.batch) * static_cast<size_t>(d.num_feat_rows);
    const size_t n_samp = static_cast<size_t>(pb.num_ba) * static_cast<size_t>(pb.pk);  // (b,a,p,k)

    da_pipeline *p = new (std::nothrow) da_pipeline();
    if (!p) return da::fail(DA_ERR_CUDA, "out of host memory");
    p->dims = d;
    const size_t nmaps = static_cast<size_t>(pb.nmaps);
    p->ss.assign(spatial_shape, spatial_shape + 2 * nmaps);
    p->ls.assign(level_start_index, level_start_index + nmaps);
    p->backward = with_backward == 1;
    p->depth = depth;
    p->b_feat = n_rows * d.num_embeds * elem;
    p->b_loc = n_samp * 2 * sizeof(float);
    p->b_w = n_samp * d.num_scales * d.num_groups * sizeof(float);
    p->b_go = static_cast<size_t>(pb.num_ba) * d.num_embeds * sizeof(float);  // out has the same size
    if (p->backward) {
        p->b_gf = n_rows * d.num_embeds * sizeof(float);
        size_t ws = 0;
        p->binned = da_backward_workspace_size(&d, &ws) == DA_OK;
        p->b_ws = p->binned ? ws : 0;
    }
    // One arena: per slot feat, loc, w, out (+ go, gf, gl, gw, workspace).
    const size_t slot_bytes = round_up(p->b_feat) + round_up(p->b_loc) + round_up(p->b_w) + round_up(p->b_go) +
                              (p->backward ? round_up(p->b_go) + round_up(p->b_gf) + round_up(p->b_loc) +
                                                 round_up(p->b_w) + round_up(p->b_ws)
                                           : 0);
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess && slot_bytes > 0) e = cudaMalloc(&p->arena, slot_bytes * depth);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_run, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
    p->slots.resize(depth);
    char *cur = static_cast<char *>(p->arena);
    auto take = [&cur](size_t n) {
        char *r = cur;
        cur += round_up(n);
        return r;
    };
    for (int i = 0; i < depth && e == cudaSuccess; ++i) {
        Slot &s = p->slots[i];
        s.feat = take(p->b_feat);
        s.loc = reinterpret_cast<float *>(take(p->b_loc));
        s.w = reinterpret_cast<float *>(take(p->b_w));
        s.out = reinterpret_cast<float *>(take(p->b_go));
        if (p->backward) {
            s.go = reinterpret_cast<float *>(take(p->b_go));
            s.gf = reinterpret_cast<float *>(take(p->b_gf));
            s.gl = reinterpret_cast<float *>(take(p->b_loc));
            s.gw = reinterpret_cast<float *>(take(p->b_w));
            s.ws = take(p->b_ws);
        }
        e = cudaEventCreateWithFlags(&s.in_ready, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.computed, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.out_done, cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        p->release();
        delete p;
        return da::cuda_fail(e, "pipeline set-up");
    }
    *pipeline = p;
    return DA_OK;
}

da_status da_pipeline_submit(da_pipeline *p, const void *mc_ms_feat, const float *sampling_location,
                             const float *weights, const float *grad_out, float *out, float *grad_feat,
                             float *grad_loc, float *grad_weight)
{
    if (!p) return da::fail(DA_ERR_NULL, "pipeline is NULL");
    if (p->broken) return da::fail(DA_ERR_CUDA, "pipeline stopped after an earlier CUDA error");
    struct Need {
        const void *ptr;
        size_t bytes;
        const char *name;
    };
    const Need need[] = {{mc_ms_feat, p->b_feat, "mc_ms_feat"},
                         {sampling_location, p->b_loc, "sampling_location"},
                         {weights, p->b_w, "weights"},
                         {out, p->b_go, "out"},
                         {grad_out, p->backward ? p->b_go : 0, "grad_out"},
                         {grad_feat, p->b_gf, "grad_feat"},
                         {grad_loc, p->backward ? p->b_loc : 0, "grad_loc"},
                         {grad_weight, p->backward ? p->b_w : 0, "grad_weight"}};
    for (const Need &n : need)
        if (n.bytes > 0 && !n.ptr) return da::fail(DA_ERR_NULL, "%s is NULL", n.name);
    DeviceScope scope(p->device);
    if (scope.err != cudaSuccess) return da::cuda_fail(scope.err, "pipeline device selection");
    const da_status st = submit_step(p, mc_ms_feat, sampling_location, weights, grad_out, out, grad_feat,
                                     grad_loc, grad_weight);
    if (st != DA_OK) {
        // Part of the step may be enqueued; later steps cannot rely on the
        // slot's events.
        p->broken = true;
        return st;
    }
    ++p->next;
    return DA_OK;
}

da_status da_pipeline_sync(da_pipeline *p)
{
    if (!p) return da::fail(DA_ERR_NULL, "pipeline is NULL");
    DeviceScope scope(p->device);
    if (scope.err != cudaSuccess) return da::cuda_fail(scope.err, "pipeline device selection");
    const da_status st = sync_all(p);
    if (st == DA_OK && p->broken) return da::fail(DA_ERR_CUDA, "pipeline stopped after an earlier CUDA error");
    return st;
}

da_status da_pipeline_destroy(da_pipeline *p)
{
    if (!p) return DA_OK;
    da_status st = DA_OK;
    {
        DeviceScope scope(p->device);
        if (scope.err == cudaSuccess) {
            if (p->s_in) st = sync_all(p);
            p->release();
        } else {
            st = da::cuda_fail(scope.err, "pipeline device selection");
        }
    }
    delete p;
    return st;
}

}  // extern "C"
