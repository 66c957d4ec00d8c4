// Host-buffer executor (include/moe_pipeline.h): per batch, an input copy on
// one stream, moe_forward on the caller's stream and an output copy on a
// second stream, chained by events so that consecutive batches overlap.

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <new>

#include "../../include/moe_pipeline.h"
#include "moe_internal.h"

namespace {

constexpr int kMaxDepth = 4;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

size_t tile_bytes(const moe_config& c) {
    return (size_t)c.T * c.d * (c.dtype == MOE_BF16 ? 2 : 4);
}

// Offsets within the executor's workspace: moe_forward's workspace first
// (so moe_get_device_error(ws) reads its error record), then the slots.
struct Layout {
    size_t fwd, x[kMaxDepth], y[kMaxDepth], aux[kMaxDepth], total;
};

bool layout(const moe_config* c, int depth, Layout* L) {
    if (c == nullptr || depth < 1 || depth > kMaxDepth || c->T < 1) return false;
    const size_t fwd = moe_workspace_size(c);
    if (fwd == 0) return false;
    size_t o = align256(fwd);
    L->fwd = 0;
    for (int b = 0; b < depth; ++b) {
        L->x[b] = o;
        o = align256(o + tile_bytes(*c));
        L->y[b] = o;
        o = align256(o + tile_bytes(*c));
        L->aux[b] = o;
        o = align256(o + sizeof(float));
    }
    L->total = o;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Makes `dev` current for the duration of a call and restores the caller's.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

struct moe_pipeline {
    moe_config cfg;
    int depth = 0;
    int device = 0;
    char* ws = nullptr;
    size_t fwd_bytes = 0;
    Layout L{};
    const float* W_r = nullptr;
    const float* logit_bias = nullptr;
    const void *W1 = nullptr, *b1 = nullptr, *W2 = nullptr, *b2 = nullptr;
    cudaStream_t compute = nullptr;  // the caller's stream
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t fence = nullptr;     // the point of `compute` the input copies wait for
    cudaEvent_t ev_in[kMaxDepth] = {}, ev_fwd[kMaxDepth] = {}, ev_out[kMaxDepth] = {};
    bool used[kMaxDepth] = {};
    int64_t next = 0;                // batches submitted
    int last = -1;                   // slot of the last submitted batch

    void release() {
        if (s_in) cudaStreamSynchronize(s_in);
        if (s_out) cudaStreamSynchronize(s_out);
        for (int b = 0; b < kMaxDepth; ++b) {
            if (ev_in[b]) cudaEventDestroy(ev_in[b]);
            if (ev_fwd[b]) cudaEventDestroy(ev_fwd[b]);
            if (ev_out[b]) cudaEventDestroy(ev_out[b]);
        }
        if (fence) cudaEventDestroy(fence);
        if (s_in) cudaStreamDestroy(s_in);
        if (s_out) cudaStreamDestroy(s_out);
    }
};

extern "C" {

size_t moe_pipeline_workspace_size(const moe_config* cfg, int32_t depth) {
    Layout L;
    return layout(cfg, depth, &L) ? L.total : 0;
}

moe_status moe_pipeline_create(const moe_config* cfg, int32_t depth, const float* W_r,
                               const float* logit_bias, const void* W1, const void* b1,
                               const void* W2, const void* b2, void* ws, size_t ws_bytes,
                               void* stream, moe_pipeline** out) {
    if (out == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const moe_status cs = moe::config_status(cfg);
    if (cs != MOE_OK) return cs;
    Layout L;
    if (!layout(cfg, depth, &L)) return MOE_ERR_INVALID_ARG;
    if (W_r == nullptr || W1 == nullptr || b1 == nullptr || W2 == nullptr || b2 == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(W_r) || !aligned16(W1) || !aligned16(W2)) return MOE_ERR_ALIGNMENT;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < L.total)
        return MOE_ERR_WORKSPACE;

    moe_pipeline* p = new (std::nothrow) moe_pipeline;
    if (p == nullptr) return MOE_ERR_CUDA;
    p->cfg = *cfg;
    p->depth = depth;
    p->ws = static_cast<char*>(ws);
    p->fwd_bytes = moe_workspace_size(cfg);
    p->L = L;
    p->W_r = W_r;
    p->logit_bias = logit_bias;
    p->W1 = W1;
    p->b1 = b1;
    p->W2 = W2;
    p->b2 = b2;
    p->compute = reinterpret_cast<cudaStream_t>(stream);
    bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->fence, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; ok && b < depth; ++b)
        ok = cudaEventCreateWithFlags(&p->ev_in[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_fwd[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_out[b], cudaEventDisableTiming) == cudaSuccess;
    // the first input copies follow what the caller enqueued so far (the
    // workspace's zero fill among it)
    ok = ok && cudaEventRecord(p->fence, p->compute) == cudaSuccess;
    if (!ok) {
        p->release();
        delete p;
        return MOE_ERR_CUDA;
    }
    *out = p;
    return MOE_OK;
}

moe_status moe_pipeline_submit(moe_pipeline* p, const void* x_host, void* y_host,
                               float* aux_host) {
    if (p == nullptr || x_host == nullptr || y_host == nullptr) return MOE_ERR_INVALID_ARG;
    DeviceGuard g(p->device);
    if (!g.ok) return MOE_ERR_CUDA;
    const int b = (int)(p->next % p->depth);
    const size_t bytes = tile_bytes(p->cfg);
    void* x = p->ws + p->L.x[b];
    void* y = p->ws + p->L.y[b];
    float* aux = reinterpret_cast<float*>(p->ws + p->L.aux[b]);
    // input copy: after the fence, and after the forward pass that last read slot b
    if (cudaStreamWaitEvent(p->s_in, p->fence, 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (p->used[b] && cudaStreamWaitEvent(p->s_in, p->ev_fwd[b], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(x, x_host, bytes, cudaMemcpyHostToDevice, p->s_in) != cudaSuccess ||
        cudaEventRecord(p->ev_in[b], p->s_in) != cudaSuccess)
        return MOE_ERR_CUDA;
    // forward pass: after its input, and after the output copy that last read slot b
    if (cudaStreamWaitEvent(p->compute, p->ev_in[b], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (p->used[b] && cudaStreamWaitEvent(p->compute, p->ev_out[b], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    const moe_status st =
        moe_forward(&p->cfg, x, p->W_r, p->logit_bias, nullptr, p->W1, p->b1, p->W2, p->b2, y,
                    aux_host != nullptr ? aux : nullptr, nullptr, nullptr, nullptr, p->ws,
                    p->fwd_bytes, p->compute);
    if (st != MOE_OK) return st;
    if (cudaEventRecord(p->ev_fwd[b], p->compute) != cudaSuccess) return MOE_ERR_CUDA;
    // output copy
    if (cudaStreamWaitEvent(p->s_out, p->ev_fwd[b], 0) != cudaSuccess ||
        cudaMemcpyAsync(y_host, y, bytes, cudaMemcpyDeviceToHost, p->s_out) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (aux_host != nullptr &&
        cudaMemcpyAsync(aux_host, aux, sizeof(float), cudaMemcpyDeviceToHost, p->s_out) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaEventRecord(p->ev_out[b], p->s_out) != cudaSuccess) return MOE_ERR_CUDA;
    p->used[b] = true;
    p->last = b;
    ++p->next;
    return MOE_OK;
}

moe_status moe_pipeline_join(moe_pipeline* p) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    DeviceGuard g(p->device);
    if (!g.ok) return MOE_ERR_CUDA;
    // the output copies run in order on s_out: the last one covers them all
    if (p->last >= 0 && cudaStreamWaitEvent(p->compute, p->ev_out[p->last], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cudaEventRecord(p->fence, p->compute) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_pipeline_destroy(moe_pipeline* p) {
    if (p == nullptr) return MOE_OK;
    moe_status st = MOE_OK;
    {
        DeviceGuard g(p->device);
        if (!g.ok) st = MOE_ERR_CUDA;
        p->release();
    }
    delete p;
    return st;
}

}  // extern "C"
