// C ABI of libmoe: argument validation, workspace layout and kernel launches.
// The operation each entry point performs is documented in include/moe.h.

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Position of the next launch in the calling thread's current chain.
static thread_local int t_chain_pos = 0;
static thread_local bool t_chain_all = false;
void chain_begin() { t_chain_pos = 0; }
bool chain_next() { return t_chain_pos++ > 0; }
bool chain_all_programmatic() { return t_chain_all; }
ChainProgrammatic::ChainProgrammatic() { t_chain_all = true; }
ChainProgrammatic::~ChainProgrammatic() { t_chain_all = false; }

// A decode-sized batch streams every expert's weights whichever tokens reach
// them, so moe_forward evaluates every expert on all T tokens (the extra
// tensor-core work is hidden under the weight stream) and applies the routing
// in the combine: the GEMMs then wait for no routing step.  Chosen for bf16
// token-choice layers that drop on overflow, without shared experts, with
// T <= 64 (one token tile per expert in the single-CTA GEMM kernel, which the
// layer uses when T k < 96 E) and T k >= 4 E (each expert is expected to get
// four or more assignments, so hardly any expert's weights are streamed for
// nothing).
bool dense_decode(const moe_config& c) {
    return c.dtype == MOE_BF16 && c.routing == MOE_TOKEN_CHOICE && c.overflow == MOE_DROP &&
           c.n_shared == 0 && c.T > 0 && c.T <= 64 && (int64_t)c.T * c.k < 96LL * c.E &&
           (int64_t)c.T * c.k >= 4LL * c.E;
}

int num_sms() {
    static int sms[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (sms[dev] == 0) {
        int v = 148;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms[dev] = v;
    }
    return sms[dev];
}

cudaError_t launch_expert_ffn_simt(const moe_config& c, const void* x_perm, const int32_t* offsets,
                                   const void* W1, const void* b1, const void* W2, const void* b2,
                                   const float* perm_w, float* y_perm, void* h, int64_t max_seg,
                                   int64_t max_rows, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(DeviceHeader* hdr, uint64_t timeout_ns, cudaStream_t s);
cudaError_t launch_expert_ffn_tc(const moe_config& c, const void* x_perm, int64_t x_rows,
                                 const int32_t* offsets, const void* W1, const void* b1,
                                 const void* W2, const void* b2, const float* perm_w,
                                 float* y_perm, void* h, int64_t h_rows, DeviceHeader* hdr,
                                 int32_t* ksync, int32_t* ready, cudaStream_t s);

namespace {

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

size_t elem_size(const moe_config& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config* c) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d <= 0 || c->d_ff <= 0 || c->E <= 0 || c->k <= 0) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
    if (c->routing != MOE_TOKEN_CHOICE && c->routing != MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (c->overflow != MOE_DROP && c->overflow != MOE_REROUTE) return MOE_ERR_INVALID_ARG;
    if (c->n_shared < 0 || c->n_shared >= c->E) return MOE_ERR_INVALID_ARG;
    if (c->k > c->E - c->n_shared) return MOE_ERR_INVALID_ARG;
    if (c->E > kMaxExperts || c->k + c->n_shared > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (c->d % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_ALIGNMENT;
    if ((int64_t)c->T * (c->k + c->n_shared) > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (c->routing == MOE_EXPERT_CHOICE &&
        (c->n_shared != 0 || (int64_t)c->T * c->E > (int64_t)INT32_MAX / 2))
        return MOE_ERR_UNSUPPORTED;
    if (c->overflow == MOE_REROUTE &&
        (c->routing != MOE_TOKEN_CHOICE || c->n_shared != 0 || reroute_ranked(*c) > kMaxTopK))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

bool rerouting(const moe_config& c) { return c.overflow == MOE_REROUTE; }

bool expert_choice(const moe_config& c) { return c.routing == MOE_EXPERT_CHOICE; }

// The combine's view: K slots per token (expert choice: one per expert).
moe_config combine_config(const moe_config& c) {
    moe_config r = dispatch_config(c);
    if (expert_choice(c)) r.k = c.E;
    return r;
}

// Rows of the permuted buffers a stand-alone call may address: T*K for token
// choice (K = k + n_shared), E*C for expert choice.
int64_t call_rows(const moe_config& c) {
    return expert_choice(c) ? (int64_t)c.E * ec_capacity(c) : (int64_t)c.T * (c.k + c.n_shared);
}

moe_status check_ws(const moe_config& c, void* ws, size_t ws_bytes, WsLayout* L) {
    *L = ws_layout(c);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// T == 0: no token, no kernel; counts and the loss are defined as zero.
moe_status empty_batch(const moe_config& c, int32_t* expert_counts, float* aux_out,
                       float* z_loss_out, cudaStream_t s) {
    if (expert_counts && cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * c.E, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (aux_out && cudaMemsetAsync(aux_out, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (z_loss_out && cudaMemsetAsync(z_loss_out, 0, sizeof(float), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int64_t max_segment(const moe_config& c) {
    if (expert_choice(c)) return ec_capacity(c);
    int64_t m = c.T;  // a token reaches one expert at most once
    if (c.capacity >= 0 && c.capacity < m) m = c.capacity;
    return m;
}

}  // namespace

moe_status config_status(const moe_config* c) { return check_config(c); }

WsLayout ws_layout(const moe_config& c) {
    WsLayout L{};
    const bool ec = expert_choice(c);
    const moe_config cr = ec ? ec_router_config(c) : routed_config(c);
    // assignments of the router's top-k (token choice: all of them)
    const int64_t n = (int64_t)c.T * (ec ? 1 : c.k + c.n_shared);
    L.route = route_geom(cr);
    L.count_blocks = (int)((n + kCountBlock - 1) / kCountBlock);
    L.hist_blocks = L.route.blocks > L.count_blocks ? L.route.blocks : L.count_blocks;
    L.rows = n;
    if (ec) {
        L.rows = (int64_t)c.E * ec_capacity(c);
    } else if (c.capacity >= 0) {  // shared experts keep every token, routed ones at most capacity
        const int64_t cap_rows = (int64_t)c.n_shared * c.T + (int64_t)cr.E * c.capacity;
        if (cap_rows < L.rows) L.rows = cap_rows;
    }
    const int64_t slots = ec ? (int64_t)c.T * c.E : n;    // slot_of entries
    const int64_t perm = ec ? L.rows : n;                 // perm_token / perm_w entries
    const size_t es = elem_size(c);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.header = take(sizeof(DeviceHeader));
    L.counts = take(sizeof(int32_t) * c.E);
    L.top1 = take(sizeof(int32_t) * c.E);
    L.sched = take(sizeof(int32_t) * (1 + c.E));  // zeroed with the counts (same memset)
    // the fused expert FFN's counters: zeroed with the counts by the router's
    // memset (moe_expert_ffn zeroes them itself)
    L.ksync = take(sizeof(int32_t) * kKsyncCap);
    L.ready = take(sizeof(int32_t) * (size_t)ready_tiles(L.rows, c.E));
    L.blk_p = take(sizeof(float) * (size_t)L.route.blocks * cr.E);
    L.blk_z = take(sizeof(float) * (size_t)L.route.blocks);
    L.blk_hist = take(sizeof(int32_t) * (size_t)L.hist_blocks * c.E);
    L.blk_base = take(sizeof(int32_t) * (size_t)L.hist_blocks * c.E);
    L.local_rank = take(sizeof(int32_t) * (size_t)n);
    L.wsplit = take(L.route.tc ? sizeof(uint16_t) * 3 * (size_t)L.route.epad * c.d : 0);
    const size_t nr = c.n_shared > 0 ? (size_t)c.T * c.k : 0;
    L.route_idx = take(sizeof(int32_t) * nr);
    L.route_w = take(sizeof(float) * nr);
    const int64_t ranked = rerouting(c) ? (int64_t)c.T * reroute_ranked(c) : n;
    L.topk_idx = take(sizeof(int32_t) * (size_t)ranked);
    L.topk_w = take(sizeof(float) * (size_t)ranked);
    L.offsets = take(sizeof(int32_t) * (size_t)(c.E + 1));
    L.slot_of = take(sizeof(int32_t) * (size_t)slots);
    L.perm_token = take(sizeof(int32_t) * (size_t)perm);
    L.perm_w = take(sizeof(float) * (size_t)perm);
    // the dense decode path keeps every expert's rows for all T tokens in h and y_perm
    const int64_t frows = dense_decode(c) && (int64_t)c.E * c.T > L.rows ? (int64_t)c.E * c.T
                                                                        : L.rows;
    L.x_perm = take(es * (size_t)L.rows * c.d);
    L.h = take(es * (size_t)frows * c.d_ff);
    L.y_perm = take(sizeof(float) * (size_t)frows * c.d);
    L.probs_t = take(ec ? sizeof(float) * (size_t)c.E * c.T : 0);
    const bool rr = rerouting(c);
    L.rr_hist = take(rr ? sizeof(int32_t) * (size_t)L.count_blocks * c.E : 0);
    L.rr_base = take(rr ? sizeof(int32_t) * (size_t)L.count_blocks * c.E : 0);
    L.rr_rank = take(rr ? sizeof(int32_t) * (size_t)n : 0);
    L.rr_kept = take(rr ? sizeof(int32_t) * (size_t)n : 0);
    L.rr_alt = take(rr ? sizeof(int32_t) * (size_t)n : 0);
    L.rr_off1 = take(rr ? sizeof(int32_t) * (size_t)(c.E + 1) : 0);
    L.rr_off2 = take(rr ? sizeof(int32_t) * (size_t)(c.E + 1) : 0);
    L.total = o;
    return L;
}

cudaError_t launch_expert_ffn(const moe_config& c, const void* x_perm, int64_t x_rows,
                              const int32_t* offsets, const void* W1, const void* b1,
                              const void* W2, const void* b2, const float* perm_w, float* y_perm,
                              void* ws, const WsLayout& L, cudaStream_t s) {
    if (c.dtype == MOE_BF16)
        return launch_expert_ffn_tc(c, x_perm, x_rows, offsets, W1, b1, W2, b2, perm_w, y_perm,
                                    at<void>(ws, L.h), L.rows, at<DeviceHeader>(ws, L.header),
                                    at<int32_t>(ws, L.ksync), at<int32_t>(ws, L.ready), s);
    return launch_expert_ffn_simt(c, x_perm, offsets, W1, b1, W2, b2, perm_w, y_perm,
                                  at<void>(ws, L.h), max_segment(c), L.rows, s);
}

}  // namespace moe

using namespace moe;

extern "C" {

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t moe_workspace_size(const moe_config* cfg) {
    if (check_config(cfg) != MOE_OK) return 0;
    return ws_layout(*cfg).total;
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_ALIGNMENT: return "misaligned pointer or row length";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE: return "device-side error recorded";
    }
    return "unknown status";
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r,
                     const float* logit_bias, const float* logit_noise,
                     const float* logits_in, float* logits_out,
                     int32_t* topk_idx, float* topk_w, int32_t* expert_counts, float* aux_out,
                     float* z_loss_out, void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;  // moe_route_expert_choice
    WsLayout L;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c.T == 0) return empty_batch(c, expert_counts, aux_out, z_loss_out, s);
    if (topk_idx == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
    if (logits_in == nullptr && (x == nullptr || W_r == nullptr)) return MOE_ERR_INVALID_ARG;
    if (logits_in == nullptr && (!aligned16(x) || !aligned16(W_r))) return MOE_ERR_ALIGNMENT;
    if ((st = check_ws(c, ws, ws_bytes, &L)) != MOE_OK) return st;
    chain_begin();
    if (rerouting(c))  // K2 ranked experts per token, the first k the choices
        return from_cuda(launch_route(reroute_router_config(c), x, W_r, logit_bias, logit_noise,
                                      logits_in, logits_out, topk_idx, topk_w, expert_counts,
                                      aux_out, z_loss_out, ws, L, false, s, nullptr, c.k));
    if (c.n_shared == 0)
        return from_cuda(launch_route(c, x, W_r, logit_bias, logit_noise, logits_in, logits_out,
                                      topk_idx, topk_w, expert_counts, aux_out, z_loss_out, ws,
                                      L, false, s));
    // shared experts: route the routed experts into the workspace, then join
    int32_t* idx_r = at<int32_t>(ws, L.route_idx);
    float* w_r = at<float>(ws, L.route_w);
    cudaError_t e = launch_route(routed_config(c), x, W_r, logit_bias, logit_noise, logits_in,
                                 logits_out, idx_r, w_r, nullptr, aux_out, z_loss_out, ws, L,
                                 false, s);
    if (e == cudaSuccess)
        e = launch_join_shared(c, idx_r, w_r, topk_idx, topk_w, at<int32_t>(ws, L.counts),
                               expert_counts, s);
    return from_cuda(e);
}

moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        const float* topk_w, int32_t* offsets, int32_t* slot_of,
                        int32_t* perm_token, float* perm_w, void* x_perm,
                        void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;  // moe_route_expert_choice
    if (offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (c.T == 0) {
        const cudaError_t e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1),
                                              reinterpret_cast<cudaStream_t>(stream));
        return from_cuda(e);
    }
    if (x == nullptr || topk_idx == nullptr || slot_of == nullptr || perm_token == nullptr ||
        x_perm == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (perm_w != nullptr && topk_w == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    WsLayout L;
    if ((st = check_ws(c, ws, ws_bytes, &L)) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const moe_config cd = dispatch_config(c);
    chain_begin();
    if (rerouting(c))
        return from_cuda(launch_reroute_dispatch(c, reroute_ranked(c), x, topk_idx, topk_w,
                                                 offsets, slot_of, perm_token, perm_w, x_perm, ws,
                                                 L, LossArgs{}, s));
    cudaError_t e = launch_count(cd, topk_idx, ws, L, s);
    if (e == cudaSuccess)
        e = launch_scan_permute(cd, x, topk_idx, topk_w, kCountBlock, L.count_blocks, offsets,
                                slot_of, perm_token, perm_w, x_perm, ws, L, LossArgs{}, s);
    return from_cuda(e);
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const void* W1, const void* b1, const void* W2, const void* b2,
                          const float* perm_w, float* y_perm,
                          void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (x_perm == nullptr || offsets == nullptr || W1 == nullptr || b1 == nullptr ||
        W2 == nullptr || b2 == nullptr || y_perm == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(W1) || !aligned16(W2) || !aligned16(y_perm))
        return MOE_ERR_ALIGNMENT;
    WsLayout L;
    if ((st = check_ws(c, ws, ws_bytes, &L)) != MOE_OK) return st;
    const moe_config cd = dispatch_config(c);
    // the fused expert FFN's counters start at zero (moe_forward zeroes them
    // with the router's counts)
    const size_t cnt_end = L.ready + sizeof(int32_t) * (size_t)ready_tiles(L.rows, c.E);
    if (cudaMemsetAsync(at<char>(ws, L.ksync), 0, cnt_end - L.ksync,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    chain_begin();
    return from_cuda(launch_expert_ffn(cd, x_perm, call_rows(c), offsets, W1, b1, W2, b2,
                                       perm_w, y_perm, ws, L,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* slot_of,
                       void* y, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (y_perm == nullptr || slot_of == nullptr || y == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_ALIGNMENT;
    chain_begin();
    return from_cuda(launch_combine(combine_config(c), y_perm, slot_of, y, call_rows(c),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_r,
                       const float* logit_bias, const float* logit_noise,
                       const void* W1, const void* b1,
                       const void* W2, const void* b2, void* y, float* aux_out,
                       int32_t* expert_counts, float* logits_out, float* z_loss_out,
                       void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c.T == 0) return empty_batch(c, expert_counts, aux_out, z_loss_out, s);
    if (x == nullptr || W_r == nullptr || W1 == nullptr || b1 == nullptr || W2 == nullptr ||
        b2 == nullptr || y == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_r) || !aligned16(W1) || !aligned16(W2) || !aligned16(y))
        return MOE_ERR_ALIGNMENT;
    WsLayout L;
    if ((st = check_ws(c, ws, ws_bytes, &L)) != MOE_OK) return st;
    int32_t* idx = at<int32_t>(ws, L.topk_idx);
    float* w = at<float>(ws, L.topk_w);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* slot_of = at<int32_t>(ws, L.slot_of);
    int32_t* perm_token = at<int32_t>(ws, L.perm_token);
    float* perm_w = at<float>(ws, L.perm_w);
    void* x_perm = at<void>(ws, L.x_perm);
    float* y_perm = at<float>(ws, L.y_perm);
    const moe_config cd = dispatch_config(c);
    if (expert_choice(c)) {
        // no balancing loss under expert choice: aux is 0
        if (aux_out && cudaMemsetAsync(aux_out, 0, sizeof(float), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        chain_begin();
        cudaError_t e = launch_route(ec_router_config(c), x, W_r, logit_bias, logit_noise, nullptr,
                                     logits_out, idx, w, nullptr, nullptr, z_loss_out, ws, L,
                                     false, s, at<float>(ws, L.probs_t));
        if (e == cudaSuccess)
            e = launch_ec_select(c, at<float>(ws, L.probs_t), offsets, perm_token, perm_w,
                                 slot_of, expert_counts, s);
        if (e == cudaSuccess) e = launch_ec_gather(c, x, perm_token, x_perm, s);
        if (e == cudaSuccess)
            e = launch_expert_ffn(c, x_perm, L.rows, offsets, W1, b1, W2, b2, perm_w, y_perm, ws,
                                  L, s);
        if (e == cudaSuccess) e = launch_combine(combine_config(c), y_perm, slot_of, y, L.rows, s);
        return from_cuda(e);
    }
    if (dense_decode(c)) {
        // every expert on all T tokens: the router, then both expert GEMMs in
        // one persistent kernel that starts beside it (the GEMMs read only the
        // layer's inputs), then the combine, which applies the routing
        // weights and drops and finishes the loss.  The counters (router
        // counts, the FFN's work-item and ready counters) start at zero.
        if (cudaMemsetAsync(at<char>(ws, L.counts), 0, L.blk_p - L.counts, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        DeviceHeader* hdr = at<DeviceHeader>(ws, L.header);
        WsLayout Lr = L;  // the router in few blocks: it runs beside the FFN
        Lr.route = route_geom_beside(routed_config(c));
        chain_begin();
        ChainProgrammatic pdl_chain;
        cudaError_t e = launch_route_no_finish(c, x, W_r, logit_bias, logit_noise, logits_out, idx,
                                               w, ws, Lr, s);
        if (e == cudaSuccess)
            e = launch_dense_ffn(c, x, W1, b1, W2, b2, at<void>(ws, L.h), y_perm,
                                 at<int32_t>(ws, L.sched), hdr, s);
        if (e == cudaSuccess)
            e = launch_dense_combine(c, y_perm, idx, w, y, hdr,
                                     route_loss_args(c, ws, Lr, expert_counts, aux_out, z_loss_out),
                                     expert_counts != nullptr || aux_out != nullptr ||
                                         z_loss_out != nullptr,
                                     s);
        return from_cuda(e);
    }
    chain_begin();
    cudaError_t e;
    bool loss_in_combine = false;
    if (rerouting(c) && c.capacity >= 0) {
        // K2 ranked experts per token; the drop pass (whose scan also
        // finishes the loss and counts), the offers, the layout
        e = launch_route(reroute_router_config(c), x, W_r, logit_bias, logit_noise, nullptr,
                         logits_out, idx, w, nullptr, nullptr, nullptr, ws, L, false, s,
                         nullptr, c.k);
        if (e == cudaSuccess)
            e = launch_reroute_dispatch(
                c, reroute_ranked(c), x, idx, w, offsets, slot_of, perm_token, perm_w, x_perm, ws,
                L, route_loss_args(c, ws, L, expert_counts, aux_out, z_loss_out), s);
    } else if (c.n_shared == 0) {  // (rerouting without a cap drops nothing: this path)
        // the router also counts (blk_hist, local_rank); the combine finishes its loss
        e = launch_route(c, x, W_r, logit_bias, logit_noise, nullptr, logits_out, idx, w,
                         expert_counts, aux_out, z_loss_out, ws, L, true, s);
        if (e == cudaSuccess)
            e = launch_scan_permute(c, x, idx, w, L.route.tokens * c.k, L.route.blocks, offsets,
                                    slot_of, perm_token, perm_w, x_perm, ws, L, LossArgs{}, s);
        loss_in_combine = expert_counts != nullptr || aux_out != nullptr || z_loss_out != nullptr;
    } else {
        // shared experts: route the routed experts, join the shared ones, count all
        int32_t* idx_r = at<int32_t>(ws, L.route_idx);
        float* w_r = at<float>(ws, L.route_w);
        e = launch_route(routed_config(c), x, W_r, logit_bias, logit_noise, nullptr, logits_out,
                         idx_r, w_r, nullptr, aux_out, z_loss_out, ws, L, false, s);
        if (e == cudaSuccess)
            e = launch_join_shared(c, idx_r, w_r, idx, w, at<int32_t>(ws, L.counts),
                                   expert_counts, s);
        if (e == cudaSuccess) e = launch_count(cd, idx, ws, L, s);
        if (e == cudaSuccess)
            e = launch_scan_permute(cd, x, idx, w, kCountBlock, L.count_blocks, offsets, slot_of,
                                    perm_token, perm_w, x_perm, ws, L, LossArgs{}, s);
    }
    if (e == cudaSuccess)
        e = launch_expert_ffn(cd, x_perm, L.rows, offsets, W1, b1, W2, b2, perm_w, y_perm, ws,
                              L, s);
    if (e == cudaSuccess) {
        const LossArgs loss = route_loss_args(c, ws, L, expert_counts, aux_out, z_loss_out);
        e = launch_combine(cd, y_perm, slot_of, y, L.rows, s, loss_in_combine ? &loss : nullptr);
    }
    return from_cuda(e);
}

moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const float* W_r,
                                   const float* logit_bias, const float* logit_noise,
                                   const float* logits_in, float* logits_out, int32_t* offsets,
                                   int32_t* perm_token, float* perm_w, int32_t* slot_of,
                                   void* x_perm, int32_t* expert_counts, float* z_loss_out,
                                   void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (c.T == 0) {
        if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return empty_batch(c, expert_counts, nullptr, z_loss_out, s);
    }
    if (perm_token == nullptr || perm_w == nullptr || slot_of == nullptr) return MOE_ERR_INVALID_ARG;
    if (logits_in == nullptr && (x == nullptr || W_r == nullptr)) return MOE_ERR_INVALID_ARG;
    if (x_perm != nullptr && x == nullptr) return MOE_ERR_INVALID_ARG;
    if (logits_in == nullptr && (!aligned16(x) || !aligned16(W_r))) return MOE_ERR_ALIGNMENT;
    if (x_perm != nullptr && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_ALIGNMENT;
    WsLayout L;
    if ((st = check_ws(c, ws, ws_bytes, &L)) != MOE_OK) return st;
    chain_begin();
    cudaError_t e = launch_route(ec_router_config(c), x, W_r, logit_bias, logit_noise, logits_in,
                                 logits_out, at<int32_t>(ws, L.topk_idx), at<float>(ws, L.topk_w),
                                 nullptr, nullptr, z_loss_out, ws, L, false, s,
                                 at<float>(ws, L.probs_t));
    if (e == cudaSuccess)
        e = launch_ec_select(c, at<float>(ws, L.probs_t), offsets, perm_token, perm_w, slot_of,
                             expert_counts, s);
    if (e == cudaSuccess && x_perm != nullptr) e = launch_ec_gather(c, x, perm_token, x_perm, s);
    return from_cuda(e);
}

int32_t moe_expert_choice_capacity(const moe_config* cfg) {
    if (check_config(cfg) != MOE_OK) return -1;
    return ec_capacity(*cfg);
}

moe_status moe_update_balance_bias(const moe_config* cfg, const int32_t* expert_counts,
                                   float* logit_bias, float step, void* stream) {
    moe_status st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (expert_counts == nullptr || logit_bias == nullptr) return MOE_ERR_INVALID_ARG;
    chain_begin();
    return from_cuda(launch_balance_bias(*cfg, expert_counts, logit_bias, step,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_check_wait_timeout(void* ws, uint64_t timeout_ns, void* stream) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
    return from_cuda(launch_wait_timeout_probe(reinterpret_cast<DeviceHeader*>(ws), timeout_ns,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_get_device_error(void* ws, void* stream, int32_t* code, int32_t* info) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    DeviceHeader h;
    if (cudaMemcpy(&h, ws, sizeof(int32_t) * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (code) *code = h.err_code;
    if (info) *info = h.err_info;
    if (h.err_code == 0) return MOE_OK;
    if (cudaMemset(ws, 0, sizeof(int32_t) * 2) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE;
}

}  // extern "C"
