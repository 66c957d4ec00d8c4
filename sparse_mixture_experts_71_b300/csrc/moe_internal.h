// Internal declarations shared by the kernels and the C-ABI layer of libmoe.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
// assignments covered by one block of the stand-alone counting kernel
constexpr int kCountBlock = 256;

// Device error record at the start of every workspace.
struct DeviceHeader {
    int32_t err_code;   // first error recorded (0 = none)
    int32_t err_info;
    int32_t pad[62];
};
static_assert(sizeof(DeviceHeader) == 256, "header is one 256-byte line");

enum DeviceError : int32_t { kErrExpertRange = 1, kErrTimeout = 2 };

// Shared experts: the router sees the routed experts only (E - n_shared of
// them, k picks); dispatch, the expert GEMMs and the combine see all E
// experts with K = k + n_shared assignments per token.  Both views equal the
// caller's config when n_shared == 0.
inline moe_config routed_config(const moe_config& c) {
    moe_config r = c;
    r.E = c.E - c.n_shared;
    r.n_shared = 0;
    return r;
}
inline moe_config dispatch_config(const moe_config& c) {
    moe_config r = c;
    r.k = c.k + c.n_shared;
    return r;
}

// How the router kernel tiles the batch: `warp` kernel (E <= 32: one warp per
// `tw` tokens, 8 warps per block) or `tile` kernel (SIMT GEMM tile).
struct RouteGeom {
    bool tc;           // tcgen05 kernel (bf16 x, 16 < E <= 64)
    bool mma;          // mma.sync kernel (bf16 x, E <= 16)
    int epad;          // rows per router-weight part (tensor-core kernels)
    int mt;            // 16-token tiles per block (tensor-core kernel)
    bool warp;
    int tw;            // tokens per warp group (warp kernel)
    int ds;            // warps splitting one group's d columns (warp kernel)
    int tokens;        // tokens per block
    int blocks;
};
RouteGeom route_geom(const moe_config& c);
// Geometry of a router that runs beside a long kernel and only has to finish
// before a later one (the dense decode path): the fewest blocks of the same
// kernel, never more than route_geom's (so it fits the workspace regions
// route_geom sized).
RouteGeom route_geom_beside(const moe_config& c);

// Tiles of the second expert GEMM whose K may be split in two (CTA-pair
// kernel): one first-half counter each in the workspace.
constexpr int kKsyncCap = 512;
// 256-token tiles the expert segments of `rows` permuted rows can form (one
// ready counter each for the fused expert FFN).
inline int ready_tiles(int64_t rows, int E) { return (int)((rows + 255) / 256) + E + 1; }

// Byte offsets of the workspace regions for one configuration.
struct WsLayout {
    size_t header;       // DeviceHeader
    size_t counts;       // int32 [E]   assignments per expert (all slots)
    size_t top1;         // int32 [E]   first-slot choices per expert
    size_t sched;        // int32 [1+E] work-item counter and per-expert ready counts (dense decode FFN)
    size_t ksync;        // int32 [kKsyncCap] second expert GEMM: first-K-half counts per tile
    size_t ready;        // int32 [ready_tiles] fused expert FFN: first-GEMM counts per token tile
    size_t blk_p;        // fp32 [route.blocks][E] per-block sums of p
    size_t blk_z;        // fp32 [route.blocks] per-block sums of the squared log-sum-exp
    size_t blk_hist;     // int32 [hist_blocks][E]
    size_t blk_base;     // int32 [hist_blocks][E]
    size_t local_rank;   // int32 [T*k]
    size_t wsplit;       // bf16 [3][roundup(E, 8)][d] router weight parts (tensor-core router)
    size_t route_idx;    // int32 [T*k] routed choices before the shared experts join (n_shared > 0)
    size_t route_w;      // fp32  [T*k]
    size_t topk_idx;     // int32 [T*K]     (moe_forward; K = k + n_shared)
    size_t topk_w;       // fp32  [T*k]     (moe_forward)
    size_t offsets;      // int32 [E+1]     (moe_forward)
    size_t slot_of;      // int32 [T*k]     (moe_forward)
    size_t perm_token;   // int32 [T*k]     (moe_forward)
    size_t perm_w;       // fp32  [T*k]     (moe_forward)
    size_t x_perm;       // dtype [rows][d] (moe_forward)
    size_t h;            // dtype [rows][d_ff]
    size_t y_perm;       // fp32  [rows][d] (moe_forward)
    size_t probs_t;      // fp32  [E][T] router probabilities (expert choice)
    size_t rr_hist;      // int32 [count_blocks][E] offer histograms (rerouting)
    size_t rr_base;      // int32 [count_blocks][E]
    size_t rr_rank;      // int32 [T*k] offer ranks within their block
    size_t rr_kept;      // int32 [T*k] drop-pass rank of a kept slot, -1 if dropped
    size_t rr_alt;       // int32 [T*k] expert a dropped slot is offered to, -1 if none
    size_t rr_off1;      // int32 [E+1] drop-pass offsets
    size_t rr_off2;      // int32 [E+1] offer-count prefix
    size_t total;
    RouteGeom route;
    int count_blocks;    // blocks of the stand-alone counting kernel
    int hist_blocks;     // max(route.blocks, count_blocks)
    int64_t rows;        // upper bound of kept assignments
};

WsLayout ws_layout(const moe_config& c);

// Host validation of a configuration (the status every entry point returns
// for an invalid one).
moe_status config_status(const moe_config* c);

// Kernel launches enqueued so far (moe_launch_count).
void count_launches(int n);
int num_sms();

// Raise kernel Kern's dynamic shared-memory limit, once per device.
template <auto Kern>
cudaError_t ensure_smem(int bytes) {
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable && done[dev]) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cacheable) done[dev] = true;
    return e;
}

// ---- kernel launches
// The kernels one entry point enqueues form a chain: the first is launched
// normally (it waits for whatever the caller enqueued before it), every later
// one with programmatic stream serialization, so its blocks may become
// resident and run their set-up while the previous kernel finishes; the
// kernel's pdl_wait() orders its memory accesses after the previous kernel.
// chain_begin() starts a new chain (at each entry point, and after any memset
// an entry point enqueues between kernels); chain_next() reports whether the
// next launch may use the attribute and advances the chain.
void chain_begin();
bool chain_next();
// While set (ChainProgrammatic), every launch after the first of the chain
// uses programmatic stream serialization, the SIMT kernels' included.
bool chain_all_programmatic();
struct ChainProgrammatic {
    ChainProgrammatic();
    ~ChainProgrammatic();
};

// Launch `kern` on stream s; cluster > 1 launches clusters of that many
// blocks along x.  `programmatic` lets the launch use programmatic stream
// serialization when it is not the first of its chain; the tensor-core
// kernels ask for it (their set-up - barriers, TMEM allocation, tensor-map
// prefetch - then overlaps the previous kernel's tail).  The short SIMT
// kernels do not: chained programmatically they ran slower on B300.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, int cluster, bool programmatic, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (chain_next() && (programmatic || chain_all_programmatic())) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

template <typename T> __host__ __device__ inline T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(base) + off);
}

// ---- launchers (kernels live in route.cu, dispatch.cu, gemm_*.cu, combine.cu)

// Router.  With `fuse_count` the router also writes, per router block, the
// expert histogram (blk_hist) and each assignment's rank among the block's
// earlier assignments to the same expert (local_rank), which the scan and
// permute kernels consume with granularity route.tokens * k.
// Without fuse_count the router also runs its one-block finishing kernel
// (loss, per-expert counts); with it the caller leaves that to the scan.
cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r,
                         const float* logit_bias, const float* logit_noise,
                         const float* logits_in, float* logits_out,
                         int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                         float* aux_out, float* z_loss_out, void* ws, const WsLayout& L,
                         bool fuse_count, cudaStream_t s, float* probs_t = nullptr,
                         int knorm = 0);
// knorm > 0 (rerouting): the router ranks c.k experts per token, of which the
// first knorm are the choices (counts, loss and weight normalisation) and the
// rest the next-best experts.

// Counting kernel over a strided id array (a = t*k + j reads idx[t*ld + j];
// skip_none: -1 means no assignment) and the scan of its block histograms
// (no shared experts; with loss.blk_p set it also finishes the router's
// loss and counts); granularity kCountBlock assignments.
struct LossArgs;
cudaError_t launch_count_strided(const int32_t* idx, int T, int k, int ld, int E, bool skip_none,
                                 int32_t* blk_hist, int32_t* local_rank, DeviceHeader* hdr,
                                 cudaStream_t s);
cudaError_t launch_scan(const int32_t* blk_hist, int nblk, int E, int capacity,
                        int32_t* blk_base, int32_t* offsets, const LossArgs& loss,
                        cudaStream_t s);

// Rerouting on overflow (reroute.cu): the drop pass, the offers of dropped
// slots to each token's next-best experts, and the layout and gather, from
// the router's K2 = ld ranked experts per token.
// With loss.blk_p set, the drop-pass scan also finishes the router's loss
// and counts (the forward pass).
cudaError_t launch_reroute_dispatch(const moe_config& c, int ld, const void* x,
                                    const int32_t* topk_idx, const float* topk_w,
                                    int32_t* offsets, int32_t* slot_of, int32_t* perm_token,
                                    float* perm_w, void* x_perm, void* ws, const WsLayout& L,
                                    const LossArgs& loss, cudaStream_t s);
inline int reroute_ranked(const moe_config& c) { return 2 * c.k < c.E ? 2 * c.k : c.E; }

// Router view of a rerouting layer: K2 ranked experts per token (the first k
// are the choices; the router gets knorm = k).
inline moe_config reroute_router_config(const moe_config& c) {
    moe_config r = c;
    r.k = reroute_ranked(c);
    r.overflow = MOE_DROP;
    return r;
}

// Router view of an expert-choice layer: p and the z-loss only (its top-1
// outputs go to scratch and are not used).
inline moe_config ec_router_config(const moe_config& c) {
    moe_config r = c;
    r.k = 1;
    r.capacity = -1;
    r.routing = MOE_TOKEN_CHOICE;
    return r;
}

// Backward pass of fp32 layers (backward_f32.cu): C = A B_e^T per expert
// segment with B_e = W[e] ([N][K]; epi 1: C = acc + bias and C2 = GELU(C);
// epi 2: C = (acc + bias) * row_w) or, with bkn, C = A W[e] (W[e] [K][N],
// no epilogue); C[e] = A_e^T B_e over each segment's rows ([E][M][N]); and
// dH *= GELU'(U) over the kept rows.
cudaError_t launch_seg_gemm_f32(bool bkn, int epi, const float* A, const int32_t* offsets, int E,
                                const float* W, const float* bias, const float* row_w, float* C,
                                float* C2, int N, int K, int64_t max_seg, int64_t rows_cap,
                                cudaStream_t s);
cudaError_t launch_seg_atb_f32(const float* A, const float* B, const int32_t* offsets, int E,
                               int M, int N, int64_t rows_cap, float* C, cudaStream_t s);
cudaError_t launch_gelu_grad_f32(const float* U, float* dH, const int32_t* offsets, int E, int F,
                                 int64_t rows_cap, cudaStream_t s);

// Backward pass of bf16 layers on the CTA-pair tcgen05 kernel (gemm_tc.cu):
//   launch_grouped_gemm_tc   out = A W_e^T (+ bias) per segment, W [E][n_out][K]
//                            (the forward pass's GEMMs; optionally the
//                            pre-activation beside the GELU output too);
//   launch_grouped_gemm_mn   out = A W_e per segment, W [E][K][n_out] read
//                            MN-major (bf16 out optionally times GELU'(U),
//                            with the rows' partial dots with GELU(U));
//   launch_segment_reduction_tc  out[e] = TOK_e^T WT_e over each segment's
//                            rows, both row-major [rows][*] and read MN-major
//                            through 2E per-segment tensor maps it writes
//                            into `maps` (workspace, 128-byte aligned).
// check_segment_maps: those maps' device-side edits against the driver's
// encoding (moe_check_segment_maps; ws of at least kSegMapCheckBytes).
cudaError_t launch_grouped_gemm_tc(const moe_config& c, bool bf16_out, bool act, const void* A,
                                   int64_t a_rows, const int32_t* offsets, const void* W,
                                   const void* bias, const float* row_w, void* out,
                                   int64_t out_rows, int n_out, int K, DeviceHeader* hdr,
                                   cudaStream_t s, void* pre_out = nullptr);
cudaError_t launch_grouped_gemm_mn(const moe_config& c, bool bf16_out, const void* A,
                                   int64_t a_rows, const int32_t* offsets, const void* W,
                                   const void* gelu_u, float* spart, void* out, int64_t out_rows,
                                   int n_out, int K, DeviceHeader* hdr, cudaStream_t s);
constexpr size_t kSegMapBytes = 128;  // one tensor map
cudaError_t launch_segment_reduction_tc(int E, const int32_t* offsets, int64_t rows_cap,
                                        const void* TOK, int tok_rows, const void* WT, int n_out,
                                        float* out, CUtensorMap* maps, DeviceHeader* hdr,
                                        cudaStream_t s);
constexpr size_t kSegMapCheckBytes = 3u << 20;
moe_status check_segment_maps(void* ws, size_t ws_bytes, cudaStream_t s);

// Expert choice (expert_choice.cu): C; the per-expert top-C selection from
// the router probabilities probs_t [E][T] (offsets, rows, slot_of [T][E]);
// the gather of the E*C rows.
int ec_capacity(const moe_config& c);
cudaError_t launch_ec_select(const moe_config& c, const float* probs_t, int32_t* offsets,
                             int32_t* perm_token, float* perm_w, int32_t* slot_of,
                             int32_t* expert_counts, cudaStream_t s);
cudaError_t launch_ec_gather(const moe_config& c, const void* x, const int32_t* perm_token,
                             void* x_perm, cudaStream_t s);

// Shared experts: K = k + n_shared columns per token from the router's k
// routed choices (ids offset by n_shared) followed by the shared experts with
// weight 1, and the per-expert counts over all E experts (shared: T).
cudaError_t launch_join_shared(const moe_config& c, const int32_t* idx_r, const float* w_r,
                               int32_t* topk_idx, float* topk_w, const int32_t* counts_r,
                               int32_t* expert_counts, cudaStream_t s);

// Auxiliary-loss-free balancing step on the router logit bias.
cudaError_t launch_balance_bias(const moe_config& c, const int32_t* counts, float* bias,
                                float step, cudaStream_t s);

// Counting kernel over topk_idx (granularity kCountBlock assignments).
cudaError_t launch_count(const moe_config& c, const int32_t* topk_idx, void* ws,
                         const WsLayout& L, cudaStream_t s);

// Scan of the block histograms and the permute/gather, given histograms of
// `hist_blocks` blocks of `asg_per_block` assignments.
// With loss.blk_p set, the scan kernel also computes the router's loss and
// per-expert counts (the forward pass); otherwise loss is ignored.
struct LossArgs;
cudaError_t launch_scan_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                                const float* topk_w, int asg_per_block, int hist_blocks,
                                int32_t* offsets, int32_t* slot_of, int32_t* perm_token,
                                float* perm_w, void* x_perm, void* ws, const WsLayout& L,
                                const LossArgs& loss, cudaStream_t s);
// Loss inputs/outputs of the router's per-block statistics in workspace ws.
LossArgs route_loss_args(const moe_config& c, void* ws, const WsLayout& L,
                         int32_t* expert_counts, float* aux_out, float* z_loss_out);

// Decode-sized layers that stream every expert's weights (dense_decode):
// moe_forward evaluates every expert on all T tokens, so the expert GEMMs do
// not depend on the routing (launch_dense_ffn in gemm_tc.cu, the combine in
// combine.cu).
bool dense_decode(const moe_config& c);
cudaError_t launch_dense_ffn(const moe_config& c, const void* x, const void* W1, const void* b1,
                             const void* W2, const void* b2, void* h_all, float* y_all,
                             int32_t* sched, DeviceHeader* hdr, cudaStream_t s);
cudaError_t launch_dense_combine(const moe_config& c, const float* y_all, const int32_t* idx,
                                 const float* w, void* y, DeviceHeader* hdr, const LossArgs& loss,
                                 bool do_loss, cudaStream_t s);
// The router kernel alone: no memset of its counters and no finishing
// kernel (the caller zeroes the counters and finishes the loss).
cudaError_t launch_route_no_finish(const moe_config& c, const void* x, const float* W_r,
                                   const float* logit_bias, const float* logit_noise,
                                   float* logits_out, int32_t* topk_idx, float* topk_w, void* ws,
                                   const WsLayout& L, cudaStream_t s);

cudaError_t launch_expert_ffn(const moe_config& c, const void* x_perm, int64_t x_rows,
                              const int32_t* offsets, const void* W1, const void* b1,
                              const void* W2, const void* b2, const float* perm_w, float* y_perm,
                              void* ws, const WsLayout& L, cudaStream_t s);

// rows: rows of y_perm (slots at or past it are skipped as dropped).  With
// `loss`, one more block finishes the router's loss and counts beside the
// combine (the forward pass).
cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* slot_of,
                           void* y, int64_t rows, cudaStream_t s,
                           const LossArgs* loss = nullptr);

}  // namespace moe
