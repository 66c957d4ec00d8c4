// Pieces shared by the router kernels (route.cu, route_tc.cu): argument
// block, per-token softmax / top-k, per-block statistics and the
// deterministic auxiliary-loss reduction.
#pragma once

#include <cuda_runtime.h>
#include <float.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace rt {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct RouteArgs {
    const void* x;
    const float* W_r;
    const float* bias;
    const float* noise;   // [T][E] added to the logits (noisy gating) or null
    const float* logits_in;
    float* logits_out;
    float* probs_t;       // [E][T] router probabilities (expert choice) or null
    int32_t* topk_idx;
    float* topk_w;
    int32_t* expert_counts;
    float* aux_out;
    DeviceHeader* hdr;
    int32_t* counts;      // ws: [E] all-slot assignments
    int32_t* top1;        // ws: [E] first-slot choices
    float* blk_p;         // ws: [nblk][E]
    float* blk_z;         // ws: [nblk] per-block sums of the squared log-sum-exp
    int32_t* blk_hist;    // ws: [nblk][E] or null (no fused counting)
    int32_t* local_rank;  // ws: [T*k]
    int T, d, E, k, renormalize, nblk;
    int knorm;            // slots that are choices (the rest: next-best experts)
};

// Histogram of the block's n assignments (expert ids in s_idx, in (token,
// slot) order) and the rank of each among the earlier ones of its expert.
template <int EMAX>
__device__ void block_rank(const int* s_idx, int n, int E, int (*wh)[EMAX], int* carry,
                           int32_t* hist_row, int32_t* rank_out) {
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int e = tid; e < E; e += kThreads) carry[e] = 0;
    for (int base = 0; base < n; base += kThreads) {
        for (int i = tid; i < kWarps * EMAX; i += kThreads) (&wh[0][0])[i] = 0;
        __syncthreads();
        const int a = base + tid;
        const int e = a < n ? s_idx[a] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int r = __popc(same & ((1u << lane) - 1u));
        if (e >= 0 && r == 0) wh[warp][e] = __popc(same);
        __syncthreads();
        if (e >= 0) {
            int rr = carry[e] + r;
            for (int w = 0; w < warp; ++w) rr += wh[w][e];
            rank_out[a] = rr;
        }
        __syncthreads();
        for (int x = tid; x < E; x += kThreads) {
            int s = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += wh[w][x];
            carry[x] += s;
        }
        __syncthreads();
    }
    for (int e = tid; e < E; e += kThreads) hist_row[e] = carry[e];
}

// Per-block sums of p (rows of s_p, fixed order) and of the squared
// log-sum-exp (column EMAX of s_p, the rows' pad slot), counts, and the fused
// dispatch histogram.
// blk: the block's index among the router blocks (its tokens start at
// blk * TB).
template <int EMAX>
__device__ void finish_block(const RouteArgs& a, const float* s_p, int lds, int TB,
                             const int* s_idx, const int* s_cnt, const int* s_top1,
                             int (*wh)[EMAX], int* carry, int blk) {
    const int tid = threadIdx.x;
    const int t0 = blk * TB;
    if (tid < 32) {  // warp 0: tokens tid, tid + 32, ... then a fixed shuffle tree
        float z = 0.f;
        for (int tok = tid; tok < TB; tok += 32) z += s_p[tok * lds + EMAX];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (tid == 0) a.blk_z[blk] = z;
    }
    if (a.probs_t != nullptr) {  // transposed, token-contiguous per expert
        const int n = min(TB, a.T - t0);
        for (int i = tid; i < n * a.E; i += kThreads) {
            const int e = i / n, tok = i % n;
            a.probs_t[(size_t)e * a.T + t0 + tok] = s_p[tok * lds + e];
        }
    }
    for (int e = tid; e < a.E; e += kThreads) {
        float v = 0.f;
        for (int tok = 0; tok < TB; ++tok) v += s_p[tok * lds + e];
        a.blk_p[(size_t)blk * a.E + e] = v;
        if (s_cnt[e]) atomicAdd(&a.counts[e], s_cnt[e]);
        if (s_top1[e]) atomicAdd(&a.top1[e], s_top1[e]);
    }
    if (a.blk_hist != nullptr) {
        const int n = min(TB, a.T - t0) * a.k;
        block_rank<EMAX>(s_idx, n, a.E, wh, carry, a.blk_hist + (size_t)blk * a.E,
                         a.local_rank + (size_t)t0 * a.k);
    }
}

// The block's staged logits (rows of s_rows, lds apart; TB tokens from t0)
// finished by the whole block before the per-token pass: the caller's
// noise [T][E] added (noisy gating) and the logits written to logits_out.
// The block's rows of both arrays are one contiguous range of TB * E
// floats, so consecutive threads take consecutive floats (coalesced), where
// a thread per token would stride E floats between neighbouring lanes.
template <int EMAX>
__device__ void stage_logits(const RouteArgs& a, float* s_rows, int lds, int TB, int t0) {
    if (a.noise == nullptr && a.logits_out == nullptr) return;
    const int n = min(TB, a.T - t0) * a.E;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int tok = i / a.E, e = i - tok * a.E;
        float g = s_rows[tok * lds + e];
        if (a.noise != nullptr) {
            g += __ldg(a.noise + (size_t)t0 * a.E + i);
            s_rows[tok * lds + e] = g;  // the logits used for routing
        }
        if (a.logits_out != nullptr) a.logits_out[(size_t)t0 * a.E + i] = g;
    }
}

// Softmax, top-k and gate weights of token t from its logits in prow
// (EMAX slots, E used; noise already added by stage_logits); the
// probabilities replace the logits in prow (zeros for a token past the end
// of the batch).  One thread per token.
template <int EMAX>
__device__ __forceinline__ void token_epilogue(const RouteArgs& a, float* prow, int t, int slot,
                                               int* s_idx, int* s_cnt, int* s_top1) {
    if (t >= a.T) {
#pragma unroll
        for (int e = 0; e <= EMAX; ++e) prow[e] = 0.f;
        return;
    }
    float g[EMAX];
    float m = -FLT_MAX;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        g[e] = e < a.E ? prow[e] : -FLT_MAX;
        m = fmaxf(m, g[e]);
    }
    // exp(g - m) is evaluated where it is needed rather than kept (one more
    // register array would not fit at two tcgen05-router CTAs per SM); expf
    // gives the same value for the same argument each time
    float ssum = 0.f;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) ssum += e < a.E ? expf(g[e] - m) : 0.f;
    const float inv = 1.0f / ssum;
    const float lse = m + logf(ssum);
    prow[EMAX] = lse * lse;  // squared log-sum-exp (router z-loss), the row's pad slot
#pragma unroll
    for (int e = 0; e < EMAX; ++e) prow[e] = (e < a.E ? expf(g[e] - m) : 0.f) * inv;  // p replaces g
    // top-k on the logits, larger first, ties to the lower expert index
    uint64_t taken = 0;
    int sel_e[kMaxTopK];
    float sel_x[kMaxTopK];
    float sel_sum = 0.f;
    for (int j = 0; j < a.k; ++j) {
        float bv = -FLT_MAX, bx;
        int be = -1;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            if (e < a.E && !((taken >> e) & 1ull) && (be < 0 || g[e] > bv)) {
                bv = g[e];
                be = e;
            }
        }
        bx = expf(bv - m);
        taken |= 1ull << be;
        sel_e[j] = be;
        sel_x[j] = bx;
        sel_sum += j < a.knorm ? bx : 0.f;
    }
    const float wden = a.renormalize ? 1.0f / sel_sum : inv;
    for (int j = 0; j < a.k; ++j) {
        a.topk_idx[(size_t)t * a.k + j] = sel_e[j];
        a.topk_w[(size_t)t * a.k + j] = sel_x[j] * wden;
        s_idx[slot * a.k + j] = sel_e[j];
        if (j < a.knorm) atomicAdd(&s_cnt[sel_e[j]], 1);
    }
    atomicAdd(&s_top1[sel_e[0]], 1);
}

// token_epilogue with two threads per token (lanes 2j and 2j + 1 of a warp,
// half = the lane's low bit), for EMAX = 64: each thread holds the
// exponentials of its 32 logits (experts half * 32 + i), so every exp is
// taken once, and the pair combines its maximum, sum and top-k candidates
// with one shuffle each; both threads end with the same values.  The sum of
// exponentials is each half's sum in expert order, then the two added
// (a different rounding order from token_epilogue's single sweep).  Half 0
// writes the token's outputs.
template <int EMAX>
__device__ __forceinline__ void token_epilogue_pair(const RouteArgs& a, float* prow, int t,
                                                    int slot, int half, int* s_idx, int* s_cnt,
                                                    int* s_top1) {
    static_assert(EMAX == 64, "two halves of 32 experts");
    constexpr int H = EMAX / 2;
    float* ph = prow + half * H;
    // a token past the end of the batch still runs the pair's shuffles (every
    // lane of the warp takes part) on zero logits, then writes zeros
    const bool valid = t < a.T;
    const int e0 = half * H;
    float x[H];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        x[i] = e0 + i < a.E ? (valid ? ph[i] : 0.f) : -FLT_MAX;
        m = fmaxf(m, x[i]);
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    // top-k on the logits (x still holds them), larger first, ties to the
    // lower expert index; each round takes the pair's better candidate
    uint32_t taken = 0;
    int sel_e[kMaxTopK];
    float sel_g[kMaxTopK];
    for (int j = 0; j < a.k; ++j) {
        float bv = -FLT_MAX;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < H; ++i)
            if (e0 + i < a.E && !((taken >> i) & 1u) && (be == 0x7fffffff || x[i] > bv)) {
                bv = x[i];
                be = e0 + i;
            }
        const float ov = __shfl_xor_sync(0xffffffffu, bv, 1);
        const int oe = __shfl_xor_sync(0xffffffffu, be, 1);
        if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
            bv = ov;
            be = oe;
        }
        if (be >= e0 && be < e0 + H) taken |= 1u << (be - e0);
        sel_e[j] = be;
        sel_g[j] = bv;
    }
    float ssum = 0.f;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        x[i] = e0 + i < a.E ? expf(x[i] - m) : 0.f;
        ssum += x[i];
    }
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);  // a + b == b + a: the same on both
    const float inv = 1.0f / ssum;
    if (half == 0) {
        const float lse = m + logf(ssum);
        prow[EMAX] = valid ? lse * lse : 0.f;  // squared log-sum-exp (router z-loss), pad slot
    }
#pragma unroll
    for (int i = 0; i < H; ++i) ph[i] = valid ? x[i] * inv : 0.f;  // p replaces g
    if (half != 0 || !valid) return;
    float sel_x[kMaxTopK];
    float sel_sum = 0.f;
    for (int j = 0; j < a.k; ++j) {
        sel_x[j] = expf(sel_g[j] - m);
        sel_sum += j < a.knorm ? sel_x[j] : 0.f;
    }
    const float wden = a.renormalize ? 1.0f / sel_sum : inv;
    for (int j = 0; j < a.k; ++j) {
        a.topk_idx[(size_t)t * a.k + j] = sel_e[j];
        a.topk_w[(size_t)t * a.k + j] = sel_x[j] * wden;
        s_idx[slot * a.k + j] = sel_e[j];
        if (j < a.knorm) atomicAdd(&s_cnt[sel_e[j]], 1);
    }
    atomicAdd(&s_top1[sel_e[0]], 1);
}

// tcgen05 router (route_tc.cu); np = rows per weight part (16, 32 or 64).
cudaError_t launch_route_tc(const RouteArgs& a, const __nv_bfloat16* wsplit, int np,
                            cudaStream_t s);

}  // namespace rt
}  // namespace moe
