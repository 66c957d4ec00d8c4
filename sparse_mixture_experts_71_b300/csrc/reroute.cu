// Rerouting on overflow: a slot the capacity cap drops is offered once to the
// token's next-best expert.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The central problem: load balancing" (an overflowing token is dropped or
// sent elsewhere) and "Mixture of Experts (MoE)" (inferensys glossary),
// expert capacity (one option sends it to its next-ranked expert).  One hop:
// after
// the drop pass, the r-th dropped slot of a token goes to the token's
// (k + r)-th ranked expert; offers are taken in (token, slot) order while the
// expert's kept slots plus accepted offers stay below the capacity.
//
// Kernels, given the router's K2 ranked experts per token (ld = K2):
//   count    drop pass: the counting kernel over the first k columns
//   scan     drop-pass block bases and offsets (kept counts, capped)
//   offer    one thread per token: which slots the drop pass kept (their
//            rank; -1 dropped, -2 an invalid id) and the expert each dropped
//            slot is offered to
//   count    offers: the counting kernel over the offer ids (-1: none)
//   scan     offer block bases and the prefix of the offer totals (uncapped)
//   permute  final offsets (kept + accepted per expert), each slot's row
//            (kept: after the expert's earlier kept slots; accepted: after
//            all its kept slots and its earlier accepted offers), the gather.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) offer_kernel(
    const int32_t* __restrict__ idx, int T, int k, int ld, int E, int capacity,
    const int32_t* __restrict__ blk_base, const int32_t* __restrict__ local_rank,
    int32_t* __restrict__ kept_rank, int32_t* __restrict__ alt) {
    pdl_wait();
    pdl_trigger();
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        int r = 0;  // dropped slots of this token so far
        for (int j = 0; j < k; ++j) {
            const int a = t * k + j;
            const int e = __ldg(idx + (size_t)t * ld + j);
            const int lr = __ldg(local_rank + a);
            int rank = -2, to = -1;  // -2: an invalid id (flagged by the count), not dropped
            if (e >= 0 && e < E && lr >= 0) {
                const int rr = __ldg(blk_base + (size_t)(a / kCountBlock) * E + e) + lr;
                if (capacity < 0 || rr < capacity) {
                    rank = rr;
                } else {  // dropped (rank -1): offered to the next-best expert
                    rank = -1;
                    if (k + r < ld) to = __ldg(idx + (size_t)t * ld + k + r);
                    ++r;
                }
            }
            kept_rank[a] = rank;
            alt[a] = to;
        }
    }
}

template <typename TX>
__global__ void __launch_bounds__(256) reroute_permute_kernel(
    const TX* __restrict__ x, const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    int T, int k, int ld, int E, int d, int capacity, const int32_t* __restrict__ kept_rank,
    const int32_t* __restrict__ alt, const int32_t* __restrict__ off1,
    const int32_t* __restrict__ off2, const int32_t* __restrict__ blk_base2,
    const int32_t* __restrict__ local_rank2, int32_t* __restrict__ offsets,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ perm_token, float* __restrict__ perm_w,
    TX* __restrict__ x_perm) {
    __shared__ int s_off[kMaxExperts + 1], s_kept1[kMaxExperts], s_kept2[kMaxExperts];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid % 32;
    for (int e = tid; e < E; e += blockDim.x) {
        const int k1 = off1[e + 1] - off1[e];
        const int spare = capacity < 0 ? 0 : capacity - k1;  // no cap: nothing was dropped
        const int k2 = min(off2[e + 1] - off2[e], spare > 0 ? spare : 0);
        s_kept1[e] = k1;
        s_kept2[e] = k2;
    }
    __syncthreads();
    if (tid < 32) {  // exclusive prefix of kept + accepted, one warp
        int carry = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < E ? s_kept1[e] + s_kept2[e] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (e < E) s_off[e] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_off[E] = carry;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = tid; e <= E; e += blockDim.x) offsets[e] = s_off[e];

    const int n = T * k;
    const int nwarps = gridDim.x * (blockDim.x / 32);
    const int nvec = d * (int)sizeof(TX) / 16;
    for (int a = blockIdx.x * (blockDim.x / 32) + tid / 32; a < n; a += nwarps) {
        const int t = a / k, j = a % k;
        int row = -1;
        float w = 0.f;
        const int r1 = __ldg(kept_rank + a);
        if (r1 >= 0) {
            const int e = __ldg(idx + (size_t)t * ld + j);
            row = s_off[e] + r1;
            if (topk_w != nullptr) w = __ldg(topk_w + (size_t)t * ld + j);
        } else {
            const int e2 = __ldg(alt + a);
            const int lr2 = __ldg(local_rank2 + a);
            if (e2 >= 0 && e2 < E && lr2 >= 0) {
                const int r2 = __ldg(blk_base2 + (size_t)(a / kCountBlock) * E + e2) + lr2;
                if (r2 < s_kept2[e2]) {
                    row = s_off[e2] + s_kept1[e2] + r2;
                    int col = k;  // k + (dropped slots of the token before j)
                    for (int jj = 0; jj < j; ++jj) col += __ldg(kept_rank + t * k + jj) == -1;
                    if (topk_w != nullptr) w = __ldg(topk_w + (size_t)t * ld + col);
                }
            }
        }
        if (lane == 0) {
            slot_of[a] = row;
            if (row >= 0) {
                perm_token[row] = t;
                if (perm_w != nullptr) perm_w[row] = w;
            }
        }
        if (row < 0 || x_perm == nullptr) continue;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)row * d);
        int v = lane;
        for (; v + 96 < nvec; v += 128) {
            const uint4 q0 = __ldg(src + v), q1 = __ldg(src + v + 32);
            const uint4 q2 = __ldg(src + v + 64), q3 = __ldg(src + v + 96);
            dst[v] = q0; dst[v + 32] = q1; dst[v + 64] = q2; dst[v + 96] = q3;
        }
        for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
    }
}

}  // namespace

cudaError_t launch_reroute_dispatch(const moe_config& c, int ld, const void* x,
                                    const int32_t* topk_idx, const float* topk_w,
                                    int32_t* offsets, int32_t* slot_of, int32_t* perm_token,
                                    float* perm_w, void* x_perm, void* ws, const WsLayout& L,
                                    const LossArgs& loss, cudaStream_t s) {
    DeviceHeader* hdr = at<DeviceHeader>(ws, L.header);
    int32_t* kept_rank = at<int32_t>(ws, L.rr_kept);
    int32_t* alt = at<int32_t>(ws, L.rr_alt);
    int32_t* off1 = at<int32_t>(ws, L.rr_off1);
    int32_t* off2 = at<int32_t>(ws, L.rr_off2);
    const int nblk = (c.T * c.k + kCountBlock - 1) / kCountBlock;
    // drop pass
    cudaError_t e = launch_count_strided(topk_idx, c.T, c.k, ld, c.E, false,
                                         at<int32_t>(ws, L.blk_hist),
                                         at<int32_t>(ws, L.local_rank), hdr, s);
    if (e == cudaSuccess)
        e = launch_scan(at<int32_t>(ws, L.blk_hist), nblk, c.E, c.capacity,
                        at<int32_t>(ws, L.blk_base), off1, loss, s);
    // offers
    if (e == cudaSuccess) {
        int blocks = (c.T + 255) / 256;
        e = launch_kernel(offer_kernel, dim3(blocks), dim3(256), 0, s, 1, false, topk_idx, c.T,
                          c.k, ld, c.E, c.capacity, (const int32_t*)at<int32_t>(ws, L.blk_base),
                          (const int32_t*)at<int32_t>(ws, L.local_rank), kept_rank, alt);
    }
    if (e == cudaSuccess)
        e = launch_count_strided(alt, c.T * c.k, 1, 1, c.E, true, at<int32_t>(ws, L.rr_hist),
                                 at<int32_t>(ws, L.rr_rank), hdr, s);
    if (e == cudaSuccess)
        e = launch_scan(at<int32_t>(ws, L.rr_hist), nblk, c.E, -1, at<int32_t>(ws, L.rr_base),
                        off2, LossArgs{}, s);
    if (e != cudaSuccess) return e;
    // rows and gather
    int blocks = (c.T * c.k + 7) / 8;
    blocks = blocks < num_sms() * 8 ? blocks : num_sms() * 8;
    if (c.dtype == MOE_BF16)
        return launch_kernel(reroute_permute_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
                             1, false, reinterpret_cast<const __nv_bfloat16*>(x), topk_idx, topk_w,
                             c.T, c.k, ld, c.E, c.d, c.capacity, (const int32_t*)kept_rank,
                             (const int32_t*)alt, (const int32_t*)off1, (const int32_t*)off2,
                             (const int32_t*)at<int32_t>(ws, L.rr_base),
                             (const int32_t*)at<int32_t>(ws, L.rr_rank), offsets, slot_of,
                             perm_token, perm_w, reinterpret_cast<__nv_bfloat16*>(x_perm));
    return launch_kernel(reroute_permute_kernel<float>, dim3(blocks), dim3(256), 0, s, 1, false,
                         reinterpret_cast<const float*>(x), topk_idx, topk_w, c.T, c.k, ld, c.E,
                         c.d, c.capacity, (const int32_t*)kept_rank, (const int32_t*)alt,
                         (const int32_t*)off1, (const int32_t*)off2,
                         (const int32_t*)at<int32_t>(ws, L.rr_base),
                         (const int32_t*)at<int32_t>(ws, L.rr_rank), offsets, slot_of, perm_token,
                         perm_w, reinterpret_cast<float*>(x_perm));
}

}  // namespace moe
