// Dispatch: expert offsets, token-order capacity drop and the gather of token
// rows into expert-contiguous order.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer" (each expert receives the rows routed to it, in ascending
// token order) and section "The central problem: load balancing" (each expert
// takes at most `capacity` tokens; the overflow is dropped).
//
// A stable counting sort keyed by expert, in three kernels:
//   count   one block per kCountBlock consecutive assignments a = t*k + j:
//           per-block expert histogram and the rank of each assignment among
//           the block's earlier assignments to the same expert (warp match +
//           per-warp histograms; no atomics, so the result is exact).
//   scan    one block: for every (block, expert) the number of assignments to
//           that expert in earlier blocks, the per-expert totals, the kept
//           counts min(total, capacity) (shared experts: total) and their
//           exclusive prefix sum (offsets).
//   permute one warp per group of four assignments (looked up on four lanes at
//           once): rank = base + local rank; kept iff rank < capacity; row =
//           offsets[e] + rank; writes slot_of / perm_token / perm_w, then the
//           warp copies each kept token row with 16-byte vector accesses.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kWarps = kCountBlock / 32;

// Assignment a = t*k + j reads idx[t*ld + j]; with skip_none an id of -1 is
// "no assignment" (skipped without an error record).
__global__ void __launch_bounds__(kCountBlock) count_kernel(const int32_t* __restrict__ idx, int n,
                                                            int k, int ld, int E, bool skip_none,
                                                            int32_t* __restrict__ blk_hist,
                                                            int32_t* __restrict__ local_rank,
                                                            DeviceHeader* hdr) {
    __shared__ int wh[kWarps][kMaxExperts];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < kWarps * kMaxExperts; i += kCountBlock) (&wh[0][0])[i] = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int a = blockIdx.x * kCountBlock + tid;
    int e = -1;
    if (a < n) {
        e = __ldg(idx + (size_t)(a / k) * ld + a % k);
        if (e < 0 || e >= E) {
            if (!(skip_none && e == -1)) record_error(hdr, kErrExpertRange, a);
            e = -1;
        }
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0) wh[warp][e] = __popc(same);
    __syncthreads();
    if (a < n) {
        int r = -1;
        if (e >= 0) {
            r = rank_in_warp;
            for (int w = 0; w < warp; ++w) r += wh[w][e];
        }
        local_rank[a] = r;
    }
    for (int x = tid; x < E; x += kCountBlock) {
        int s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += wh[w][x];
        blk_hist[(size_t)blockIdx.x * E + x] = s;
    }
}

// One block of 1024 threads.  Thread (part, e) with part < P = 1024 / E owns
// a contiguous range of blocks for expert e.
// With loss.blk_p set it also finishes the router's statistics (loss and
// per-expert counts), which removes a launch from the layer's forward pass.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ blk_hist,
                                                    int nblk, int E, int capacity, int n_shared,
                                                    int32_t* __restrict__ blk_base,
                                                    int32_t* __restrict__ offsets, LossArgs loss) {
    __shared__ int part_sum[1024];
    __shared__ int s_total[kMaxExperts];
    __shared__ float s_part[256];
    __shared__ float s_d[kMaxExperts];
    pdl_wait();
    pdl_trigger();
    if (loss.blk_p != nullptr) loss_and_counts(loss, s_part, s_d);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int P = 1024 / E;
    const int part = tid / E, e = tid % E;
    const bool active = part < P;
    const int per = (nblk + P - 1) / P;
    const int b0 = part * per, b1 = min(nblk, b0 + per);
    int s = 0;
    if (active)
        for (int b = b0; b < b1; ++b) s += blk_hist[(size_t)b * E + e];
    part_sum[tid] = s;
    __syncthreads();
    // exclusive scan over the P parts of each expert: one warp per expert
    for (int x = warp; x < E; x += 32) {
        int carry_in = 0;
        for (int p0 = 0; p0 < P; p0 += 32) {
            const int p = p0 + lane;
            const int v = p < P ? part_sum[p * E + x] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (p < P) part_sum[p * E + x] = carry_in + incl - v;
            carry_in += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_total[x] = carry_in;
    }
    __syncthreads();
    if (active) {
        int run = part_sum[tid];
        for (int b = b0; b < b1; ++b) {
            blk_base[(size_t)b * E + e] = run;
            run += blk_hist[(size_t)b * E + e];
        }
    }
    if (warp == 0) {  // offsets: exclusive scan of the kept counts
        int carry_in = 0;
        for (int x0 = 0; x0 < E; x0 += 32) {
            const int x = x0 + lane;
            const int tot = x < E ? s_total[x] : 0;
            const int kept = capacity < 0 || x < n_shared ? tot : min(tot, capacity);
            int incl = kept;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (x < E) offsets[x] = carry_in + incl - kept;
            carry_in += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) offsets[E] = carry_in;
    }
}

// Assignments per permute group: the group's lanes 0 .. kPermG-1 look up
// their assignments' rows at the same time (four dependent loads each), then
// the warp copies the kept rows one after another.
constexpr int kPermG = 4;

template <typename TX>
__global__ void __launch_bounds__(256) permute_kernel(
    const TX* __restrict__ x, const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ local_rank, const int32_t* __restrict__ blk_base,
    const int32_t* __restrict__ offsets, int n, int k, int E, int d, int capacity, int n_shared,
    int asg_per_block, int32_t* __restrict__ slot_of, int32_t* __restrict__ perm_token, float* __restrict__ perm_w,
    TX* __restrict__ x_perm) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x % 32;
    const int nwarps = gridDim.x * (blockDim.x / 32);
    const int nvec = d * (int)sizeof(TX) / 16;  // 16-byte vectors per row
    for (int a0 = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kPermG; a0 < n;
         a0 += nwarps * kPermG) {
        const int a = a0 + lane;
        int slot = -1;
        if (lane < kPermG && a < n) {
            const int r_local = __ldg(local_rank + a);
            if (r_local >= 0) {
                const int e = __ldg(idx + a);
                const int r = __ldg(blk_base + (size_t)(a / asg_per_block) * E + e) + r_local;
                if (capacity < 0 || r < capacity || e < n_shared) slot = __ldg(offsets + e) + r;
            }
            slot_of[a] = slot;
            if (slot >= 0) {
                perm_token[slot] = a / k;
                if (perm_w != nullptr) perm_w[slot] = __ldg(topk_w + a);
            }
        }
        if (x_perm == nullptr) continue;
        unsigned kept = __ballot_sync(0xffffffffu, slot >= 0);
        while (kept) {
            const int src = __ffs(kept) - 1;
            kept &= kept - 1;
            const int sl = __shfl_sync(0xffffffffu, slot, src);
            const int t = (a0 + src) / k;
            const uint4* srow = reinterpret_cast<const uint4*>(x + (size_t)t * d);
            uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)sl * d);
            int v = lane;
            for (; v + 96 < nvec; v += 128) {
                const uint4 q0 = __ldg(srow + v), q1 = __ldg(srow + v + 32);
                const uint4 q2 = __ldg(srow + v + 64), q3 = __ldg(srow + v + 96);
                dst[v] = q0; dst[v + 32] = q1; dst[v + 64] = q2; dst[v + 96] = q3;
            }
            for (; v < nvec; v += 32) dst[v] = __ldg(srow + v);
        }
    }
}

}  // namespace

cudaError_t launch_count(const moe_config& c, const int32_t* topk_idx, void* ws,
                         const WsLayout& L, cudaStream_t s) {
    const int n = c.T * c.k;
    if (n == 0) return cudaSuccess;
    return launch_kernel(count_kernel, dim3(L.count_blocks), dim3(kCountBlock), 0, s, 1, false,
                         topk_idx, n, c.k, c.k, c.E, false, at<int32_t>(ws, L.blk_hist),
                         at<int32_t>(ws, L.local_rank), at<DeviceHeader>(ws, L.header));
}

cudaError_t launch_count_strided(const int32_t* idx, int T, int k, int ld, int E, bool skip_none,
                                 int32_t* blk_hist, int32_t* local_rank, DeviceHeader* hdr,
                                 cudaStream_t s) {
    const int n = T * k;
    if (n == 0) return cudaSuccess;
    return launch_kernel(count_kernel, dim3((n + kCountBlock - 1) / kCountBlock),
                         dim3(kCountBlock), 0, s, 1, false, idx, n, k, ld, E, skip_none, blk_hist,
                         local_rank, hdr);
}

cudaError_t launch_scan(const int32_t* blk_hist, int nblk, int E, int capacity,
                        int32_t* blk_base, int32_t* offsets, const LossArgs& loss,
                        cudaStream_t s) {
    return launch_kernel(scan_kernel, dim3(1), dim3(1024), 0, s, 1, false, blk_hist, nblk, E,
                         capacity, 0, blk_base, offsets, loss);
}

cudaError_t launch_scan_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                                const float* topk_w, int asg_per_block, int hist_blocks,
                                int32_t* offsets, int32_t* slot_of, int32_t* perm_token,
                                float* perm_w, void* x_perm, void* ws, const WsLayout& L,
                                const LossArgs& loss, cudaStream_t s) {
    const int n = c.T * c.k;
    int32_t* blk_hist = at<int32_t>(ws, L.blk_hist);
    int32_t* blk_base = at<int32_t>(ws, L.blk_base);
    int32_t* local_rank = at<int32_t>(ws, L.local_rank);
    cudaError_t e = launch_kernel(scan_kernel, dim3(1), dim3(1024), 0, s, 1, false,
                                  (const int32_t*)blk_hist, hist_blocks, c.E, c.capacity,
                                  c.n_shared, blk_base, offsets, loss);
    if (e != cudaSuccess || n == 0) return e;
    int blocks = (n + 8 * kPermG - 1) / (8 * kPermG);
    blocks = blocks < num_sms() * 8 ? blocks : num_sms() * 8;
    if (c.dtype == MOE_BF16)
        return launch_kernel(permute_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s, 1, false,
                             reinterpret_cast<const __nv_bfloat16*>(x), topk_idx, topk_w,
                             (const int32_t*)local_rank, (const int32_t*)blk_base,
                             (const int32_t*)offsets, n, c.k, c.E, c.d, c.capacity,
                             c.n_shared, asg_per_block, slot_of, perm_token, perm_w,
                             reinterpret_cast<__nv_bfloat16*>(x_perm));
    return launch_kernel(permute_kernel<float>, dim3(blocks), dim3(256), 0, s, 1, false,
                         reinterpret_cast<const float*>(x), topk_idx, topk_w,
                         (const int32_t*)local_rank, (const int32_t*)blk_base,
                         (const int32_t*)offsets, n, c.k, c.E, c.d, c.capacity, c.n_shared,
                         asg_per_block,
                         slot_of, perm_token, perm_w, reinterpret_cast<float*>(x_perm));
}

}  // namespace moe
