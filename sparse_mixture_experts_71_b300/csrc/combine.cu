// Combine: the weighted expert outputs of each token summed back into token
// order.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer", step 3 (the output is the weighted combination of the
// selected experts' outputs; the weights were applied by the second expert
// GEMM).  A token whose assignments were all dropped by the capacity cap
// ("The central problem: load balancing") gets zero.
//
// One warp per (token, 512-column chunk), fp32 accumulation in slot order,
// 16-byte loads of the fp32 expert rows and 8- or 16-byte stores of y.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// With do_loss the grid's last block finishes the router's auxiliary loss,
// z-loss and per-expert counts (off the dispatch's critical path) while the
// others combine.
template <typename TY>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_of, int T,
                                                      int k, int d, long long rows,
                                                      TY* __restrict__ y, LossArgs loss,
                                                      int do_loss) {
    pdl_wait();
    pdl_trigger();
    if (do_loss && blockIdx.x == gridDim.x - 1) {
        __shared__ float s_part[256];
        __shared__ float s_d[kMaxExperts];
        loss_and_counts(loss, s_part, s_d);
        return;
    }
    const int lane = threadIdx.x % 32;
    const int nwarps = (gridDim.x - do_loss) * (blockDim.x / 32);
    const int nv = d / 4;                   // float4 columns per row
    const int nch = (nv + 127) / 128;       // 128-column chunks per row (4 per lane)
    const long long tasks = (long long)T * nch;
    for (long long task = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; task < tasks;
         task += nwarps) {
        const int t = (int)(task / nch);
        const int v0 = (int)(task % nch) * 128 + lane;
        float4 acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {  // slot order
            int sl = __ldg(slot_of + (size_t)t * k + j);
            if (sl < 0 || sl >= rows) continue;  // dropped (or outside y_perm)
            const float4* row = reinterpret_cast<const float4*>(y_perm + (size_t)sl * d);
            float4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + 32 * u < nv) q[u] = __ldg(row + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + 32 * u < nv) {
                    acc[u].x += q[u].x; acc[u].y += q[u].y;
                    acc[u].z += q[u].z; acc[u].w += q[u].w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v0 + 32 * u < nv) store4(y + (size_t)t * d + 4 * (v0 + 32 * u), acc[u]);
    }
}

// Combine of the dense decode path (see moe_forward): token t's output is the
// sum, over its kept slots j in slot order, of w[t][j] * y_all[e * T + t]
// with e = idx[t][j] (fp32; the product and the sum rounded separately, so
// the result is the sparse path's, whose second GEMM multiplies by the
// weight and whose combine adds in slot order), 0 if every slot was dropped.
// A slot is kept when fewer than `capacity` earlier assignments, in (token,
// slot) order, went to its expert (capacity < 0: no cap) - the rank the
// sparse dispatch computes, counted here directly (T <= 64).  An expert index
// outside [0, E) is skipped and recorded.  With do_loss the grid's last block
// finishes the router's auxiliary loss, z-loss and per-expert counts.
template <typename TY>
__global__ void __launch_bounds__(256) dense_combine_kernel(
    const float* __restrict__ y_all, const int32_t* __restrict__ idx, const float* __restrict__ w,
    int T, int k, int d, int E, int capacity, TY* __restrict__ y, DeviceHeader* hdr, LossArgs loss,
    int do_loss) {
    pdl_wait();
    pdl_trigger();
    if (do_loss && blockIdx.x == gridDim.x - 1) {  // the router's loss, beside the combine
        __shared__ float s_part[256];
        __shared__ float s_d[kMaxExperts];
        loss_and_counts(loss, s_part, s_d);
        return;
    }
    const int lane = threadIdx.x % 32;
    const int nwarps = (gridDim.x - do_loss) * (blockDim.x / 32);
    const int nv = d / 4;
    const int nch = (nv + 127) / 128;
    const long long tasks = (long long)T * nch;
    for (long long task = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; task < tasks;
         task += nwarps) {
        const int t = (int)(task / nch);
        const int v0 = (int)(task % nch) * 128 + lane;
        float4 acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {  // slot order
            const int a = t * k + j;
            const int e = __ldg(idx + a);
            if (e < 0 || e >= E) {
                if (lane == 0 && task % nch == 0) record_error(hdr, kErrExpertRange, t);
                continue;
            }
            if (capacity >= 0) {
                int before = 0;
                for (int b = lane; b < a; b += 32) before += __ldg(idx + b) == e;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
                if (before >= capacity) continue;  // dropped
            }
            const float wj = __ldg(w + a);
            const float4* row = reinterpret_cast<const float4*>(y_all + ((size_t)e * T + t) * d);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + 32 * u < nv) {
                    const float4 q = __ldg(row + v0 + 32 * u);
                    acc[u].x = __fadd_rn(acc[u].x, __fmul_rn(wj, q.x));
                    acc[u].y = __fadd_rn(acc[u].y, __fmul_rn(wj, q.y));
                    acc[u].z = __fadd_rn(acc[u].z, __fmul_rn(wj, q.z));
                    acc[u].w = __fadd_rn(acc[u].w, __fmul_rn(wj, q.w));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v0 + 32 * u < nv) store4(y + (size_t)t * d + 4 * (v0 + 32 * u), acc[u]);
    }
}

}  // namespace

cudaError_t launch_dense_combine(const moe_config& c, const float* y_all, const int32_t* idx,
                                 const float* w, void* y, DeviceHeader* hdr, const LossArgs& loss,
                                 bool do_loss, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    const long long tasks = (long long)c.T * ((c.d / 4 + 127) / 128);
    long long blocks = (tasks + 7) / 8;
    if (blocks > num_sms() * 8) blocks = num_sms() * 8;
    if (do_loss) ++blocks;
    return launch_kernel(dense_combine_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0,
                         s, 1, false, y_all, idx, w, c.T, c.k, c.d, c.E, c.capacity,
                         reinterpret_cast<__nv_bfloat16*>(y), hdr, loss, do_loss ? 1 : 0);
}

cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* slot_of,
                           void* y, int64_t rows, cudaStream_t s, const LossArgs* loss) {
    if (c.T == 0) return cudaSuccess;
    const long long tasks = (long long)c.T * ((c.d / 4 + 127) / 128);
    long long blocks = (tasks + 7) / 8;
    if (blocks > num_sms() * 8) blocks = num_sms() * 8;
    const int do_loss = loss != nullptr ? 1 : 0;
    const LossArgs l = loss != nullptr ? *loss : LossArgs{};
    if (c.dtype == MOE_BF16)
        return launch_kernel(combine_kernel<__nv_bfloat16>, dim3((unsigned)(blocks + do_loss)),
                             dim3(256), 0, s, 1, false, y_perm, slot_of, c.T, c.k, c.d,
                             (long long)rows, reinterpret_cast<__nv_bfloat16*>(y), l, do_loss);
    return launch_kernel(combine_kernel<float>, dim3((unsigned)(blocks + do_loss)), dim3(256), 0, s,
                         1, false, y_perm, slot_of, c.T, c.k, c.d, (long long)rows,
                         reinterpret_cast<float*>(y), l, do_loss);
}

}  // namespace moe
