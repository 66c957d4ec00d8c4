// Grouped expert GEMMs on CUDA cores (fp32 FMA).
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer": every expert is Linear(d, d_ff) + bias, GELU,
// Linear(d_ff, d) + bias, applied to the rows dispatched to it.
//
// This is the exact-fp32 path (fp32 layers, where tensor-core TF32 would not
// meet an fp32 tolerance) and the path for shapes the tcgen05 kernels do not
// tile.  Each block computes a 64 x 64 tile C = A B^T of one expert segment
// (A: segment rows x K, B: that expert's weight, N x K, both K-major), with a
// 4 x 4 register tile per thread and 64-column shared-memory chunks.  The
// grid covers the largest possible segment; blocks past the end of their
// segment exit at once (offsets are read on the device).
//   GEMM1 epilogue: h = GELU(acc + b1) stored as the layer dtype.
//   GEMM2 epilogue: y = (acc + b2) * w_row stored as fp32.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 64, PAD = 4;
constexpr int KQ = BK / 16;  // 4-column groups each thread loads per operand and K slice

template <typename TIN, typename TOUT, bool GEMM1>
__global__ void __launch_bounds__(256) grouped_gemm_simt(
    const TIN* __restrict__ A, const int32_t* __restrict__ offsets, const TIN* __restrict__ W,
    const TIN* __restrict__ bias, const float* __restrict__ row_w, TOUT* __restrict__ C, int N,
    int K, int max_rows) {
    __shared__ float As[BK][BM + PAD];
    __shared__ float Bs[BK][BN + PAD];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.z;
    // segment bounds, clamped to the buffers (offsets come from device memory)
    const int seg1 = min(__ldg(offsets + e + 1), max_rows);
    const int seg0 = min(max(__ldg(offsets + e), 0), seg1);
    const int m0 = seg0 + blockIdx.y * BM;
    if (m0 >= seg1) return;
    const int n0 = blockIdx.x * BN;
    const TIN* We = W + (size_t)e * N * K;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    // loader: 64 rows x BK columns per operand, KQ groups of 4 consecutive
    // columns per thread; the next K slice is loaded into registers while
    // this one is multiplied (few, long K slices: the short fp32 layers are
    // latency-bound, one slice per load round trip)
    const int lr = tid / 4, lc = (tid % 4) * 4;
    float av[KQ][4], bv[KQ][4];
    auto load = [&](int k0) {
#pragma unroll
        for (int g = 0; g < KQ; ++g) {
            const int kk = k0 + lc + 16 * g;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool kin = kk + q < K;
                av[g][q] = (m0 + lr < seg1 && kin) ? to_f32(A[(size_t)(m0 + lr) * K + kk + q]) : 0.f;
                bv[g][q] = (n0 + lr < N && kin) ? to_f32(We[(size_t)(n0 + lr) * K + kk + q]) : 0.f;
            }
        }
    };
    load(0);
    for (int k0 = 0; k0 < K; k0 += BK) {
        __syncthreads();
#pragma unroll
        for (int g = 0; g < KQ; ++g)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                As[lc + 16 * g + q][lr] = av[g][q];
                Bs[lc + 16 * g + q][lr] = bv[g][q];
            }
        __syncthreads();
        if (k0 + BK < K) load(k0 + BK);
#pragma unroll
        for (int kq = 0; kq < BK; ++kq) {
            const float4 a4 = *reinterpret_cast<const float4*>(&As[kq][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kq][tx * 4]);
            const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
            const float br[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= seg1) continue;
        const float wr = GEMM1 ? 1.f : (row_w != nullptr ? __ldg(row_w + m) : 1.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            const float v = acc[i][j] + to_f32(bias[(size_t)e * N + n]);
            C[(size_t)m * N + n] = from_f32<TOUT>(GEMM1 ? gelu_erf(v) : v * wr);
        }
    }
}

template <typename TIN>
cudaError_t launch_t(const moe_config& c, const void* x_perm, const int32_t* offsets,
                     const void* W1, const void* b1, const void* W2, const void* b2,
                     const float* perm_w, float* y_perm, void* h, int64_t max_seg,
                     int64_t max_rows, cudaStream_t s) {
    const int mt = (int)((max_seg + BM - 1) / BM);
    if (mt == 0) return cudaSuccess;
    dim3 g1((c.d_ff + BN - 1) / BN, mt, c.E), g2((c.d + BN - 1) / BN, mt, c.E);
    const cudaError_t e = launch_kernel(
        grouped_gemm_simt<TIN, TIN, true>, g1, dim3(256), 0, s, 1, false,
        reinterpret_cast<const TIN*>(x_perm), offsets, reinterpret_cast<const TIN*>(W1),
        reinterpret_cast<const TIN*>(b1), (const float*)nullptr, reinterpret_cast<TIN*>(h),
        c.d_ff, c.d, (int)max_rows);
    if (e != cudaSuccess) return e;
    return launch_kernel(grouped_gemm_simt<TIN, float, false>, g2, dim3(256), 0, s, 1, false,
                         reinterpret_cast<const TIN*>(h), offsets,
                         reinterpret_cast<const TIN*>(W2), reinterpret_cast<const TIN*>(b2),
                         perm_w, y_perm, c.d, c.d_ff, (int)max_rows);
}

}  // namespace

cudaError_t launch_expert_ffn_simt(const moe_config& c, const void* x_perm, const int32_t* offsets,
                                   const void* W1, const void* b1, const void* W2, const void* b2,
                                   const float* perm_w, float* y_perm, void* h, int64_t max_seg,
                                   int64_t max_rows, cudaStream_t s) {
    if (c.dtype == MOE_BF16)
        return launch_t<__nv_bfloat16>(c, x_perm, offsets, W1, b1, W2, b2, perm_w, y_perm, h,
                                       max_seg, max_rows, s);
    return launch_t<float>(c, x_perm, offsets, W1, b1, W2, b2, perm_w, y_perm, h, max_seg,
                           max_rows, s);
}

}  // namespace moe
