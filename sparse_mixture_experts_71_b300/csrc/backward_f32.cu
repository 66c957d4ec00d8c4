// The expert GEMMs of the backward pass for fp32 layers, on CUDA cores (fp32
// FMA, no tensor-core rounding), over the expert segments of the permuted
// rows.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer": each expert is Linear(d, d_ff) + bias, GELU,
// Linear(d_ff, d) + bias; the layer is trained end to end, so the backward
// pass differentiates those two linear maps and the activation:
//   U = X W1_e^T + b1, H = GELU(U), Y = w (H W2_e^T + b2)   (the recompute)
//   dH = dY W2_e, dU = dH * GELU'(U), dX = dU W1_e           (seg_gemm_f32)
//   dW2_e = dY_e^T H_e, dW1_e = dU_e^T X_e                   (seg_atb_f32)
// with dY the routing-weighted upstream rows.  GELU is the exact
// 0.5 u (1 + erf(u / sqrt 2)) of the fp32 forward pass, and GELU'(u) =
// Phi(u) + u phi(u) with the CUDA erff / expf.
//
// Tiles: 64 x 64 outputs a block, 4 x 4 a thread, K in chunks of 32 staged
// in shared memory (each operand transposed so the inner loop reads float4
// along the output tile).  Every accumulation runs over K in increasing
// order; the segment bounds come from the device offsets.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int GB = 64, GK = 32, GPAD = 4;

enum SegEpi {
    kEpiPlain = 0,  // C = acc
    kEpiPreAct = 1,  // C = acc + bias (the pre-activation U), C2 = GELU(C)
    kEpiScaled = 2,  // C = (acc + bias) * row_w[r]
};

// Rows [s0, s1) of expert e's segment, clamped to the buffers.
__device__ __forceinline__ void seg_bounds(const int32_t* offsets, int e, int64_t rows_cap,
                                           int& s0, int& s1) {
    s1 = (int)min((int64_t)max(__ldg(offsets + e + 1), 0), rows_cap);
    s0 = min(max(__ldg(offsets + e), 0), s1);
}

// C[r][n] = sum_k A[r][k] B_e(n, k) for the rows r of segment e = blockIdx.z,
// where B_e(n, k) = W[e][n][k] (BKN false: the weight as the forward GEMMs
// use it) or W[e][k][n] (BKN true), then the epilogue.  A: [rows][K];
// C, C2: [rows][N].
template <bool BKN, int EPI>
__global__ void __launch_bounds__(256) seg_gemm_f32(const float* __restrict__ A,
                                                     const int32_t* __restrict__ offsets,
                                                     const float* __restrict__ W,
                                                     const float* __restrict__ bias,
                                                     const float* __restrict__ row_w,
                                                     float* __restrict__ C, float* __restrict__ C2,
                                                     int N, int K, int64_t rows_cap) {
    __shared__ float As[GK][GB + GPAD];
    __shared__ float Bs[GK][GB + GPAD];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.z;
    int s0, s1;
    seg_bounds(offsets, e, rows_cap, s0, s1);
    const int m0 = s0 + blockIdx.y * GB;
    if (m0 >= s1) return;
    const int n0 = blockIdx.x * GB;
    const float* We = W + (size_t)e * N * K;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += GK) {
        __syncthreads();
        for (int i = tid; i < GB * GK; i += 256) {
            const int r = i / GK, kk = i % GK;  // A: consecutive threads along k
            As[kk][r] = (m0 + r < s1 && k0 + kk < K) ? __ldg(A + (size_t)(m0 + r) * K + k0 + kk)
                                                     : 0.f;
            float b;
            if (BKN) {  // W[e][k][n]: consecutive threads along n
                const int kb = i / GB, nb = i % GB;
                b = (n0 + nb < N && k0 + kb < K) ? __ldg(We + (size_t)(k0 + kb) * N + n0 + nb) : 0.f;
                Bs[kb][nb] = b;
            } else {  // W[e][n][k]: consecutive threads along k
                b = (n0 + r < N && k0 + kk < K) ? __ldg(We + (size_t)(n0 + r) * K + k0 + kk) : 0.f;
                Bs[kk][r] = b;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int kq = 0; kq < GK; ++kq) {
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
        if (m >= s1) continue;
        const float wr = EPI == kEpiScaled ? __ldg(row_w + m) : 1.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            const size_t o = (size_t)m * N + n;
            if (EPI == kEpiPlain) {
                C[o] = acc[i][j];
            } else {
                const float v = acc[i][j] + __ldg(bias + (size_t)e * N + n);
                if (EPI == kEpiPreAct) {
                    C[o] = v;
                    C2[o] = gelu_erf(v);
                } else {
                    C[o] = v * wr;
                }
            }
        }
    }
}

// C[e][m][n] = sum over the rows r of segment e = blockIdx.z of A[r][m] B[r][n]
// (A: [rows][M], B: [rows][N], C: [E][M][N]); an empty segment gives zeros.
__global__ void __launch_bounds__(256) seg_atb_f32(const float* __restrict__ A,
                                                    const float* __restrict__ B,
                                                    const int32_t* __restrict__ offsets, int M,
                                                    int N, int64_t rows_cap,
                                                    float* __restrict__ C) {
    __shared__ float As[GK][GB + GPAD];
    __shared__ float Bs[GK][GB + GPAD];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.z;
    int s0, s1;
    seg_bounds(offsets, e, rows_cap, s0, s1);
    const int m0 = blockIdx.y * GB, n0 = blockIdx.x * GB;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int r0 = s0; r0 < s1; r0 += GK) {
        __syncthreads();
        for (int i = tid; i < GB * GK; i += 256) {
            const int kk = i / GB, c = i % GB;  // consecutive threads along the row
            const bool rin = r0 + kk < s1;
            As[kk][c] = (rin && m0 + c < M) ? __ldg(A + (size_t)(r0 + kk) * M + m0 + c) : 0.f;
            Bs[kk][c] = (rin && n0 + c < N) ? __ldg(B + (size_t)(r0 + kk) * N + n0 + c) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kq = 0; kq < GK; ++kq) {
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
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < N) C[((size_t)e * M + m) * N + n] = acc[i][j];
        }
    }
}

// dU = dH * GELU'(U) in place over the kept rows (offsets[E] of them):
// GELU'(u) = Phi(u) + u phi(u), Phi(u) = (1 + erf(u / sqrt 2)) / 2,
// phi(u) = exp(-u^2 / 2) / sqrt(2 pi).
__global__ void __launch_bounds__(256) gelu_grad_f32(const float* __restrict__ U,
                                                      float* __restrict__ dH,
                                                      const int32_t* __restrict__ offsets, int E,
                                                      int F, int64_t rows_cap) {
    pdl_wait();
    pdl_trigger();
    const int64_t rows = min((int64_t)max(__ldg(offsets + E), 0), rows_cap);
    const int64_t n = rows * F;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float u = __ldg(U + i);
        const float cdf = 0.5f * (1.0f + erff(u * 0.70710678118654752440f));
        const float pdf = expf(-0.5f * u * u) * 0.39894228040143267794f;
        dH[i] *= cdf + u * pdf;
    }
}

}  // namespace

cudaError_t launch_seg_gemm_f32(bool bkn, int epi, const float* A, const int32_t* offsets, int E,
                                const float* W, const float* bias, const float* row_w, float* C,
                                float* C2, int N, int K, int64_t max_seg, int64_t rows_cap,
                                cudaStream_t s) {
    const int mt = (int)((max_seg + GB - 1) / GB);
    if (mt == 0 || E == 0) return cudaSuccess;
    const dim3 grid((unsigned)((N + GB - 1) / GB), (unsigned)mt, (unsigned)E);
    if (bkn)
        return launch_kernel(seg_gemm_f32<true, kEpiPlain>, grid, dim3(256), 0, s, 1, false, A,
                             offsets, W, bias, row_w, C, C2, N, K, rows_cap);
    if (epi == kEpiPreAct)
        return launch_kernel(seg_gemm_f32<false, kEpiPreAct>, grid, dim3(256), 0, s, 1, false, A,
                             offsets, W, bias, row_w, C, C2, N, K, rows_cap);
    return launch_kernel(seg_gemm_f32<false, kEpiScaled>, grid, dim3(256), 0, s, 1, false, A,
                         offsets, W, bias, row_w, C, C2, N, K, rows_cap);
}

cudaError_t launch_seg_atb_f32(const float* A, const float* B, const int32_t* offsets, int E,
                               int M, int N, int64_t rows_cap, float* C, cudaStream_t s) {
    const dim3 grid((unsigned)((N + GB - 1) / GB), (unsigned)((M + GB - 1) / GB), (unsigned)E);
    return launch_kernel(seg_atb_f32, grid, dim3(256), 0, s, 1, false, A, B, offsets, M, N,
                         rows_cap, C);
}

cudaError_t launch_gelu_grad_f32(const float* U, float* dH, const int32_t* offsets, int E, int F,
                                 int64_t rows_cap, cudaStream_t s) {
    int64_t blocks = (rows_cap * F + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_kernel(gelu_grad_f32, dim3((unsigned)blocks), dim3(256), 0, s, 1, false, U, dH,
                         offsets, E, F, rows_cap);
}

}  // namespace moe
