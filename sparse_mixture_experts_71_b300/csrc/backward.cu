// Backward pass of the layer (include/moe_backward.h): the gradients of
// <dy, y> + aux_grad * aux + z_grad * z_loss with the routing held fixed.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer" (the layer being trained) and "The central problem: load
// balancing" (the auxiliary loss and the router z-loss it is trained with).
//
// Steps (one stream), bf16 layers:
//   recompute   router (logits kept) + dispatch, GEMM1 -> H = GELU(u) and the
//               pre-activation U (both bf16, from the fp32 accumulator, as the
//               forward's H)
//   dY_perm     the scaled upstream rows w_j dy_t of every kept slot
//   dH          dH = dY_perm W2_e on the CTA-pair tcgen05 kernel with W2 read
//               MN-major as stored (W2_e [d][d_ff] is dH's [K][N]); its
//               epilogue writes dU = dH * GELU'(U) and, per 16 columns, the
//               row's dot with GELU(U): the slot score s_j = <dy_t, w_j o_j> =
//               <dH_j, h_j> + w_j <dy_t, b2_e> then needs no second-GEMM
//               recompute
//   router      one warp per token: the slot scores, the logit gradient dg
//               (softmax / renormalisation, auxiliary loss, z-loss)
//   dx path     dX_perm = dU W1_e (W1 MN-major); dx = sum over the token's
//               slots of dX_perm + dg W_r (with 16-64 routed experts that
//               product as tf32 mma.sync tiles)
//   weights     dW2_e = dY_perm_e^T H_e and dW1_e = dU_e^T X_perm_e on the
//               same kernel in its segment-reduction mode (K = the segment's
//               rows; both operands read MN-major from the row-major
//               permuted rows through per-segment tensor maps, so a segment's
//               last K stage reads zeros past its end), dW_r = dg^T x
//               (row-slice partials summed in a fixed order; CUDA cores, or
//               tf32 mma.sync tiles with 16-64 routed experts), db2, db1
//               = column sums over each expert's rows.  GELU and GELU' use
//               the forward epilogue's Abramowitz & Stegun 7.1.26 erf.
// fp32 layers run the same steps on CUDA-core kernels (backward_f32.cu),
// with the second GEMM recomputed for the slot scores.

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/moe_backward.h"
#include "moe_device.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {


using bf16 = __nv_bfloat16;

__device__ __forceinline__ void unpack8(uint4 q, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return q;
}

// Eight consecutive elements of a bf16 or fp32 row (16- / 32-byte aligned).
__device__ __forceinline__ void load8(const bf16* p, float* f) {
    unpack8(__ldg(reinterpret_cast<const uint4*>(p)), f);
}
__device__ __forceinline__ void load8(const float* p, float* f) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(bf16* p, const float* f) {
    *reinterpret_cast<uint4*>(p) = pack8(f);
}
__device__ __forceinline__ void store8(float* p, const float* f) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ float2 load2(const bf16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 load2(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}

// How the routed slots of a token map to logit columns (router_grad_kernel).
enum GradMode {
    kGradChoice = 0,   // slot j < kr: the token's choice j (shared experts: routed ids)
    kGradReroute = 1,  // slot j: its choice if the drop pass kept it, else the expert it moved to
    kGradExpert = 2,   // expert choice: slot j is expert j
};

// One warp per token: the slot scores s_j = <dy_t, w_j o_j> over its K slots
// (w_j = perm_w of the slot's row), the dY_perm rows w_j dy_t, and the logit
// gradient dg[t][:] over the El routed experts:
//   dg_m = sum over the routed slots whose final expert is m of s_j
//          - S_tot * (sum over the token's choices c_i = m of w_i)   renormalised
//          - S_tot * p_m                                              otherwise,
// S_tot = the routed slots' sum of s, w_i the choices' normalised weights (a
// moved slot's weight is the new expert's p over the same normaliser), plus
// the auxiliary-loss and z-loss terms.  choice / choice_w: the token's kc
// choices at stride ld; the first kr of the K slots are routed (shared
// experts follow).  The row dg[t] first collects the slot scores by final
// expert (lane 0, slot order), then each lane finishes its columns.
// Where the slot scores come from: y_perm rows (w o in fp32; the kernel also
// writes the dY_perm rows), or, when spart is set, the dH product's partial
// dots (Params::spart of the GEMM kernels): with dH = W2_e^T (w_j dy_t),
//   s_j = <dy_t, w_j (W2_e h + b2_e)> = <dH_j, h_j> + w_j <dy_t, b2_e>,
// the first term the sum of the nparts partials of the slot's row (lane
// by lane, then across the warp in a fixed order), e the slot's expert (its
// segment in offsets); dY_perm is then already written.
template <typename T>
struct ScoreSrc {
    const float* y_perm;     // [rows][d] or null
    const float* spart;      // [rows_cap][nparts] or null
    int nparts;
    const T* b2;             // [E][d]
    const int32_t* offsets;  // [E + 1]
    int E;
};

template <typename T>
__global__ void __launch_bounds__(256) router_grad_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ choice,
    const float* __restrict__ choice_w, int ld, int kc, const int32_t* __restrict__ slot_of,
    const float* __restrict__ perm_w, const int32_t* __restrict__ kept_rank,
    const int32_t* __restrict__ alt, int mode, const ScoreSrc<T> src,
    const T* __restrict__ dy, const int32_t* __restrict__ top1, int Tn, int El, int K, int kr,
    int d, int64_t rows_cap, int renormalize, float aux_grad, float z_grad,
    float* __restrict__ dg, T* __restrict__ dY_perm) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x % 32;
    const int nwarps = gridDim.x * (blockDim.x / 32);
    const int nv = d / 8;  // 8-column groups
    for (int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; t < Tn; t += nwarps) {
        const T* dyr = dy + (size_t)t * d;
        float* dgt = dg + (size_t)t * El;
        for (int e = lane; e < El; e += 32) dgt[e] = 0.f;
        __syncwarp();
        float stot = 0.f;
        for (int j = 0; j < K; ++j) {
            const int slot = __ldg(slot_of + (size_t)t * K + j);
            if (slot < 0 || slot >= rows_cap) continue;  // dropped: s = 0
            const float w = __ldg(perm_w + slot);
            float dot = 0.f;
            if (src.spart == nullptr) {
                const float4* yr = reinterpret_cast<const float4*>(src.y_perm + (size_t)slot * d);
                T* dyp = dY_perm + (size_t)slot * d;
                for (int v = lane; v < nv; v += 32) {
                    float f[8];
                    load8(dyr + 8 * v, f);
                    const float4 a = __ldg(yr + 2 * v), b = __ldg(yr + 2 * v + 1);
                    dot += f[0] * a.x + f[1] * a.y + f[2] * a.z + f[3] * a.w + f[4] * b.x +
                           f[5] * b.y + f[6] * b.z + f[7] * b.w;
#pragma unroll
                    for (int q = 0; q < 8; ++q) f[q] *= w;
                    store8(dyp + 8 * v, f);
                }
            } else {
                if (j >= kr) continue;  // a shared expert: no logit, nothing to score
                int lo = 0, hi = src.E - 1;
                while (lo < hi) {  // the slot's expert: last segment starting at or before it
                    const int mid = (lo + hi + 1) >> 1;
                    if (__ldg(src.offsets + mid) <= slot) lo = mid; else hi = mid - 1;
                }
                const T* b2e = src.b2 + (size_t)lo * d;
                for (int v = lane; v < nv; v += 32) {
                    float f[8], b[8];
                    load8(dyr + 8 * v, f);
                    load8(b2e + 8 * v, b);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dot = fmaf(f[q], b[q], dot);
                }
                dot *= w;
                const float* sp = src.spart + (size_t)slot * src.nparts;
                for (int g = lane; g < src.nparts; g += 32) dot += __ldg(sp + g);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            if (j >= kr) continue;  // a shared expert: no logit
            stot += dot;
            int f = j;  // kGradExpert: slot j is expert j
            if (mode != kGradExpert) {
                f = __ldg(choice + (size_t)t * ld + j);
                if (mode == kGradReroute && __ldg(kept_rank + (size_t)t * kr + j) < 0)
                    f = __ldg(alt + (size_t)t * kr + j);
            }
            if (lane == 0 && f >= 0 && f < El) dgt[f] += dot;
        }
        __syncwarp();
        // softmax statistics of the token's logits
        const float* g = logits + (size_t)t * El;
        float m = -3.402823466e38f;
        for (int e = lane; e < El; e += 32) m = fmaxf(m, __ldg(g + e));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float ssum = 0.f, fp = 0.f;
        for (int e = lane; e < El; e += 32) {
            const float ex = expf(__ldg(g + e) - m);
            ssum += ex;
            if (top1 != nullptr) fp += ex * (float)__ldg(top1 + e);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
            fp += __shfl_xor_sync(0xffffffffu, fp, o);
        }
        const float inv = 1.0f / ssum;
        const float lse = m + logf(ssum);
        fp *= inv / (float)Tn;  // sum_i f_i p_i
        for (int e = lane; e < El; e += 32) {
            const float pe = expf(__ldg(g + e) - m) * inv;
            float v = dgt[e];
            if (renormalize) {
                for (int i = 0; i < kc; ++i)
                    if (__ldg(choice + (size_t)t * ld + i) == e)
                        v -= stot * __ldg(choice_w + (size_t)t * ld + i);
            } else {
                v -= pe * stot;
            }
            if (top1 != nullptr) {
                const float fe = (float)__ldg(top1 + e) / (float)Tn;
                v += aux_grad * (float)El / (float)Tn * pe * (fe - fp);
            }
            v += z_grad * 2.0f / (float)Tn * lse * pe;
            dgt[e] = v;
        }
    }
}

// dY_perm[slot] = w_slot dy_t for every kept slot of every token; a warp per
// token (the rows the dH product reads before the slot scores exist).
template <typename T>
__global__ void __launch_bounds__(256) scaled_rows_kernel(const int32_t* __restrict__ slot_of,
                                                           const float* __restrict__ perm_w,
                                                           const T* __restrict__ dy, int Tn,
                                                           int K, int d, int64_t rows_cap,
                                                           T* __restrict__ dY_perm) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x % 32;
    const int nwarps = gridDim.x * (blockDim.x / 32);
    const int nv = d / 8;
    for (int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; t < Tn; t += nwarps) {
        const T* dyr = dy + (size_t)t * d;
        for (int j = 0; j < K; ++j) {
            const int slot = __ldg(slot_of + (size_t)t * K + j);
            if (slot < 0 || slot >= rows_cap) continue;
            const float w = __ldg(perm_w + slot);
            T* dyp = dY_perm + (size_t)slot * d;
            for (int v = lane; v < nv; v += 32) {
                float f[8];
                load8(dyr + 8 * v, f);
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] *= w;
                store8(dyp + 8 * v, f);
            }
        }
    }
}

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(bf16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// dx[t] = sum over the token's slots of dX_perm rows + sum_e dg[t][e] W_r[e];
// one warp per (token, 512-column chunk).
template <typename TX>
__global__ void __launch_bounds__(256) dx_kernel(const float* __restrict__ dX_perm,
                                                  const int32_t* __restrict__ slot_of,
                                                  const float* __restrict__ dg,
                                                  const float* __restrict__ W_r, int T, int K,
                                                  int El, int d, int64_t rows_cap,
                                                  TX* __restrict__ dx) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x % 32;
    const int nwarps = gridDim.x * (blockDim.x / 32);
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
        for (int j = 0; j < K; ++j) {
            const int sl = __ldg(slot_of + (size_t)t * K + j);
            if (sl < 0 || sl >= rows_cap) continue;
            const float4* row = reinterpret_cast<const float4*>(dX_perm + (size_t)sl * d);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + 32 * u < nv) {
                    const float4 q = __ldg(row + v0 + 32 * u);
                    acc[u].x += q.x; acc[u].y += q.y; acc[u].z += q.z; acc[u].w += q.w;
                }
            }
        }
        for (int e = 0; e < El; ++e) {
            const float ge = __ldg(dg + (size_t)t * El + e);
            const float4* wr = reinterpret_cast<const float4*>(W_r + (size_t)e * d);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + 32 * u < nv) {
                    const float4 q = __ldg(wr + v0 + 32 * u);
                    acc[u].x = fmaf(ge, q.x, acc[u].x); acc[u].y = fmaf(ge, q.y, acc[u].y);
                    acc[u].z = fmaf(ge, q.z, acc[u].z); acc[u].w = fmaf(ge, q.w, acc[u].w);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v0 + 32 * u < nv) store4(dx + (size_t)t * d + 4 * (v0 + 32 * u), acc[u]);
    }
}

// dx for bf16 layers with many routed experts, where the dg W_r term (T x El
// by El x d) dominates: that product on the tensor cores as tf32 mma.sync
// m16n8k8 (dg and W_r rounded to tf32, fp32 accumulation; dx is rounded to
// bf16 after), a block per 64 tokens x 128 columns, each of its 4 warps 16
// tokens; W_r's 128 columns of every expert and the tokens' dg rows staged
// in shared memory (rows padded so the fragment reads hit distinct banks);
// then each lane adds its tokens' slots' dX_perm values and stores dx.
// Fragments (PTX m16n8k8 .tf32): A a0 (g, q), a1 (g + 8, q), a2 (g, q + 4),
// a3 (g + 8, q + 4); B b0 (k = q, n = g), b1 (q + 4, g); D (g, 2q), (g, 2q + 1),
// (g + 8, 2q), (g + 8, 2q + 1), with g = lane / 4, q = lane % 4.
constexpr int kDxTok = 64, kDxCols = 128, kDxMaxE = 64;
constexpr int kDxWld = kDxCols + 8, kDxGld = kDxMaxE + 4;  // shared row lengths (floats)
constexpr int kDxSmem = (kDxMaxE * kDxWld + kDxTok * kDxGld) * 4;

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__global__ void __launch_bounds__(128) dx_tc_kernel(const float* __restrict__ dX_perm,
                                                     const int32_t* __restrict__ slot_of,
                                                     const float* __restrict__ dg,
                                                     const float* __restrict__ W_r, int T, int K,
                                                     int El, int d, int64_t rows_cap,
                                                     bf16* __restrict__ dx) {
    extern __shared__ __align__(16) float dx_smem[];
    float* sW = dx_smem;                    // [kDxMaxE][kDxWld]
    float* sG = dx_smem + kDxMaxE * kDxWld;  // [kDxTok][kDxGld]
    pdl_wait();
    pdl_trigger();
    const int t0 = blockIdx.x * kDxTok, c0 = blockIdx.y * kDxCols;
    const int Ep = (El + 7) & ~7;  // K rounded up to the MMA's 8 (zeros past El)
    for (int i = threadIdx.x; i < Ep * (kDxCols / 4); i += blockDim.x) {
        const int e = i / (kDxCols / 4), c4 = (i % (kDxCols / 4)) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < El && c0 + c4 < d) v = __ldg(reinterpret_cast<const float4*>(W_r + (size_t)e * d + c0 + c4));
        *reinterpret_cast<float4*>(sW + e * kDxWld + c4) = v;
    }
    for (int i = threadIdx.x; i < kDxTok * Ep; i += blockDim.x) {
        const int r = i / Ep, e = i % Ep;
        sG[r * kDxGld + e] = t0 + r < T && e < El ? __ldg(dg + (size_t)(t0 + r) * El + e) : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, g = lane >> 2, q = lane & 3;
    const int m0 = warp * 16;
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    for (int k0 = 0; k0 < Ep; k0 += 8) {
        const uint32_t a0 = to_tf32(sG[(m0 + g) * kDxGld + k0 + q]);
        const uint32_t a1 = to_tf32(sG[(m0 + g + 8) * kDxGld + k0 + q]);
        const uint32_t a2 = to_tf32(sG[(m0 + g) * kDxGld + k0 + q + 4]);
        const uint32_t a3 = to_tf32(sG[(m0 + g + 8) * kDxGld + k0 + q + 4]);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const uint32_t b0 = to_tf32(sW[(k0 + q) * kDxWld + nt * 8 + g]);
            const uint32_t b1 = to_tf32(sW[(k0 + q + 4) * kDxWld + nt * 8 + g]);
            asm volatile(
                "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // token rows g and g + 8 of the warp's 16
        const int t = t0 + m0 + g + 8 * h;
        if (t >= T) continue;
        float2 v[16];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) v[nt] = make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
        for (int j = 0; j < K; ++j) {
            const int sl = __ldg(slot_of + (size_t)t * K + j);
            if (sl < 0 || sl >= rows_cap) continue;
            const float* row = dX_perm + (size_t)sl * d + c0 + 2 * q;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                if (c0 + nt * 8 + 2 * q < d) {
                    const float2 r2 = __ldg(reinterpret_cast<const float2*>(row + nt * 8));
                    v[nt].x += r2.x;
                    v[nt].y += r2.y;
                }
        }
        bf16* out = dx + (size_t)t * d + c0 + 2 * q;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
            if (c0 + nt * 8 + 2 * q < d)
                *reinterpret_cast<__nv_bfloat162*>(out + nt * 8) = __floats2bfloat162_rn(v[nt].x, v[nt].y);
    }
}

// Partial router-weight gradients: part[z][e][j] = sum over the tokens t of
// row slice z of dg[t][e] x[t][j].  A thread per column j (256 a block),
// EG experts per pass with their accumulators in registers, 64-token chunks
// of dg staged in shared memory.
constexpr int WR_CHUNK = 64;

template <int WR_EG, typename TX>
__global__ void __launch_bounds__(256) wr_grad_kernel(const float* __restrict__ dg,
                                                       const TX* __restrict__ x, int T, int E,
                                                       int d, int slice, float* __restrict__ part) {
    __shared__ float sg[WR_CHUNK][WR_EG];
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    const int z = blockIdx.y;
    const int t0 = min(z * slice, T), t1 = min(t0 + slice, T);
    for (int e0 = 0; e0 < E; e0 += WR_EG) {
        float acc[WR_EG];
#pragma unroll
        for (int c = 0; c < WR_EG; ++c) acc[c] = 0.f;
        for (int tb = t0; tb < t1; tb += WR_CHUNK) {
            __syncthreads();
            for (int i = threadIdx.x; i < WR_CHUNK * WR_EG; i += blockDim.x) {
                const int r = i / WR_EG, c = i % WR_EG;
                sg[r][c] = (tb + r < t1 && e0 + c < E) ? __ldg(dg + (size_t)(tb + r) * E + e0 + c)
                                                       : 0.f;
            }
            __syncthreads();
            if (j < d) {
                const int rows = min(WR_CHUNK, t1 - tb);
#pragma unroll 4
                for (int r = 0; r < rows; ++r) {
                    const float xv = to_f32(x[(size_t)(tb + r) * d + j]);
#pragma unroll
                    for (int c = 0; c < WR_EG; ++c) acc[c] = fmaf(sg[r][c], xv, acc[c]);
                }
            }
        }
        if (j < d)
            for (int c = 0; c < WR_EG && e0 + c < E; ++c)
                part[((size_t)z * E + e0 + c) * d + j] = acc[c];
    }
}

// Partial router-weight gradients for bf16 layers with 16-64 routed experts
// on the tensor cores: part[z][e][j] = sum over the tokens t of slice z
// (kWrSlice tokens) of dg[t][e] x[t][j] as tf32 mma.sync m16n8k8 (M = the
// experts, 16 a warp; N = 128 columns a block; K = the slice's tokens in
// chunks of 32 staged in shared memory; dg rounded to tf32, x exact, fp32
// accumulation).  sum_parts_kernel then adds the slices in order.
constexpr int kWrCols = 128, kWrChunk = 32, kWrSlice = 1024;
constexpr int kWrGld = kDxMaxE + 8, kWrXld = kWrCols + 8;  // shared row lengths (floats)

__global__ void __launch_bounds__(128) wr_tc_kernel(const float* __restrict__ dg,
                                                     const bf16* __restrict__ x, int T, int El,
                                                     int d, float* __restrict__ part) {
    __shared__ __align__(16) float sG[kWrChunk][kWrGld];
    __shared__ __align__(16) float sX[kWrChunk][kWrXld];
    pdl_wait();
    pdl_trigger();
    const int z = blockIdx.x, c0 = blockIdx.y * kWrCols;
    const int tb = z * kWrSlice, te = min(T, tb + kWrSlice);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, g = lane >> 2, q = lane & 3;
    const int m0 = warp * 16;  // this warp's 16 experts
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    for (int tc = tb; tc < te; tc += kWrChunk) {
        __syncthreads();  // the previous chunk's fragments are read
        for (int i = threadIdx.x; i < kWrChunk * kDxMaxE; i += blockDim.x) {
            const int r = i / kDxMaxE, e = i % kDxMaxE;
            sG[r][e] = tc + r < te && e < El ? __ldg(dg + (size_t)(tc + r) * El + e) : 0.f;
        }
        for (int i = threadIdx.x; i < kWrChunk * (kWrCols / 8); i += blockDim.x) {
            const int r = i / (kWrCols / 8), c8 = (i % (kWrCols / 8)) * 8;
            float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (tc + r < te && c0 + c8 < d) load8(x + (size_t)(tc + r) * d + c0 + c8, f);
#pragma unroll
            for (int u = 0; u < 8; ++u) sX[r][c8 + u] = f[u];
        }
        __syncthreads();
        if (m0 < El) {
#pragma unroll
            for (int k0 = 0; k0 < kWrChunk; k0 += 8) {
                const uint32_t a0 = to_tf32(sG[k0 + q][m0 + g]);
                const uint32_t a1 = to_tf32(sG[k0 + q][m0 + g + 8]);
                const uint32_t a2 = to_tf32(sG[k0 + q + 4][m0 + g]);
                const uint32_t a3 = to_tf32(sG[k0 + q + 4][m0 + g + 8]);
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const uint32_t b0 = __float_as_uint(sX[k0 + q][nt * 8 + g]);  // bf16: exact in tf32
                    const uint32_t b1 = __float_as_uint(sX[k0 + q + 4][nt * 8 + g]);
                    asm volatile(
                        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
                        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                        : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                }
            }
        }
    }
    if (m0 >= El) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = m0 + g + 8 * h;
        if (e >= El) continue;
        float* out = part + ((size_t)z * El + e) * d + c0 + 2 * q;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
            if (c0 + nt * 8 + 2 * q < d)
                *reinterpret_cast<float2*>(out + nt * 8) =
                    make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
    }
}

// out[e][m] = sum over the rows of segment e of A[r][m].  A cluster of
// kColSlices CTAs per (256 columns, expert): CTA z, warp w sums the rows
// i = 8z + w (mod 64) of the segment, eight columns a lane (16- or 32-byte
// loads, four rows in flight); each CTA adds its warps' sums in warp order,
// then CTA 0 adds the CTAs' sums in rank order from their shared memory, so
// the result does not depend on timing.
constexpr int kColSlices = 8;

template <typename T>
__global__ void __launch_bounds__(256) colsum_kernel(const T* __restrict__ A,
                                                      const int32_t* __restrict__ offsets,
                                                      int64_t rows_cap, int M,
                                                      float* __restrict__ out) {
    __shared__ float part[8][256];
    __shared__ float blk[256];
    pdl_wait();
    pdl_trigger();
    const int z = (int)tc::cluster_ctarank(), e = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int m = blockIdx.y * 256 + 8 * lane;
    const int r1 = (int)min((int64_t)max(__ldg(offsets + e + 1), 0), rows_cap);
    const int r0 = min(max(__ldg(offsets + e), 0), r1);
    const int n = r1 - r0;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (m < M) {  // M is a multiple of 8: a lane's eight columns are all in or all out
        const T* col = A + (size_t)r0 * M + m;
        int i = z * 8 + warp;
        for (; i + 192 < n; i += 256) {  // four rows 64 apart in flight
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) load8(col + (size_t)(i + 64 * u) * M, v[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += v[u][j];
        }
        for (; i < n; i += 64) {
            float v[8];
            load8(col + (size_t)i * M, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += v[j];
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) part[warp][8 * lane + j] = acc[j];
    __syncthreads();
    {
        const int t = threadIdx.x;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += part[w][t];
        blk[t] = v;
    }
    tc::cluster_sync();  // every CTA's sums are in its shared memory
    if (z == 0) {
        const int t = threadIdx.x, mc = blockIdx.y * 256 + t;
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < kColSlices; ++r) v += tc::ld_shared_cluster_f32(tc::cluster_addr(&blk[t], r));
        if (mc < M) out[(size_t)e * M + mc] = v;
    }
    tc::cluster_sync();  // no CTA leaves while CTA 0 reads its shared memory
}

// colsum_kernel's launch: grid (kColSlices, 256-column chunks, E), clusters
// of kColSlices along x.
template <typename T>
cudaError_t launch_colsum(const T* A, const int32_t* offsets, int64_t rows_cap, int E, int M,
                          float* out, cudaStream_t s) {
    return launch_kernel(colsum_kernel<T>, dim3(kColSlices, (M + 255) / 256, E), dim3(256), 0, s,
                         kColSlices, false, A, offsets, rows_cap, M, out);
}

// out[i] = sum over z < S of part[z][i], in z order.
__global__ void __launch_bounds__(256) sum_parts_kernel(const float* __restrict__ part, int S,
                                                         int64_t n, float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
#pragma unroll 8
        for (int z = 0; z < S; ++z) v += __ldg(part + (size_t)z * n + i);  // loads ahead, adds in z order
        out[i] = v;
    }
}

int grid_for(int64_t work, int per_block) {
    int64_t b = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

// Backward workspace: the forward layout, then these regions.
struct BwdLayout {
    size_t logits, u, dyp, dh, dg, maps, spart, parts, total;
    int nparts;        // 16-column partial dots per row (bf16 layers)
    int wr_slices;     // row slices of the router-weight gradient
};

// Row slices of dW_r = dg^T x (partial sums, then a fixed-order sum): 64
// rows, or T / 256 for the largest batches (at most 256 slices).
int wr_slice_rows(int T) {
    const int s = (T + 255) / 256;
    return s > 64 ? s : 64;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

BwdLayout bwd_layout(const moe_config& c, const WsLayout& L) {
    BwdLayout B{};
    size_t o = align256(L.total);
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const size_t rows = (size_t)L.rows;
    const bool f32 = c.dtype == MOE_F32;  // fp32: no tensor maps, no slot-score partials
    const size_t es = f32 ? 4 : 2;         // bytes of a token-row element
    B.logits = take(sizeof(float) * (size_t)c.T * c.E);
    B.u = take(es * rows * c.d_ff);
    B.dyp = take(es * rows * c.d);
    B.dh = take(es * rows * c.d_ff);
    B.dg = take(sizeof(float) * (size_t)c.T * c.E);
    // per-segment tensor maps of the two weight-gradient reductions (2E each)
    B.maps = take(f32 ? 0 : 4 * kSegMapBytes * (size_t)c.E);
    // the dH product's partial dots per 16 columns (the slot scores)
    B.nparts = (c.d_ff + 15) / 16;
    B.spart = take(f32 ? 0 : sizeof(float) * (size_t)B.nparts * rows);
    const int chunk = wr_slice_rows(c.T);
    B.wr_slices = (c.T + chunk - 1) / chunk;
    B.parts = take(sizeof(float) * (size_t)B.wr_slices * c.E * c.d);
    B.total = o;
    return B;
}

bool backward_supported(const moe_config& c) {
    return c.dtype == MOE_BF16 || c.dtype == MOE_F32;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_check_segment_maps(void* ws, size_t ws_bytes, void* stream) {
    return check_segment_maps(ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_backward_workspace_size(const moe_config* cfg) {
    if (config_status(cfg) != MOE_OK || !backward_supported(*cfg)) return 0;
    const WsLayout L = ws_layout(*cfg);
    return bwd_layout(*cfg, L).total;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_r,
                        const float* logit_bias, const void* W1, const void* b1, const void* W2,
                        const void* b2, const void* dy, float aux_grad, float z_grad, void* dx,
                        float* dW_r, float* dW1, float* db1, float* dW2, float* db2, void* ws,
                        size_t ws_bytes, void* stream) {
    moe_status st = config_status(cfg);
    if (st != MOE_OK) return st;
    const moe_config& c = *cfg;
    if (!backward_supported(c)) return MOE_ERR_UNSUPPORTED;
    if (dW_r == nullptr || dW1 == nullptr || db1 == nullptr || dW2 == nullptr || db2 == nullptr)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int E = c.E, d = c.d, F = c.d_ff, T = c.T, k = c.k;
    // (an empty batch reads no token array: x, dy and dx may be null then)
    if (T > 0 && (x == nullptr || W_r == nullptr || W1 == nullptr || b1 == nullptr ||
                  W2 == nullptr || b2 == nullptr || dy == nullptr || dx == nullptr))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(W_r) ||
                  !aligned16(W1) || !aligned16(W2)))
        return MOE_ERR_ALIGNMENT;
    const WsLayout L = ws_layout(c);
    const BwdLayout Bw = bwd_layout(c, L);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < Bw.total)
        return MOE_ERR_WORKSPACE;
    const bool ec = c.routing == MOE_EXPERT_CHOICE;
    const bool rr = c.overflow == MOE_REROUTE && c.capacity >= 0;  // (no cap: nothing moves)
    const int El = E - c.n_shared;                                 // logit columns
    if (T == 0) {  // no token: every gradient is zero
        const size_t wsz = sizeof(float) * (size_t)E * d * F;
        if (cudaMemsetAsync(dW_r, 0, sizeof(float) * (size_t)El * d, s) != cudaSuccess ||
            cudaMemsetAsync(dW1, 0, wsz, s) != cudaSuccess ||
            cudaMemsetAsync(dW2, 0, wsz, s) != cudaSuccess ||
            cudaMemsetAsync(db1, 0, sizeof(float) * (size_t)E * F, s) != cudaSuccess ||
            cudaMemsetAsync(db2, 0, sizeof(float) * (size_t)E * d, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    DeviceHeader* hdr = at<DeviceHeader>(ws, L.header);
    int32_t* idx = at<int32_t>(ws, L.topk_idx);
    float* w = at<float>(ws, L.topk_w);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* slot_of = at<int32_t>(ws, L.slot_of);
    int32_t* perm_token = at<int32_t>(ws, L.perm_token);
    float* perm_w = at<float>(ws, L.perm_w);
    bf16* x_perm = at<bf16>(ws, L.x_perm);
    bf16* H = at<bf16>(ws, L.h);
    float* y_perm = at<float>(ws, L.y_perm);  // w * o, then dX_perm
    float* logits = at<float>(ws, Bw.logits);
    bf16* U = at<bf16>(ws, Bw.u);
    bf16* dYp = at<bf16>(ws, Bw.dyp);
    bf16* dH = at<bf16>(ws, Bw.dh);
    float* dg = at<float>(ws, Bw.dg);
    const int64_t rows = L.rows;

    // slots per token and the token's choices (the routed experts' normaliser)
    const int K = ec ? E : k + c.n_shared;
    const int kr = ec ? E : k;  // routed slots
    const int32_t* choice = idx;
    const float* choice_w = w;
    int ld = k;
    chain_begin();
    // ---- recompute the forward intermediates (the forward pass's routing and dispatch)
    cudaError_t e;
    if (ec) {
        float* probs_t = at<float>(ws, L.probs_t);
        e = launch_route(ec_router_config(c), x, W_r, logit_bias, nullptr, nullptr, logits, idx, w,
                         nullptr, nullptr, nullptr, ws, L, false, s, probs_t);
        if (e == cudaSuccess)
            e = launch_ec_select(c, probs_t, offsets, perm_token, perm_w, slot_of, nullptr, s);
        if (e == cudaSuccess) e = launch_ec_gather(c, x, perm_token, x_perm, s);
    } else if (rr) {
        ld = reroute_ranked(c);
        e = launch_route(reroute_router_config(c), x, W_r, logit_bias, nullptr, nullptr, logits,
                         idx, w, nullptr, nullptr, nullptr, ws, L, false, s, nullptr, k);
        if (e == cudaSuccess)
            e = launch_reroute_dispatch(c, ld, x, idx, w, offsets, slot_of, perm_token, perm_w,
                                        x_perm, ws, L, LossArgs{}, s);
    } else if (c.n_shared > 0) {
        int32_t* idx_r = at<int32_t>(ws, L.route_idx);
        float* w_r = at<float>(ws, L.route_w);
        choice = idx_r;
        choice_w = w_r;
        const moe_config cd = dispatch_config(c);
        e = launch_route(routed_config(c), x, W_r, logit_bias, nullptr, nullptr, logits, idx_r,
                         w_r, nullptr, nullptr, nullptr, ws, L, false, s);
        if (e == cudaSuccess)
            e = launch_join_shared(c, idx_r, w_r, idx, w, at<int32_t>(ws, L.counts), nullptr, s);
        if (e == cudaSuccess) e = launch_count(cd, idx, ws, L, s);
        if (e == cudaSuccess)
            e = launch_scan_permute(cd, x, idx, w, kCountBlock, L.count_blocks, offsets, slot_of,
                                    perm_token, perm_w, x_perm, ws, L, LossArgs{}, s);
    } else {
        e = launch_route(c, x, W_r, logit_bias, nullptr, nullptr, logits, idx, w, nullptr,
                         nullptr, nullptr, ws, L, true, s);
        if (e == cudaSuccess)
            e = launch_scan_permute(c, x, idx, w, L.route.tokens * k, L.route.blocks, offsets,
                                    slot_of, perm_token, perm_w, x_perm, ws, L,
                                    route_loss_args(c, ws, L, nullptr, nullptr, nullptr), s);
    }
    const int grad_mode = ec ? (int)kGradExpert : rr ? (int)kGradReroute : (int)kGradChoice;
    const int32_t* kept_rank = rr ? at<int32_t>(ws, L.rr_kept) : nullptr;
    const int32_t* alt = rr ? at<int32_t>(ws, L.rr_alt) : nullptr;
    const int32_t* top1 = ec ? nullptr : at<int32_t>(ws, L.top1);
    if (c.dtype == MOE_F32) {
        // fp32 layers: every product on CUDA cores in fp32 (backward_f32.cu)
        float* Uf = at<float>(ws, Bw.u);     // pre-activations, then (in dH) dU
        float* Hf = at<float>(ws, L.h);      // GELU(U)
        float* dYf = at<float>(ws, Bw.dyp);  // w dy per row
        float* dHf = at<float>(ws, Bw.dh);
        const float* xp = at<float>(ws, L.x_perm);
        const int64_t max_seg = ec ? rows / E : (rows < T ? rows : (int64_t)T);
        const float* W1f = reinterpret_cast<const float*>(W1);
        const float* W2f = reinterpret_cast<const float*>(W2);
        if (e == cudaSuccess)
            e = launch_seg_gemm_f32(false, 1, xp, offsets, E, W1f,
                                    reinterpret_cast<const float*>(b1), nullptr, Uf, Hf, F, d,
                                    max_seg, rows, s);
        if (e == cudaSuccess)
            e = launch_seg_gemm_f32(false, 2, Hf, offsets, E, W2f,
                                    reinterpret_cast<const float*>(b2), perm_w, y_perm, nullptr,
                                    d, F, max_seg, rows, s);
        if (e == cudaSuccess)
            e = launch_kernel(router_grad_kernel<float>, dim3(grid_for(T, 8)), dim3(256), 0, s, 1,
                              false, (const float*)logits, choice, choice_w, ld, ec ? 0 : k,
                              (const int32_t*)slot_of, (const float*)perm_w, kept_rank, alt,
                              grad_mode,
                              ScoreSrc<float>{(const float*)y_perm, nullptr, 0, nullptr, nullptr, E},
                              reinterpret_cast<const float*>(dy), top1, T, El, K, kr, d, rows,
                              ec ? 0 : c.renormalize, aux_grad, z_grad, dg, dYf);
        if (e == cudaSuccess) e = launch_seg_atb_f32(dYf, Hf, offsets, E, d, F, rows, dW2, s);
        if (e == cudaSuccess)
            e = launch_colsum((const float*)dYf, (const int32_t*)offsets, rows, E, d, db2, s);
        if (e == cudaSuccess)  // dH = dY W2_e (W2_e: [d][d_ff] = [K][N])
            e = launch_seg_gemm_f32(true, 0, dYf, offsets, E, W2f, nullptr, nullptr, dHf, nullptr,
                                    F, d, max_seg, rows, s);
        if (e == cudaSuccess) e = launch_gelu_grad_f32(Uf, dHf, offsets, E, F, rows, s);
        if (e == cudaSuccess) e = launch_seg_atb_f32(dHf, xp, offsets, E, F, d, rows, dW1, s);
        if (e == cudaSuccess)
            e = launch_colsum((const float*)dHf, (const int32_t*)offsets, rows, E, F, db1, s);
        if (e == cudaSuccess)  // dX_perm = dU W1_e (W1_e: [d_ff][d] = [K][N]), over y_perm
            e = launch_seg_gemm_f32(true, 0, dHf, offsets, E, W1f, nullptr, nullptr, y_perm,
                                    nullptr, d, F, max_seg, rows, s);
        if (e == cudaSuccess) {
            const long long tasks = (long long)T * ((d / 4 + 127) / 128);
            e = launch_kernel(dx_kernel<float>, dim3(grid_for(tasks, 8)), dim3(256), 0, s, 1,
                              false, (const float*)y_perm, (const int32_t*)slot_of,
                              (const float*)dg, W_r, T, K, El, d, rows, reinterpret_cast<float*>(dx));
        }
        if (e == cudaSuccess)
            e = launch_kernel(El <= 8 ? wr_grad_kernel<8, float> : wr_grad_kernel<32, float>,
                              dim3((d + 255) / 256, Bw.wr_slices), dim3(256), 0, s, 1, false,
                              (const float*)dg, reinterpret_cast<const float*>(x), T, El, d,
                              wr_slice_rows(T), at<float>(ws, Bw.parts));
        if (e == cudaSuccess)
            e = launch_kernel(sum_parts_kernel, dim3(grid_for((int64_t)El * d, 256)), dim3(256), 0,
                              s, 1, false, (const float*)at<float>(ws, Bw.parts), Bw.wr_slices,
                              (int64_t)El * d, dW_r);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    const moe_config cg = dispatch_config(c);  // the GEMMs as the forward pass runs them
    CUtensorMap* maps = at<CUtensorMap>(ws, Bw.maps);
    float* spart = at<float>(ws, Bw.spart);
    if (e == cudaSuccess)  // H = GELU(x_perm W1^T + b1), and the pre-activation U
        e = launch_grouped_gemm_tc(cg, true, true, x_perm, rows, offsets, W1, b1, nullptr, H, rows,
                                   F, d, hdr, s, U);
    // ---- the scaled upstream rows dY_perm = w dy_t
    if (e == cudaSuccess)
        e = launch_kernel(scaled_rows_kernel<bf16>, dim3(grid_for(T, 8)), dim3(256), 0, s, 1,
                          false, (const int32_t*)slot_of, (const float*)perm_w,
                          reinterpret_cast<const bf16*>(dy), T, K, d, rows, dYp);
    // ---- dU = (dY_perm W2_e) GELU'(U) (in dH's buffer), with the rows' partial
    // dots <dH, GELU(U)> that make the slot scores (no second-GEMM recompute)
    if (e == cudaSuccess)
        e = launch_grouped_gemm_mn(cg, true, dYp, rows, offsets, W2, U, spart, dH, rows, F, d, hdr,
                                   s);
    // ---- router gradient
    if (e == cudaSuccess)
        e = launch_kernel(router_grad_kernel<bf16>, dim3(grid_for(T, 8)), dim3(256), 0, s, 1, false,
                          (const float*)logits, choice, choice_w, ld, ec ? 0 : k,
                          (const int32_t*)slot_of, (const float*)perm_w, kept_rank, alt,
                          grad_mode,
                          ScoreSrc<bf16>{nullptr, spart, Bw.nparts,
                                         reinterpret_cast<const bf16*>(b2), offsets, E},
                          reinterpret_cast<const bf16*>(dy), top1, T, El, K, kr, d, rows,
                          ec ? 0 : c.renormalize, aux_grad, z_grad, dg, (bf16*)nullptr);
    // ---- dW2_e = dY_perm_e^T H_e, db2
    if (e == cudaSuccess)
        e = launch_segment_reduction_tc(E, offsets, rows, dYp, d, H, F, dW2, maps, hdr, s);
    if (e == cudaSuccess)
        e = launch_colsum((const bf16*)dYp, (const int32_t*)offsets, rows, E, d, db2, s);
    // ---- dX_perm = dU W1_e (over y_perm), dx
    if (e == cudaSuccess)
        e = launch_grouped_gemm_mn(cg, false, dH, rows, offsets, W1, nullptr, nullptr, y_perm, rows,
                                   d, F, hdr, s);
    if (e == cudaSuccess && El >= 16 && El <= kDxMaxE) {  // the dg W_r term dominates
        e = ensure_smem<dx_tc_kernel>(kDxSmem);
        if (e == cudaSuccess)
            e = launch_kernel(dx_tc_kernel, dim3((T + kDxTok - 1) / kDxTok, (d + kDxCols - 1) / kDxCols),
                              dim3(128), kDxSmem, s, 1, false, (const float*)y_perm,
                              (const int32_t*)slot_of, (const float*)dg, W_r, T, K, El, d, rows,
                              reinterpret_cast<bf16*>(dx));
    } else if (e == cudaSuccess) {
        const long long tasks = (long long)T * ((d / 4 + 127) / 128);
        e = launch_kernel(dx_kernel<bf16>, dim3(grid_for(tasks, 8)), dim3(256), 0, s, 1, false,
                          (const float*)y_perm, (const int32_t*)slot_of, (const float*)dg, W_r, T,
                          K, El, d, rows, reinterpret_cast<bf16*>(dx));
    }
    // ---- dW1_e = dU_e^T X_perm_e, db1
    if (e == cudaSuccess)
        e = launch_segment_reduction_tc(E, offsets, rows, dH, F, x_perm, d, dW1, maps + 2 * E, hdr,
                                        s);
    if (e == cudaSuccess)
        e = launch_colsum((const bf16*)dH, (const int32_t*)offsets, rows, E, F, db1, s);
    // ---- dW_r = dg^T x: row-slice partials, then their sum
    const bool wr_tc = El >= 16 && El <= kDxMaxE;
    const int wr_slices = wr_tc ? (T + kWrSlice - 1) / kWrSlice : Bw.wr_slices;
    if (e == cudaSuccess && wr_tc)
        e = launch_kernel(wr_tc_kernel, dim3(wr_slices, (d + kWrCols - 1) / kWrCols), dim3(128), 0,
                          s, 1, false, (const float*)dg, reinterpret_cast<const bf16*>(x), T, El,
                          d, at<float>(ws, Bw.parts));
    else if (e == cudaSuccess)
        e = launch_kernel(El <= 8 ? wr_grad_kernel<8, bf16> : wr_grad_kernel<32, bf16>,
                          dim3((d + 255) / 256, Bw.wr_slices), dim3(256), 0, s, 1, false,
                          (const float*)dg, reinterpret_cast<const bf16*>(x), T, El, d,
                          wr_slice_rows(T), at<float>(ws, Bw.parts));
    if (e == cudaSuccess)
        e = launch_kernel(sum_parts_kernel, dim3(grid_for((int64_t)El * d, 256)), dim3(256), 0, s,
                          1, false, (const float*)at<float>(ws, Bw.parts), wr_slices,
                          (int64_t)El * d, dW_r);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
