// Device helpers shared by the libmoe kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

// Programmatic dependent launch.  Inside one entry-point call every kernel
// after the first is launched with programmatic stream serialization (see
// launch_kernel), so the GPU may make its blocks resident while the previous
// kernel is still running.  Each kernel therefore calls pdl_wait() before its
// first access to global memory: it returns once the previous kernel has
// completed and its writes are visible.  pdl_trigger() then allows the next
// kernel to be scheduled.  Both are no-ops for a kernel launched without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Widen 8 consecutive stored elements (16 bytes of bf16, or 32 bytes of fp32)
// to fp32.  `p` is 16-byte aligned.
__device__ __forceinline__ void load8_f32(const __nv_bfloat16* p, float v[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8_f32(const float* p, float v[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Exact GELU in fp32: 0.5 u (1 + erf(u / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float u) {
    return 0.5f * u * (1.0f + erff(u * 0.70710678118654752440f));
}

// GELU 0.5 u (1 + erf(u / sqrt 2)) for two values at once, with packed fp32
// arithmetic (two lanes per instruction).  erf comes from the rational
// approximation of Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (Hastings): for z >= 0, erf(z) = 1 - q(t) exp(-z^2),
// t = 1 / (1 + p z), q(t) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))), with
// |error| <= 1.5e-7.  With z = |u| / sqrt 2 the GELU is u - 0.5 u q e^{-z^2}
// for u >= 0 and 0.5 u q e^{-z^2} for u < 0, i.e.
//   gelu(u) = max(u, 0) - 0.5 |u| q(t) e^{-z^2},
// which has no cancellation in the negative tail and needs no select.  With
// y = |u| sqrt(log2(e) / 2), e^{-z^2} is 2^{-y^2} and p z is
// (p / sqrt(log2 e)) y; the factor -0.5 |u| / y is folded into the
// coefficients.  Used where the result is rounded to bf16 (relative step
// 2^-8), far above the approximation error.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 gelu2_as7126(float2 u) {
    constexpr float c = 0.84932180028801904f;  // sqrt(log2(e) / 2)
    constexpr float pz = 0.27273748f;          // 0.3275911 / sqrt(log2 e)
    constexpr float k = -0.5f / c;             // -0.5 |u| = k y
    const float2 y = make_float2(fabsf(u.x) * c, fabsf(u.y) * c);
    const float2 den = __ffma2_rn(y, make_float2(pz, pz), make_float2(1.f, 1.f));
    const float2 t = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
    float2 q = __ffma2_rn(t, make_float2(k * 1.061405429f, k * 1.061405429f),
                          make_float2(k * -1.453152027f, k * -1.453152027f));
    q = __ffma2_rn(t, q, make_float2(k * 1.421413741f, k * 1.421413741f));
    q = __ffma2_rn(t, q, make_float2(k * -0.284496736f, k * -0.284496736f));
    q = __ffma2_rn(t, q, make_float2(k * 0.254829592f, k * 0.254829592f));
    q = __fmul2_rn(q, t);
    const float2 s = __fmul2_rn(y, y);
    const float2 e = make_float2(ex2_approx(-s.x), ex2_approx(-s.y));
    return __ffma2_rn(y, __fmul2_rn(q, e), make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)));
}

// d/du of the GELU u Phi(u): Phi(u) + u phi(u).  Phi from the erf
// approximation of Abramowitz & Stegun, formula 7.1.26 (|erf error| <=
// 1.5e-7, the form the forward GEMM's epilogue uses): with z = |u| / sqrt 2,
// erf(z) = 1 - q(t) e^{-z^2}, t = 1 / (1 + p z), so Phi(u) = 1 - h for
// u >= 0 and h for u < 0, h = 0.5 q(t) e^{-u^2/2}; phi(u) = e^{-u^2/2} /
// sqrt(2 pi) shares the exponential.  e^{-u^2/2} = 2^{-y^2} with
// y = |u| sqrt(log2(e) / 2), and p z = (p / sqrt(log2 e)) y.
__device__ __forceinline__ float gelu_grad(float u) {
    constexpr float c = 0.84932180028801904f;  // sqrt(log2(e) / 2)
    constexpr float pz = 0.27273748f;          // 0.3275911 / sqrt(log2 e)
    const float y = fabsf(u) * c;
    const float t = __fdividef(1.0f, fmaf(y, pz, 1.0f));
    float q = fmaf(t, 1.061405429f, -1.453152027f);
    q = fmaf(t, q, 1.421413741f);
    q = fmaf(t, q, -0.284496736f);
    q = fmaf(t, q, 0.254829592f);
    q *= t;
    const float e = ex2_approx(-y * y);
    const float h = 0.5f * q * e;
    return (u >= 0.f ? 1.0f - h : h) + u * e * 0.39894228040143268f;
}

// gelu_grad for two values at once with packed fp32 arithmetic (the same
// formula; for epilogues where the scalar form's instruction count shows).
__device__ __forceinline__ float2 gelu_grad2(float2 u) {
    constexpr float c = 0.84932180028801904f;  // sqrt(log2(e) / 2)
    constexpr float pz = 0.27273748f;          // 0.3275911 / sqrt(log2 e)
    const float2 y = make_float2(fabsf(u.x) * c, fabsf(u.y) * c);
    const float2 den = __ffma2_rn(y, make_float2(pz, pz), make_float2(1.f, 1.f));
    const float2 t = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
    float2 q = __ffma2_rn(t, make_float2(1.061405429f, 1.061405429f),
                          make_float2(-1.453152027f, -1.453152027f));
    q = __ffma2_rn(t, q, make_float2(1.421413741f, 1.421413741f));
    q = __ffma2_rn(t, q, make_float2(-0.284496736f, -0.284496736f));
    q = __ffma2_rn(t, q, make_float2(0.254829592f, 0.254829592f));
    q = __fmul2_rn(q, t);
    const float2 s = __fmul2_rn(y, y);
    const float2 e = make_float2(ex2_approx(-s.x), ex2_approx(-s.y));
    const float2 h = __fmul2_rn(__fmul2_rn(make_float2(0.5f, 0.5f), q), e);
    const float2 phi0 = make_float2(u.x >= 0.f ? 1.0f - h.x : h.x, u.y >= 0.f ? 1.0f - h.y : h.y);
    return __ffma2_rn(__fmul2_rn(u, e), make_float2(0.39894228040143268f, 0.39894228040143268f),
                      phi0);
}

// gelu_grad2 and the GELU itself from the same intermediate terms: with
// h = 0.5 q(t) e^{-u^2/2} as in gelu_grad, GELU(u) = u Phi(u) = max(u, 0) -
// |u| h.  Returns GELU'(u); *g receives GELU(u).
__device__ __forceinline__ float2 gelu_and_grad2(float2 u, float2* g) {
    constexpr float c = 0.84932180028801904f;  // sqrt(log2(e) / 2)
    constexpr float pz = 0.27273748f;          // 0.3275911 / sqrt(log2 e)
    const float2 au = make_float2(fabsf(u.x), fabsf(u.y));
    const float2 y = make_float2(au.x * c, au.y * c);
    const float2 den = __ffma2_rn(y, make_float2(pz, pz), make_float2(1.f, 1.f));
    const float2 t = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
    float2 q = __ffma2_rn(t, make_float2(1.061405429f, 1.061405429f),
                          make_float2(-1.453152027f, -1.453152027f));
    q = __ffma2_rn(t, q, make_float2(1.421413741f, 1.421413741f));
    q = __ffma2_rn(t, q, make_float2(-0.284496736f, -0.284496736f));
    q = __ffma2_rn(t, q, make_float2(0.254829592f, 0.254829592f));
    q = __fmul2_rn(q, t);
    const float2 s = __fmul2_rn(y, y);
    const float2 e = make_float2(ex2_approx(-s.x), ex2_approx(-s.y));
    const float2 h = __fmul2_rn(__fmul2_rn(make_float2(0.5f, 0.5f), q), e);
    *g = __ffma2_rn(make_float2(-au.x, -au.y), h,
                    make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)));
    const float2 phi0 = make_float2(u.x >= 0.f ? 1.0f - h.x : h.x, u.y >= 0.f ? 1.0f - h.y : h.y);
    return __ffma2_rn(__fmul2_rn(u, e), make_float2(0.39894228040143268f, 0.39894228040143268f),
                      phi0);
}

// Inputs of the auxiliary-loss reduction: per-block sums of p written by the
// router (blk_p, nblk rows of E) and the first-slot / all-slot counts.
struct LossArgs {
    const float* blk_p;
    const float* blk_z;      // per-block sums of the squared log-sum-exp
    const int32_t* top1;
    const int32_t* counts;
    int32_t* expert_counts;  // output or null
    float* aux_out;          // output or null
    float* z_out;            // router z-loss output or null
    int nblk, E, T;
};

// Switch auxiliary loss E * sum_e f_e P_e (f_e = top1_e / T, P_e = the mean
// probability, summed over the router blocks in block order) and the copy of
// the per-expert counts, by one block.  Only the first 256 threads take part,
// so the summation order is the same in every kernel that calls it.  fp32
// throughout (the sums of at most T probabilities keep ~1e-6 relative error).
// s_part: 256 floats, s_d: E floats of shared memory.
__device__ __forceinline__ void loss_and_counts(const LossArgs& l, float* s_part, float* s_d) {
    const int tid = threadIdx.x;
    const int per = 256 / l.E;  // threads per expert
    const int stride = per * l.E;
    if (tid < 256) {
        float v = 0.f;
        if (tid < stride) {
            const int e = tid % l.E;
            // blocks tid/E, tid/E + per, ... in order; eight loads in flight
            for (int b0 = tid / l.E; b0 < l.nblk; b0 += 8 * per) {
                float q[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int b = b0 + u * per;
                    q[u] = b < l.nblk ? __ldcg(l.blk_p + (size_t)b * l.E + e) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) v += q[u];
            }
        }
        s_part[tid] = v;
    }
    __syncthreads();
    for (int e = tid; e < l.E; e += blockDim.x) {
        float pe = 0.f;
        for (int j = 0; j < per; ++j) pe += s_part[j * l.E + e];
        s_d[e] = (float)__ldcg(l.top1 + e) * pe;
        if (l.expert_counts != nullptr) l.expert_counts[e] = __ldcg(l.counts + e);
    }
    __syncthreads();
    if (tid == 0 && l.aux_out != nullptr) {
        float s = 0.f;
        for (int e = 0; e < l.E; ++e) s += s_d[e];
        const float Tf = (float)l.T;
        l.aux_out[0] = (float)l.E * (s / Tf) / Tf;
    }
    if (l.z_out != nullptr) {  // router z-loss: block sums in 256 strided parts, then a fixed tree
        __syncthreads();
        if (tid < 256) {
            float v = 0.f;
            for (int b = tid; b < l.nblk; b += 256) v += __ldcg(l.blk_z + b);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if ((tid & 31) == 0) s_part[tid >> 5] = v;
        }
        __syncthreads();
        if (tid < 32) {
            float v = tid < 8 ? s_part[tid] : 0.f;
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (tid == 0) l.z_out[0] = v / (float)l.T;
        }
    }
}

// Record the first device error in the workspace header (later ones are dropped).
__device__ __forceinline__ void record_error(DeviceHeader* h, int32_t code, int32_t info) {
    if (atomicCAS(&h->err_code, 0, code) == 0) h->err_info = info;
}

}  // namespace moe
