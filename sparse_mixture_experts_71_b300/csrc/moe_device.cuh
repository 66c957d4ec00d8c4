// Device helpers shared by the libmoe kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

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

// GELU 0.5 u (1 + erf(z)), z = u / sqrt 2, with erf from the rational
// approximation of Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (Hastings): for z >= 0, erf(z) = 1 - q(t) exp(-z^2),
// t = 1 / (1 + p z), q(t) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))), with
// |error| <= 1.5e-7.  1 + erf(z) is q e^{-z^2} for z < 0 and 2 - q e^{-z^2}
// for z >= 0, which keeps the negative tail free of cancellation.  Used where
// the result is rounded to bf16 (relative step 2^-8), far above the error.
__device__ __forceinline__ float gelu_as7126(float u) {
    const float z = fabsf(u) * 0.70710678118654752440f;
    const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
    float q = fmaf(t, 1.061405429f, -1.453152027f);
    q = fmaf(t, q, 1.421413741f);
    q = fmaf(t, q, -0.284496736f);
    q = fmaf(t, q, 0.254829592f);
    q *= t;
    const float r = q * __expf(-z * z);
    return 0.5f * u * (u < 0.f ? r : 2.0f - r);
}

// Record the first device error in the workspace header (later ones are dropped).
__device__ __forceinline__ void record_error(DeviceHeader* h, int32_t code, int32_t info) {
    if (atomicCAS(&h->err_code, 0, code) == 0) h->err_info = info;
}

}  // namespace moe
