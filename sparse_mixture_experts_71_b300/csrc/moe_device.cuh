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

// Record the first device error in the workspace header (later ones are dropped).
__device__ __forceinline__ void record_error(DeviceHeader* h, int32_t code, int32_t info) {
    if (atomicCAS(&h->err_code, 0, code) == 0) h->err_info = info;
}

}  // namespace moe
