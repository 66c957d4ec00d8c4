// Expert-choice routing: each expert takes the C tokens of the batch with the
// largest router probability p[t][e], and the chosen rows are gathered into
// expert-contiguous order.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "Design variations" (each expert selects the tokens it takes, which
// balances the load by construction).  Larger p first, the lower token index first among equal p; each
// expert's rows are its chosen tokens in ascending token order, so expert e
// owns rows e*C .. e*C + C - 1.
//
// Selection: one block per expert over its column of p (stored [E][T] by the
// router, held in shared memory when it fits).  p >= 0, so the fp32 bit
// patterns order like the values; a 4-pass radix select (8 bits a pass)
// finds the bit pattern of the C-th largest value, v, and how many of the C
// are equal to v; a pass in token order then takes every token above v and
// the first of those equal to v, with two block-wide prefix counts giving
// each taken token its row.

#include <cuda_runtime.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
// columns of up to 50,176 tokens are cached in shared memory (196 KB)
constexpr size_t kMaxCachedKeyBytes = 196 * 1024;

// Exclusive prefix count of `flag` over the block (in thread order) and the
// block total.  Every thread must call it; it synchronises the block.
__device__ __forceinline__ int block_prefix(bool flag, int* s_warp, int* total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) s_warp[warp] = __popc(b);
    __syncthreads();
    int before = __popc(b & ((1u << lane) - 1u)), sum = 0;
#pragma unroll 4
    for (int w = 0; w < kSelWarps; ++w) {
        const int v = s_warp[w];
        before += w < warp ? v : 0;
        sum += v;
    }
    *total = sum;
    __syncthreads();  // s_warp is reused by the next call
    return before;
}

// CACHED: the expert's column is first copied to shared memory (T keys) and
// every pass reads it there; otherwise every pass reads it from global memory.
template <bool CACHED>
__global__ void __launch_bounds__(kSelThreads) ec_select_kernel(
    const float* __restrict__ probs_t, int T, int E, int C, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm_token, float* __restrict__ perm_w, int32_t* __restrict__ slot_of,
    int32_t* __restrict__ expert_counts) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ unsigned s_keys[];
    __shared__ unsigned hist[256];
    __shared__ int s_warp[kSelWarps];
    __shared__ unsigned s_prefix;
    __shared__ int s_need;
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid % 32;
    const unsigned* col = reinterpret_cast<const unsigned*>(probs_t + (size_t)e * T);
    if (tid == 0) {
        offsets[e] = e * C;
        if (e == E - 1) offsets[E] = E * C;
        if (expert_counts != nullptr) expert_counts[e] = C;
    }
    if (C == 0) {
        for (int t = tid; t < T; t += kSelThreads) slot_of[(size_t)t * E + e] = -1;
        return;
    }
    if (CACHED) {
        for (int t = tid; t < T; t += kSelThreads) s_keys[t] = __ldg(col + t);
    }
    auto key = [&](int t) -> unsigned { return CACHED ? s_keys[t] : __ldg(col + t); };
    // radix select of the C-th largest bit pattern
    unsigned prefix = 0, mask = 0;
    int need = C;  // rank of the wanted value among those matching prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < T; base += kSelThreads) {  // uniform trip count
            const int t = base + tid;
            const unsigned u = t < T ? key(t) : 0u;
            const bool ok = t < T && (u & mask) == prefix;
            const unsigned dig = (u >> shift) & 255u;
            // lanes with the same digit add once (the top bits of p are few)
            const unsigned grp = __match_any_sync(0xffffffffu, ok ? dig : 0x100u);
            if (ok && lane == __ffs(grp) - 1) atomicAdd(&hist[dig], (unsigned)__popc(grp));
        }
        __syncthreads();
        if (tid < 32) {
            // lane l holds digits 255-8l down to 248-8l; a prefix sum over the
            // lanes finds the lane, then the digit, holding the need-th largest
            unsigned c[8];
            int sl = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sl += (int)c[j];
            }
            int incl = sl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int above = incl - sl;
            if (above < need && need <= incl) {
                int j = 0;
                for (; j < 7; ++j) {
                    if (above + (int)c[j] >= need) break;
                    above += (int)c[j];
                }
                s_prefix = prefix | ((unsigned)(255 - 8 * lane - j) << shift);
                s_need = need - above;
            }
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 255u << shift;
    }
    const unsigned v = prefix;  // the C-th largest; `need` of the chosen equal it
    // take, in token order, every token above v and the first `need` equal to v
    int eq_before = 0, taken_before = 0;
    for (int base = 0; base < T; base += kSelThreads) {
        const int t = base + tid;
        const unsigned u = t < T ? key(t) : 0u;
        const bool gt = t < T && u > v, eq = t < T && u == v;
        int eq_total, take_total;
        const int eq_rank = eq_before + block_prefix(eq, s_warp, &eq_total);
        const bool take = gt || (eq && eq_rank < need);
        const int pos = taken_before + block_prefix(take, s_warp, &take_total);
        if (t < T) {
            int row = -1;
            if (take) {
                row = e * C + pos;
                perm_token[row] = t;
                perm_w[row] = __uint_as_float(u);
            }
            slot_of[(size_t)t * E + e] = row;
        }
        eq_before += eq_total;
        taken_before += take_total;
    }
}

// x_perm[r] = x[perm_token[r]], one warp per row, 16-byte vectors.
template <typename TX>
__global__ void __launch_bounds__(256) ec_gather_kernel(const TX* __restrict__ x,
                                                         const int32_t* __restrict__ perm_token,
                                                         int64_t rows, int T, int d,
                                                         TX* __restrict__ x_perm) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x % 32;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int nvec = d * (int)sizeof(TX) / 16;
    for (int64_t r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += nwarps) {
        const int t = __ldg(perm_token + r);
        if (t < 0 || t >= T) continue;  // never written by the selection kernel
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * d);
        int vv = lane;
        for (; vv + 96 < nvec; vv += 128) {
            const uint4 q0 = __ldg(src + vv), q1 = __ldg(src + vv + 32);
            const uint4 q2 = __ldg(src + vv + 64), q3 = __ldg(src + vv + 96);
            dst[vv] = q0; dst[vv + 32] = q1; dst[vv + 64] = q2; dst[vv + 96] = q3;
        }
        for (; vv < nvec; vv += 32) dst[vv] = __ldg(src + vv);
    }
}

}  // namespace

int ec_capacity(const moe_config& c) {
    int64_t cap = c.capacity >= 0 ? (int64_t)c.capacity
                                  : ((int64_t)c.T * c.k + c.E - 1) / c.E;  // ceil(T k / E)
    if (cap > c.T) cap = c.T;
    return (int)cap;
}

cudaError_t launch_ec_select(const moe_config& c, const float* probs_t, int32_t* offsets,
                             int32_t* perm_token, float* perm_w, int32_t* slot_of,
                             int32_t* expert_counts, cudaStream_t s) {
    const size_t keys = sizeof(unsigned) * (size_t)c.T;
    if (keys <= kMaxCachedKeyBytes) {
        cudaError_t err = ensure_smem<ec_select_kernel<true>>((int)kMaxCachedKeyBytes);
        if (err != cudaSuccess) return err;
        return launch_kernel(ec_select_kernel<true>, dim3(c.E), dim3(kSelThreads), keys, s, 1,
                             false, probs_t, c.T, c.E, ec_capacity(c), offsets, perm_token,
                             perm_w, slot_of, expert_counts);
    }
    return launch_kernel(ec_select_kernel<false>, dim3(c.E), dim3(kSelThreads), 0, s, 1, false,
                         probs_t, c.T, c.E, ec_capacity(c), offsets, perm_token, perm_w, slot_of,
                         expert_counts);
}

cudaError_t launch_ec_gather(const moe_config& c, const void* x, const int32_t* perm_token,
                             void* x_perm, cudaStream_t s) {
    const int64_t rows = (int64_t)c.E * ec_capacity(c);
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > num_sms() * 8) blocks = num_sms() * 8;
    if (c.dtype == MOE_BF16)
        return launch_kernel(ec_gather_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0,
                             s, 1, false, reinterpret_cast<const __nv_bfloat16*>(x), perm_token,
                             rows, c.T, c.d, reinterpret_cast<__nv_bfloat16*>(x_perm));
    return launch_kernel(ec_gather_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, 1, false,
                         reinterpret_cast<const float*>(x), perm_token, rows, c.T, c.d,
                         reinterpret_cast<float*>(x_perm));
}

}  // namespace moe
