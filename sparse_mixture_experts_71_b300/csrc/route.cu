// Router kernel: logits g = W_r x (+ bias), softmax, top-k, gate weights,
// per-expert counts and the Switch auxiliary loss, fused in one pass over x.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer" (steps 1-2) and section "The central problem: load
// balancing" (auxiliary loss E * sum_i f_i P_i, f_i from the top-1 choice,
// P_i the mean probability).
//
// One block owns TB tokens and every expert.  The logits tile is an fp32 SIMT
// GEMM: x and W_r are staged through shared memory in chunks of KC columns,
// each thread accumulates a 4-token x 8-expert register tile over a 1/S
// slice of the chunk columns, and the S partial tiles are summed in a fixed
// order (deterministic).  Softmax and top-k run one warp per token.  The last
// block to finish reduces the per-block probability sums (fixed order) and
// writes the auxiliary loss and the per-expert counts.

#include <cuda_runtime.h>
#include <float.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int KC = 32;   // columns of x / W_r per shared-memory chunk
constexpr int RT = 4;    // tokens per thread tile
constexpr int RE = 8;    // experts per thread tile

struct RouteArgs {
    const void* x;
    const float* W_r;
    const float* bias;
    const float* logits_in;
    float* logits_out;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* expert_counts;
    float* aux_out;
    DeviceHeader* hdr;
    int32_t* counts;     // ws: [E] all-slot assignments
    int32_t* top1;       // ws: [E] first-slot choices
    float* blk_p;        // ws: [nblk][E]
    int T, d, E, k, renormalize, nblk;
};

template <int EMAX> struct Geo {
    static constexpr int TB = EMAX > 128 ? 32 : 64;  // tokens per block
    static constexpr int TG = TB / RT;                // token groups
    static constexpr int EG = EMAX / RE;              // expert groups
    static constexpr int G = TG * EG;                 // thread tiles per block
    static constexpr int S = kThreads / G;            // column splits
    static_assert(S >= 1 && G * S == kThreads, "tile geometry");
    static constexpr int LGS = EMAX + 1;              // logits tile row stride
    // shared memory (floats): x chunk, W chunk, then partial tiles / logits
    static constexpr int XS = KC * TB;
    static constexpr int WS = KC * EMAX;
    static constexpr int RED = (S > 1 ? S * G * RT * RE : 0);
    static constexpr int LG = TB * LGS;
    static constexpr int SMEM_FLOATS = XS + WS + (RED > LG ? RED : LG);
};

// Stage a TB x KC chunk of x (transposed to [col][token]) and a EMAX x KC
// chunk of W_r (to [col][expert]) in shared memory; zero outside the matrix.
template <typename TX, int EMAX>
__device__ __forceinline__ void stage_chunk(const RouteArgs& a, int t0, int c0, float* xs,
                                            float* wsm) {
    using Gm = Geo<EMAX>;
    const TX* x = reinterpret_cast<const TX*>(a.x);
    // x: TB tokens x (KC/8) groups of 8 columns
    for (int i = threadIdx.x; i < Gm::TB * (KC / 8); i += kThreads) {
        const int tok = i % Gm::TB, cg = i / Gm::TB;
        const int t = t0 + tok, c = c0 + cg * 8;
        float v[8];
        if (t < a.T && c < a.d) {
            load8_f32(x + (size_t)t * a.d + c, v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) xs[(cg * 8 + q) * Gm::TB + tok] = v[q];
    }
    // W_r: EMAX experts x (KC/8) groups
    for (int i = threadIdx.x; i < EMAX * (KC / 8); i += kThreads) {
        const int e = i % EMAX, cg = i / EMAX;
        const int c = c0 + cg * 8;
        float v[8];
        if (e < a.E && c < a.d) {
            load8_f32(a.W_r + (size_t)e * a.d + c, v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) wsm[(cg * 8 + q) * EMAX + e] = v[q];
    }
}

template <typename TX, int EMAX>
__global__ void __launch_bounds__(kThreads) route_kernel(RouteArgs a) {
    using Gm = Geo<EMAX>;
    extern __shared__ float4 smem_f4[];
    float* smem = reinterpret_cast<float*>(smem_f4);
    float* xs = smem;
    float* wsm = xs + Gm::XS;
    float* lg = wsm + Gm::WS;                 // logits tile [TB][LGS] (after reduction)
    float* red = lg;                          // partial tiles, aliases lg
    __shared__ int s_cnt[EMAX];
    __shared__ int s_top1[EMAX];
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * Gm::TB;
    for (int e = tid; e < EMAX; e += kThreads) { s_cnt[e] = 0; s_top1[e] = 0; }

    if (a.logits_in == nullptr) {
        // ---- logits tile: SIMT GEMM with a per-thread 4x8 register tile
        const int g = tid % Gm::G, s = tid / Gm::G;
        const int tg = g % Gm::TG, eg = g / Gm::TG;
        float acc[RT][RE];
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
            for (int j = 0; j < RE; ++j) acc[i][j] = 0.f;
        for (int c0 = 0; c0 < a.d; c0 += KC) {
            __syncthreads();
            stage_chunk<TX, EMAX>(a, t0, c0, xs, wsm);
            __syncthreads();
#pragma unroll 4
            for (int c = s; c < KC; c += Gm::S) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + c * Gm::TB + tg * RT);
                const float4 w0 = *reinterpret_cast<const float4*>(wsm + c * EMAX + eg * RE);
                const float4 w1 = *reinterpret_cast<const float4*>(wsm + c * EMAX + eg * RE + 4);
                const float xr[RT] = {xv.x, xv.y, xv.z, xv.w};
                const float wr[RE] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int i = 0; i < RT; ++i)
#pragma unroll
                    for (int j = 0; j < RE; ++j) acc[i][j] = fmaf(xr[i], wr[j], acc[i][j]);
            }
        }
        __syncthreads();
        if (Gm::S > 1) {
            // partial tiles -> red[s][g][RT*RE], then a fixed-order sum over s
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int j = 0; j < RE; ++j) red[((s * Gm::G) + g) * (RT * RE) + i * RE + j] = acc[i][j];
            __syncthreads();
            float out[(Gm::G * RT * RE) / kThreads];
#pragma unroll
            for (int q = 0; q < (Gm::G * RT * RE) / kThreads; ++q) {
                const int o = tid + q * kThreads;  // o = gg * (RT*RE) + r
                float v = 0.f;
                for (int ss = 0; ss < Gm::S; ++ss) v += red[ss * Gm::G * RT * RE + o];
                out[q] = v;
            }
            __syncthreads();  // red aliases lg
#pragma unroll
            for (int q = 0; q < (Gm::G * RT * RE) / kThreads; ++q) {
                const int o = tid + q * kThreads;
                const int gg = o / (RT * RE), r = o % (RT * RE);
                const int tok = (gg % Gm::TG) * RT + r / RE, e = (gg / Gm::TG) * RE + r % RE;
                lg[tok * Gm::LGS + e] = out[q];
            }
        } else {
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int j = 0; j < RE; ++j) lg[(tg * RT + i) * Gm::LGS + eg * RE + j] = acc[i][j];
        }
        __syncthreads();
        if (a.bias != nullptr) {
            for (int i = tid; i < Gm::TB * a.E; i += kThreads) {
                const int tok = i / a.E, e = i % a.E;
                lg[tok * Gm::LGS + e] += __ldg(a.bias + e);
            }
        }
    } else {
        __syncthreads();
        for (int i = tid; i < Gm::TB * a.E; i += kThreads) {
            const int tok = i / a.E, e = i % a.E;
            const int t = t0 + tok;
            lg[tok * Gm::LGS + e] = t < a.T ? __ldg(a.logits_in + (size_t)t * a.E + e) : 0.f;
        }
    }
    __syncthreads();

    // ---- softmax and top-k, one warp per token; lane l owns experts l + 32 i
    const int warp = tid / 32, lane = tid % 32;
    constexpr int PER_LANE = (EMAX + 31) / 32;
    for (int tok = warp; tok < Gm::TB; tok += kThreads / 32) {
        const int t = t0 + tok;
        if (t >= a.T) {
            for (int e = lane; e < EMAX; e += 32) lg[tok * Gm::LGS + e] = 0.f;
            continue;
        }
        float gv[PER_LANE];
        float m = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            gv[i] = e < a.E ? lg[tok * Gm::LGS + e] : -FLT_MAX;
            if (e < a.E) {
                m = fmaxf(m, gv[i]);
                if (a.logits_out != nullptr)
                    a.logits_out[(size_t)t * a.E + e] = gv[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float ex[PER_LANE];
        float ssum = 0.f;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            ex[i] = e < a.E ? expf(gv[i] - m) : 0.f;
            ssum += ex[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
        const float inv = 1.0f / ssum;
        // top-k: k rounds of a warp arg-max on the logits (ties -> lower index)
        bool taken[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) taken[i] = false;
        int sel_e[kMaxTopK];
        float sel_x[kMaxTopK];
        float sel_sum = 0.f;
        for (int j = 0; j < a.k; ++j) {
            float bv = -FLT_MAX;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i) {
                const int e = lane + 32 * i;
                if (e < a.E && !taken[i] && (gv[i] > bv || (gv[i] == bv && e < be))) {
                    bv = gv[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
            }
            float xe = 0.f;
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i) {
                if (lane + 32 * i == be) { taken[i] = true; xe = ex[i]; }
            }
            xe = __shfl_sync(0xffffffffu, xe, be % 32);
            sel_e[j] = be;
            sel_x[j] = xe;
            sel_sum += xe;
        }
        if (lane == 0) {
            const float wden = a.renormalize ? 1.0f / sel_sum : inv;
            for (int j = 0; j < a.k; ++j) {
                a.topk_idx[(size_t)t * a.k + j] = sel_e[j];
                a.topk_w[(size_t)t * a.k + j] = sel_x[j] * wden;
                atomicAdd(&s_cnt[sel_e[j]], 1);
            }
            atomicAdd(&s_top1[sel_e[0]], 1);
        }
        // probabilities replace the logits in the tile (for the column sums)
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (e < EMAX) lg[tok * Gm::LGS + e] = e < a.E ? ex[i] * inv : 0.f;
        }
    }
    __syncthreads();

    // ---- per-block sums of p (fixed token order) and counts
    for (int e = tid; e < a.E; e += kThreads) {
        float v = 0.f;
        for (int tok = 0; tok < Gm::TB; ++tok) v += lg[tok * Gm::LGS + e];
        a.blk_p[(size_t)blockIdx.x * a.E + e] = v;
        if (s_cnt[e]) atomicAdd(&a.counts[e], s_cnt[e]);
        if (s_top1[e]) atomicAdd(&a.top1[e], s_top1[e]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&a.hdr->route_done, 1u) == (unsigned)(a.nblk - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last block: P_e over all blocks in block order, then the loss
    double* dsum = reinterpret_cast<double*>(smem);  // the x chunk region is free now
    for (int e = tid; e < a.E; e += kThreads) {
        double v = 0.0;
        for (int b = 0; b < a.nblk; ++b) v += (double)__ldcg(a.blk_p + (size_t)b * a.E + e);
        const int c1 = __ldcg(a.top1 + e);
        dsum[e] = (double)c1 * v;
        if (a.expert_counts != nullptr) a.expert_counts[e] = __ldcg(a.counts + e);
    }
    __syncthreads();
    if (tid == 0 && a.aux_out != nullptr) {
        double s = 0.0;
        for (int e = 0; e < a.E; ++e) s += dsum[e];
        const double Td = (double)a.T;
        a.aux_out[0] = (float)((double)a.E * s / (Td * Td));
    }
}

template <typename TX, int EMAX>
cudaError_t launch_t(const RouteArgs& a, cudaStream_t s) {
    using Gm = Geo<EMAX>;
    const size_t smem = (size_t)Gm::SMEM_FLOATS * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(route_kernel<TX, EMAX>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    route_kernel<TX, EMAX><<<a.nblk, kThreads, smem, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

template <typename TX>
cudaError_t launch_e(const RouteArgs& a, cudaStream_t s) {
    if (a.E <= 8) return launch_t<TX, 8>(a, s);
    if (a.E <= 16) return launch_t<TX, 16>(a, s);
    if (a.E <= 32) return launch_t<TX, 32>(a, s);
    if (a.E <= 64) return launch_t<TX, 64>(a, s);
    if (a.E <= 128) return launch_t<TX, 128>(a, s);
    return launch_t<TX, 256>(a, s);
}

}  // namespace

int route_tokens_per_block(int E) { return E > 128 ? Geo<256>::TB : Geo<8>::TB; }

cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r,
                         const float* logit_bias, const float* logits_in, float* logits_out,
                         int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                         float* aux_out, void* ws, const WsLayout& L, cudaStream_t s) {
    RouteArgs a;
    a.x = x; a.W_r = W_r; a.bias = logit_bias; a.logits_in = logits_in; a.logits_out = logits_out;
    a.topk_idx = topk_idx; a.topk_w = topk_w; a.expert_counts = expert_counts; a.aux_out = aux_out;
    a.hdr = at<DeviceHeader>(ws, L.header);
    a.counts = at<int32_t>(ws, L.counts);
    a.top1 = at<int32_t>(ws, L.top1);
    a.blk_p = at<float>(ws, L.blk_p);
    a.T = c.T; a.d = c.d; a.E = c.E; a.k = c.k; a.renormalize = c.renormalize;
    a.nblk = L.route_blocks;
    // per-call counters: route_done and the two count arrays start at zero
    cudaError_t err = cudaMemsetAsync(at<char>(ws, L.header + offsetof(DeviceHeader, route_done)),
                                      0, sizeof(uint32_t), s);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(at<char>(ws, L.counts), 0, L.blk_p - L.counts, s);
    if (err != cudaSuccess) return err;
    return c.dtype == MOE_BF16 ? launch_e<__nv_bfloat16>(a, s) : launch_e<float>(a, s);
}

}  // namespace moe
