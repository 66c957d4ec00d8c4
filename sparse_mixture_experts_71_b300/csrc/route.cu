// Router kernels: logits g = W_r x (+ bias), softmax, top-k, gate weights,
// per-expert counts and the Switch auxiliary loss, fused in one pass over x.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer" (steps 1-2) and section "The central problem: load
// balancing" (auxiliary loss E * sum_i f_i P_i, f_i from the top-1 choice,
// P_i the mean probability).
//
// Two tilings of the logits GEMM (fp32 FMA, exact products, fp32 sums):
//   warp kernel (E <= 32)  one warp owns TW tokens; lanes split d into
//                          8-column chunks (16-byte loads of x, W_r rows from
//                          L1/L2), a butterfly all-reduce gives every lane the
//                          TW x E logits, and each token's softmax / top-k runs
//                          in registers.  8 warps per block.  The pass is
//                          bound by reading x once.
//   tile kernel (E > 32)   one block owns TB tokens and every expert; x and
//                          W_r chunks are staged in shared memory and each
//                          thread accumulates a 4-token x 8-expert register
//                          tile over a slice of the chunk columns; the partial
//                          tiles are summed in a fixed order.  Softmax and
//                          top-k then run one warp per token.
// Both end alike: per-block sums of p in fixed token order, integer counts,
// optionally the block's expert histogram and the rank of each assignment
// among the block's earlier assignments to the same expert (consumed by the
// dispatch scan), and in the last block to finish the auxiliary loss from the
// per-block sums taken in block order (deterministic).

#include <cuda_runtime.h>
#include <float.h>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "route_common.cuh"

namespace moe {
namespace {

using namespace rt;

// ===================================================================== warp kernel
// DS warps split one token group's d columns (DS > 1 for small batches, so
// that enough blocks exist); their partial logits meet in shared memory and
// are added in split order.
template <typename TX, int EMAX, int TW, int DS>
__global__ void __launch_bounds__(kThreads) route_warp_kernel(RouteArgs a) {
    pdl_wait();
    pdl_trigger();
    constexpr int G = kWarps / DS;   // token groups per block
    constexpr int TB = G * TW;       // tokens per block
    constexpr int LDS = EMAX + 1;
    __shared__ float s_p[TB * LDS];
    __shared__ float s_red[DS > 1 ? kWarps * TW * EMAX : 1];
    __shared__ int s_idx[TB * kMaxTopK];
    __shared__ int s_cnt[EMAX], s_top1[EMAX], carry[EMAX];
    __shared__ int wh[kWarps][EMAX];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int grp = warp / DS, split = warp % DS;
    if (tid < EMAX) { s_cnt[tid] = 0; s_top1[tid] = 0; }
    for (int i = tid; i < TB * LDS; i += kThreads) s_p[i] = 0.f;
    __syncthreads();
    const int tb = blockIdx.x * TB + grp * TW;  // first token of this warp's group

    float acc[TW][EMAX];
#pragma unroll
    for (int i = 0; i < TW; ++i)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc[i][e] = 0.f;

    if (a.logits_in == nullptr) {
        const TX* x = reinterpret_cast<const TX*>(a.x);
        const int nchunk = a.d / 8;
        for (int ch = split * 32 + lane; ch < nchunk; ch += 32 * DS) {
            const int c = ch * 8;
            float xv[TW][8];
#pragma unroll
            for (int i = 0; i < TW; ++i) {
                if (tb + i < a.T) {
                    load8_f32(x + (size_t)(tb + i) * a.d + c, xv[i]);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) xv[i][q] = 0.f;
                }
            }
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                if (e < a.E) {
                    float wv[8];
                    load8_f32(a.W_r + (size_t)e * a.d + c, wv);
#pragma unroll
                    for (int i = 0; i < TW; ++i)
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[i][e] = fmaf(xv[i][q], wv[q], acc[i][e]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < TW; ++i)
#pragma unroll
            for (int e = 0; e < EMAX; ++e)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
        if (DS > 1) {
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < TW; ++i)
#pragma unroll
                    for (int e = 0; e < EMAX; ++e) s_red[(warp * TW + i) * EMAX + e] = acc[i][e];
            }
            __syncthreads();
            if (split == 0) {
#pragma unroll
                for (int i = 0; i < TW; ++i)
#pragma unroll
                    for (int e = 0; e < EMAX; ++e) {
                        float v = 0.f;
#pragma unroll
                        for (int s2 = 0; s2 < DS; ++s2)
                            v += s_red[((grp * DS + s2) * TW + i) * EMAX + e];
                        acc[i][e] = v;
                    }
            }
        }
        if (a.bias != nullptr) {
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                const float b = e < a.E ? __ldg(a.bias + e) : 0.f;
#pragma unroll
                for (int i = 0; i < TW; ++i) acc[i][e] += b;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < TW; ++i)
#pragma unroll
            for (int e = 0; e < EMAX; ++e)
                if (tb + i < a.T && e < a.E) acc[i][e] = __ldg(a.logits_in + (size_t)(tb + i) * a.E + e);
    }

    // the group's logits go to shared memory; then one thread per token
    if (split == 0 && lane == 0) {
#pragma unroll
        for (int i = 0; i < TW; ++i)
#pragma unroll
            for (int e = 0; e < EMAX; ++e) s_p[(grp * TW + i) * LDS + e] = acc[i][e];
    }
    __syncthreads();
    stage_logits<EMAX>(a, s_p, LDS, TB, blockIdx.x * TB);
    __syncthreads();
    if (tid < TB) token_epilogue<EMAX>(a, s_p + tid * LDS, blockIdx.x * TB + tid, tid, s_idx, s_cnt, s_top1);
    __syncthreads();
    finish_block<EMAX>(a, s_p, LDS, TB, s_idx, s_cnt, s_top1, wh, carry, blockIdx.x);
}

// ===================================================================== tensor-core kernel
// bf16 x with E <= 16.  The logits are a skinny GEMM (N = E); each warp owns
// a 16-token tile and runs mma.sync m16n8k16 (bf16 in, fp32 accumulate)
// against W_r split in registers into three bf16 parts (hi + mid + lo = W_r
// exactly), so every product is exact and only the fp32 accumulation rounds,
// as in the fp32 SIMT path.  The K order inside each 32-column chunk is permuted so
// that one 16-byte load per row feeds two MMAs: MMA column slots (2t, 2t+1,
// 2t+8, 2t+9) of lane quad t map to physical columns 8t .. 8t+3 in the first
// MMA and 8t+4 .. 8t+7 in the second, identically for x and W_r.
// DS warps split the d columns of one tile when the batch is small; their
// partial tiles are added in split order.

// W_r (fp32 [E][d]) -> three bf16 parts [3][epad][d], rows >= E zero.
__global__ void __launch_bounds__(256) split_router_weight(const float* __restrict__ W, int E,
                                                           int epad, int d,
                                                           __nv_bfloat16* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const size_t n = (size_t)epad * d;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(i / d);
        const float w = e < E ? __ldg(W + i) : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        out[i] = hi;
        out[n + i] = mid;
        out[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT, int MT>
__global__ void __launch_bounds__(kThreads) route_mma_kernel(RouteArgs a) {
    pdl_wait();
    pdl_trigger();
    constexpr int EMAX = 8 * NT;
    constexpr int DS = kWarps / MT;
    constexpr int TB = 16 * MT;
    constexpr int LDS = EMAX + 1;
    constexpr int BUF = (DS > 1 && kWarps * 16 * EMAX > TB * LDS) ? kWarps * 16 * EMAX : TB * LDS;
    __shared__ float s_buf[BUF];  // split partials, then logits / probabilities [TB][LDS]
    __shared__ int s_idx[TB * kMaxTopK];
    __shared__ int s_cnt[EMAX], s_top1[EMAX], carry[EMAX];
    __shared__ int wh[kWarps][EMAX];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int mtile = warp / DS, split = warp % DS;
    const int g = lane >> 2, tq = lane & 3;
    if (tid < EMAX) { s_cnt[tid] = 0; s_top1[tid] = 0; }
    const int tok0 = blockIdx.x * TB + mtile * 16;
    const int r0 = tok0 + g, r1 = tok0 + g + 8;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

    if (a.logits_in == nullptr) {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a.x);
        const int nchunk = (a.d + 31) / 32;
#pragma unroll 2
        for (int ch = split; ch < nchunk; ch += DS) {
            const int c = ch * 32 + 8 * tq;
            const bool cin = c < a.d;
            uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
            if (cin && r0 < a.T) xa = __ldg(reinterpret_cast<const uint4*>(x + (size_t)r0 * a.d + c));
            if (cin && r1 < a.T) xb = __ldg(reinterpret_cast<const uint4*>(x + (size_t)r1 * a.d + c));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // this lane's 8 W_r values (expert nt*8+g, columns c..c+7), split
                // into hi + mid + lo bf16 parts, packed in column pairs
                float w[8];
                const int e = nt * 8 + g;
                if (cin && e < a.E) {
                    load8_f32(a.W_r + (size_t)e * a.d + c, w);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) w[q] = 0.f;
                }
                uint32_t part[3][4];
#pragma unroll
                for (int q = 0; q < 8; q += 2) {
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(w[q], w[q + 1]);
                    const float r0 = w[q] - __low2float(hi), r1 = w[q + 1] - __high2float(hi);
                    const __nv_bfloat162 mid = __floats2bfloat162_rn(r0, r1);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(r0 - __low2float(mid),
                                                                   r1 - __high2float(mid));
                    part[0][q / 2] = *reinterpret_cast<const uint32_t*>(&hi);
                    part[1][q / 2] = *reinterpret_cast<const uint32_t*>(&mid);
                    part[2][q / 2] = *reinterpret_cast<const uint32_t*>(&lo);
                }
#pragma unroll
                for (int pp = 0; pp < 3; ++pp) {
                    mma_bf16_16816(acc[nt], xa.x, xb.x, xa.y, xb.y, part[pp][0], part[pp][1]);
                    mma_bf16_16816(acc[nt], xa.z, xb.z, xa.w, xb.w, part[pp][2], part[pp][3]);
                }
            }
        }
        if (DS > 1) {
            // partial tiles of the splits -> s_buf[warp][16][EMAX]; split 0 adds them in order
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float* row0 = s_buf + (warp * 16 + g) * EMAX + nt * 8 + 2 * tq;
                float* row1 = s_buf + (warp * 16 + g + 8) * EMAX + nt * 8 + 2 * tq;
                row0[0] = acc[nt][0]; row0[1] = acc[nt][1];
                row1[0] = acc[nt][2]; row1[1] = acc[nt][3];
            }
            __syncthreads();
            if (split == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = g + (q >> 1) * 8, col = nt * 8 + 2 * tq + (q & 1);
                        float v = 0.f;
                        for (int s2 = 0; s2 < DS; ++s2)
                            v += s_buf[((mtile * DS + s2) * 16 + row) * EMAX + col];
                        acc[nt][q] = v;
                    }
                }
            }
            __syncthreads();  // s_buf is rewritten as the logits tile below
        }
        if (split == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = g + (q >> 1) * 8, col = nt * 8 + 2 * tq + (q & 1);
                    float v = acc[nt][q];
                    if (a.bias != nullptr && col < a.E) v += __ldg(a.bias + col);
                    s_buf[(mtile * 16 + row) * LDS + col] = v;
                }
            }
        }
    } else {
        for (int i = tid; i < TB * EMAX; i += kThreads) {
            const int tok = i / EMAX, e = i % EMAX;
            const int t = blockIdx.x * TB + tok;
            s_buf[tok * LDS + e] = (t < a.T && e < a.E) ? __ldg(a.logits_in + (size_t)t * a.E + e) : 0.f;
        }
    }
    __syncthreads();
    stage_logits<EMAX>(a, s_buf, LDS, TB, blockIdx.x * TB);
    __syncthreads();
    if (tid < TB) token_epilogue<EMAX>(a, s_buf + tid * LDS, blockIdx.x * TB + tid, tid, s_idx, s_cnt, s_top1);
    __syncthreads();
    finish_block<EMAX>(a, s_buf, LDS, TB, s_idx, s_cnt, s_top1, wh, carry, blockIdx.x);
}

// ===================================================================== tile kernel
constexpr int KC = 32;   // columns of x / W_r per shared-memory chunk
constexpr int RT = 4;    // tokens per thread tile
constexpr int RE = 8;    // experts per thread tile

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
__global__ void __launch_bounds__(kThreads) route_tile_kernel(RouteArgs a) {
    pdl_wait();
    pdl_trigger();
    using Gm = Geo<EMAX>;
    extern __shared__ float4 smem_f4[];
    float* smem = reinterpret_cast<float*>(smem_f4);
    float* xs = smem;
    float* wsm = xs + Gm::XS;
    float* lg = wsm + Gm::WS;                 // logits tile [TB][LGS] (after reduction)
    float* red = lg;                          // partial tiles, aliases lg
    __shared__ int s_idx[Gm::TB * kMaxTopK];
    __shared__ int s_cnt[EMAX], s_top1[EMAX], carry[EMAX];
    __shared__ int wh[kWarps][EMAX];

    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * Gm::TB;
    for (int e = tid; e < EMAX; e += kThreads) { s_cnt[e] = 0; s_top1[e] = 0; }

    if (a.logits_in == nullptr) {
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
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int j = 0; j < RE; ++j)
                    red[((s * Gm::G) + g) * (RT * RE) + i * RE + j] = acc[i][j];
            __syncthreads();
            float out[(Gm::G * RT * RE) / kThreads];
#pragma unroll
            for (int q = 0; q < (Gm::G * RT * RE) / kThreads; ++q) {
                const int o = tid + q * kThreads;
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

    // softmax and top-k, one warp per token; lane l owns experts l + 32 i
    const int warp = tid / 32, lane = tid % 32;
    constexpr int PER_LANE = (EMAX + 31) / 32;
    for (int tok = warp; tok < Gm::TB; tok += kWarps) {
        const int t = t0 + tok;
        if (t >= a.T) {
            for (int e = lane; e <= EMAX; e += 32) lg[tok * Gm::LGS + e] = 0.f;
            continue;
        }
        float gv[PER_LANE];
        float m = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            gv[i] = e < a.E ? lg[tok * Gm::LGS + e] : -FLT_MAX;
            if (e < a.E && a.noise != nullptr) gv[i] += __ldg(a.noise + (size_t)t * a.E + e);
            if (e < a.E) {
                m = fmaxf(m, gv[i]);
                if (a.logits_out != nullptr) a.logits_out[(size_t)t * a.E + e] = gv[i];
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
        if (lane == 0) {  // squared log-sum-exp (router z-loss) in the pad column
            const float lse = m + logf(ssum);
            lg[tok * Gm::LGS + EMAX] = lse * lse;
        }
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
            sel_sum += j < a.knorm ? xe : 0.f;
        }
        if (lane == 0) {
            const float wden = a.renormalize ? 1.0f / sel_sum : inv;
            for (int j = 0; j < a.k; ++j) {
                a.topk_idx[(size_t)t * a.k + j] = sel_e[j];
                a.topk_w[(size_t)t * a.k + j] = sel_x[j] * wden;
                s_idx[tok * a.k + j] = sel_e[j];
                if (j < a.knorm) atomicAdd(&s_cnt[sel_e[j]], 1);
            }
            atomicAdd(&s_top1[sel_e[0]], 1);
        }
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (e < EMAX) lg[tok * Gm::LGS + e] = e < a.E ? ex[i] * inv : 0.f;
        }
    }
    __syncthreads();
    finish_block<EMAX>(a, lg, Gm::LGS, Gm::TB, s_idx, s_cnt, s_top1, wh, carry, blockIdx.x);
}

template <typename TX, int EMAX>
cudaError_t launch_tile(const RouteArgs& a, cudaStream_t s) {
    using Gm = Geo<EMAX>;
    const size_t smem = (size_t)Gm::SMEM_FLOATS * sizeof(float);
    cudaError_t err = ensure_smem<route_tile_kernel<TX, EMAX>>((int)smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(route_tile_kernel<TX, EMAX>, dim3(a.nblk), dim3(kThreads), smem, s, 1, false, a);
}

template <typename TX, int EMAX, int TW, int DS>
cudaError_t launch_warp(const RouteArgs& a, cudaStream_t s) {
    return launch_kernel(route_warp_kernel<TX, EMAX, TW, DS>, dim3(a.nblk), dim3(kThreads), 0, s,
                         1, false, a);
}

template <typename TX, int EMAX>
cudaError_t launch_warp_tw(const RouteArgs& a, const RouteGeom& g, cudaStream_t s) {
    if (g.tw >= 4) return g.ds == kWarps ? launch_warp<TX, EMAX, 4, kWarps>(a, s)
                                         : launch_warp<TX, EMAX, 4, 1>(a, s);
    if (g.tw == 2) return g.ds == kWarps ? launch_warp<TX, EMAX, 2, kWarps>(a, s)
                                         : launch_warp<TX, EMAX, 2, 1>(a, s);
    if (g.ds >= 8) return launch_warp<TX, EMAX, 1, 8>(a, s);
    if (g.ds == 4) return launch_warp<TX, EMAX, 1, 4>(a, s);
    if (g.ds == 2) return launch_warp<TX, EMAX, 1, 2>(a, s);
    return launch_warp<TX, EMAX, 1, 1>(a, s);
}

template <int NT, int MT>
cudaError_t launch_mma_t(const RouteArgs& a, cudaStream_t s) {
    return launch_kernel(route_mma_kernel<NT, MT>, dim3(a.nblk), dim3(kThreads), 0, s, 1, false, a);
}

template <int NT>
cudaError_t launch_mma_nt(const RouteArgs& a, const RouteGeom& g, cudaStream_t s) {
    if (g.mt >= 8) return launch_mma_t<NT, 8>(a, s);
    if (g.mt == 4) return launch_mma_t<NT, 4>(a, s);
    if (g.mt == 2) return launch_mma_t<NT, 2>(a, s);
    return launch_mma_t<NT, 1>(a, s);
}

cudaError_t launch_split(const RouteArgs& a, int epad, __nv_bfloat16* wsp, cudaStream_t s) {
    if (a.logits_in != nullptr) return cudaSuccess;
    const size_t n = (size_t)epad * a.d;
    int blocks = (int)((n + 255) / 256);
    blocks = blocks < num_sms() * 4 ? blocks : num_sms() * 4;
    return launch_kernel(split_router_weight, dim3(blocks), dim3(256), 0, s, 1, false, a.W_r, a.E, epad,
                         a.d, wsp);
}

cudaError_t launch_mma(const RouteArgs& a, const RouteGeom& g, cudaStream_t s) {
    if (g.epad <= 8) return launch_mma_nt<1>(a, g, s);
    return launch_mma_nt<2>(a, g, s);
}

template <typename TX>
cudaError_t launch_e(const RouteArgs& a, const RouteGeom& g, cudaStream_t s) {
    if (g.warp) {
        if (a.E <= 8) return launch_warp_tw<TX, 8>(a, g, s);
        if (a.E <= 16) return launch_warp_tw<TX, 16>(a, g, s);
        return launch_warp_tw<TX, 32>(a, g, s);
    }
    if (a.E <= 64) return launch_tile<TX, 64>(a, s);
    if (a.E <= 128) return launch_tile<TX, 128>(a, s);
    return launch_tile<TX, 256>(a, s);
}

__global__ void __launch_bounds__(256) route_finish_kernel(LossArgs l) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_part[256];
    __shared__ float s_d[kMaxExperts];
    loss_and_counts(l, s_part, s_d);
}

// Shared experts: token t's K = k + ns columns are its k routed choices (ids
// offset by ns, weights as routed) and then experts 0 .. ns-1 with weight 1;
// block 0 also writes the per-expert counts over all E experts (a shared
// expert takes every token).
__global__ void __launch_bounds__(256) join_shared_kernel(
    const int32_t* __restrict__ idx_r, const float* __restrict__ w_r, int T, int k, int ns,
    int32_t* __restrict__ idx, float* __restrict__ w, const int32_t* __restrict__ counts_r,
    int32_t* __restrict__ expert_counts, int E) {
    pdl_wait();
    pdl_trigger();
    const int K = k + ns;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        for (int j = 0; j < k; ++j) {
            idx[(size_t)t * K + j] = __ldg(idx_r + (size_t)t * k + j) + ns;
            w[(size_t)t * K + j] = __ldg(w_r + (size_t)t * k + j);
        }
        for (int j = 0; j < ns; ++j) {
            idx[(size_t)t * K + k + j] = j;
            w[(size_t)t * K + k + j] = 1.0f;
        }
    }
    if (blockIdx.x == 0 && expert_counts != nullptr)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            expert_counts[e] = e < ns ? T : __ldcg(counts_r + e - ns);
}

// One block: sum of the counts (int64, in order by thread then tree), then
// each expert's step against the exact mean.
__global__ void __launch_bounds__(256) balance_bias_kernel(const int32_t* __restrict__ counts,
                                                           int E, float* __restrict__ bias,
                                                           float step) {
    pdl_wait();
    pdl_trigger();
    __shared__ long long s_sum[256];
    long long v = 0;
    for (int e = threadIdx.x; e < E; e += 256) v += counts[e];
    s_sum[threadIdx.x] = v;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) s_sum[threadIdx.x] += s_sum[threadIdx.x + o];
        __syncthreads();
    }
    const long long total = s_sum[0];
    for (int e = threadIdx.x; e < E; e += 256) {
        const long long scaled = (long long)counts[e] * E;
        if (scaled > total) bias[e] -= step;
        else if (scaled < total) bias[e] += step;
    }
}

}  // namespace

cudaError_t launch_join_shared(const moe_config& c, const int32_t* idx_r, const float* w_r,
                               int32_t* topk_idx, float* topk_w, const int32_t* counts_r,
                               int32_t* expert_counts, cudaStream_t s) {
    int blocks = (c.T + 255) / 256;
    blocks = blocks < num_sms() * 4 ? blocks : num_sms() * 4;
    return launch_kernel(join_shared_kernel, dim3(blocks), dim3(256), 0, s, 1, false, idx_r, w_r,
                         c.T, c.k, c.n_shared, topk_idx, topk_w, counts_r, expert_counts, c.E);
}

cudaError_t launch_balance_bias(const moe_config& c, const int32_t* counts, float* bias,
                                float step, cudaStream_t s) {
    return launch_kernel(balance_bias_kernel, dim3(1), dim3(256), 0, s, 1, false, counts, c.E,
                         bias, step);
}

LossArgs route_loss_args(const moe_config& c, void* ws, const WsLayout& L,
                         int32_t* expert_counts, float* aux_out, float* z_loss_out) {
    LossArgs l;
    l.blk_p = at<float>(ws, L.blk_p);
    l.blk_z = at<float>(ws, L.blk_z);
    l.z_out = z_loss_out;
    l.top1 = at<int32_t>(ws, L.top1);
    l.counts = at<int32_t>(ws, L.counts);
    l.expert_counts = expert_counts;
    l.aux_out = aux_out;
    l.nblk = L.route.blocks;
    l.E = c.E;
    l.T = c.T;
    return l;
}

RouteGeom route_geom(const moe_config& c) {
    RouteGeom g{};
    constexpr int kTargetBlocks = 296;  // two blocks per SM at least, where T allows
    if (c.dtype == MOE_BF16 && c.E > 16 && c.E <= 64 && c.T >= 1024) {
        g.tc = true;
        g.epad = c.E <= 32 ? 32 : 64;
        g.tokens = 128;
    } else if (c.dtype == MOE_BF16 && c.E <= 16 && c.T >= 1024) {
        g.mma = true;
        g.epad = c.E <= 8 ? 8 : 16;
        int mt = 8;
        while (mt > 1 && (c.T + 16 * mt - 1) / (16 * mt) < kTargetBlocks) mt /= 2;
        g.mt = mt;
        g.ds = kWarps / mt;
        g.tokens = 16 * mt;
    } else if (c.E <= 32) {
        g.warp = true;
        int tw = c.E <= 16 ? 4 : 2, ds = 1;
        while (tw > 1 && (c.T + kWarps * tw - 1) / (kWarps * tw) < kTargetBlocks) tw /= 2;
        while (tw == 1 && ds < kWarps && (c.T * ds + kWarps - 1) / kWarps < kTargetBlocks) ds *= 2;
        g.tw = tw;
        g.ds = ds;
        g.tokens = (kWarps / ds) * tw;
    } else {
        g.warp = false;
        g.tw = 0;
        g.ds = 1;
        g.tokens = c.E > 128 ? Geo<256>::TB : Geo<64>::TB;
    }
    g.blocks = (c.T + g.tokens - 1) / g.tokens;
    return g;
}

namespace {

RouteArgs route_args(const moe_config& c, const void* x, const float* W_r,
                     const float* logit_bias, const float* logit_noise, const float* logits_in,
                     float* logits_out, int32_t* topk_idx, float* topk_w,
                     int32_t* expert_counts, float* aux_out, void* ws, const WsLayout& L,
                     bool fuse_count, float* probs_t, int knorm) {
    RouteArgs a;
    a.probs_t = probs_t;
    a.knorm = knorm > 0 ? knorm : c.k;
    a.x = x; a.W_r = W_r; a.bias = logit_bias; a.logits_in = logits_in; a.logits_out = logits_out;
    a.noise = logits_in != nullptr ? nullptr : logit_noise;  // logits_in replaces all terms
    a.topk_idx = topk_idx; a.topk_w = topk_w; a.expert_counts = expert_counts; a.aux_out = aux_out;
    a.hdr = at<DeviceHeader>(ws, L.header);
    a.counts = at<int32_t>(ws, L.counts);
    a.top1 = at<int32_t>(ws, L.top1);
    a.blk_p = at<float>(ws, L.blk_p);
    a.blk_z = at<float>(ws, L.blk_z);
    a.blk_hist = fuse_count ? at<int32_t>(ws, L.blk_hist) : nullptr;
    a.local_rank = at<int32_t>(ws, L.local_rank);
    a.T = c.T; a.d = c.d; a.E = c.E; a.k = c.k; a.renormalize = c.renormalize;
    a.nblk = L.route.blocks;
    return a;
}

cudaError_t route_kernels(const moe_config& c, const RouteArgs& a, void* ws, const WsLayout& L,
                          cudaStream_t s) {
    if (L.route.mma) return launch_mma(a, L.route, s);
    if (L.route.tc) {
        __nv_bfloat16* wsp = at<__nv_bfloat16>(ws, L.wsplit);
        cudaError_t err = launch_split(a, L.route.epad, wsp, s);
        return err == cudaSuccess ? launch_route_tc(a, wsp, L.route.epad, s) : err;
    }
    return c.dtype == MOE_BF16 ? launch_e<__nv_bfloat16>(a, L.route, s)
                               : launch_e<float>(a, L.route, s);
}

}  // namespace

RouteGeom route_geom_beside(const moe_config& c) {
    RouteGeom g = route_geom(c);
    // the warp kernel with d split over all eight warps (as route_geom picks
    // for small batches): more tokens per warp group cut the blocks and leave
    // each token's sum - split partials added in split order - unchanged, so
    // the logits are route_geom's to the bit
    if (g.warp && g.tw == 1 && g.ds == kWarps) {
        g.tw = c.E <= 16 ? 4 : 2;
        g.tokens = (kWarps / g.ds) * g.tw;
        g.blocks = (c.T + g.tokens - 1) / g.tokens;
    }
    return g;
}

cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r,
                         const float* logit_bias, const float* logit_noise,
                         const float* logits_in, float* logits_out,
                         int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                         float* aux_out, float* z_loss_out, void* ws, const WsLayout& L,
                         bool fuse_count, cudaStream_t s, float* probs_t, int knorm) {
    const RouteArgs a = route_args(c, x, W_r, logit_bias, logit_noise, logits_in, logits_out,
                                   topk_idx, topk_w, expert_counts, aux_out, ws, L, fuse_count,
                                   probs_t, knorm);
    // per-call counters: the two count arrays start at zero
    cudaError_t err = cudaMemsetAsync(at<char>(ws, L.counts), 0, L.blk_p - L.counts, s);
    if (err != cudaSuccess) return err;
    chain_begin();  // the next kernel follows the memset
    err = route_kernels(c, a, ws, L, s);
    if (err != cudaSuccess || fuse_count) return err;
    if (expert_counts == nullptr && aux_out == nullptr && z_loss_out == nullptr) return err;
    return launch_kernel(route_finish_kernel, dim3(1), dim3(256), 0, s, 1, false,
                         route_loss_args(c, ws, L, expert_counts, aux_out, z_loss_out));
}

cudaError_t launch_route_no_finish(const moe_config& c, const void* x, const float* W_r,
                                   const float* logit_bias, const float* logit_noise,
                                   float* logits_out, int32_t* topk_idx, float* topk_w, void* ws,
                                   const WsLayout& L, cudaStream_t s) {
    const RouteArgs a = route_args(c, x, W_r, logit_bias, logit_noise, nullptr, logits_out,
                                   topk_idx, topk_w, nullptr, nullptr, ws, L, false, nullptr, 0);
    return route_kernels(c, a, ws, L, s);
}

}  // namespace moe
