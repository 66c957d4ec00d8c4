// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer": each expert is Linear(d, d_ff) + bias, GELU,
// Linear(d_ff, d) + bias, applied to the token rows dispatched to it; the
// weighted combination of the expert outputs follows (the routing weight is
// applied here, in the second GEMM's epilogue).
//
// Orientation ("weights as the M operand"): for expert e and a tile of its
// token rows r0 .. r0+n-1,
//     D[f][j] = sum_k W[e][f][k] * X[r0 + j][k]      (f: 128 weight rows)
// so the 128-row MMA dimension is always full (weight rows) and the token
// dimension N is set per tile at run time to n rounded up to 16 (single CTA)
// or 32 (CTA pair; the instruction descriptor is a register operand).  Small expert segments
// (decode, skewed routing) then cost MMA work in proportion to their size.
//
// Two persistent, warp-specialised kernels share these roles:
//   warp 0      TMA producer: weight and token boxes (64 K columns, 128-byte
//               swizzle) into a shared-memory ring, completion counted on a
//               full barrier;
//   warp 1      MMA issuer: tcgen05.mma (K = 16 each) into one of two TMEM
//               accumulators; tcgen05.commit frees a stage and, after the
//               last K-step of a tile, signals the epilogue;
//   warp 2      TMEM allocator;
//   warp 3      computes the per-expert tile table from the device offsets;
//   warps 4..   epilogue: tcgen05.ld of the accumulator, bias + GELU (first
//               GEMM, bf16 h) or bias x routing weight (second GEMM, fp32
//               y_perm), transposed through shared memory into row-major
//               output.
//   grouped_gemm_pair (token tiles of up to 256 rows): a cluster of two CTAs
//               computes 256 weight rows x 256 tokens with cta_group::2
//               MMAs (M = 256); three stages of two K atoms; 16 (first GEMM)
//               or 8 (second) epilogue warps; output by TMA tensor stores.
//               Used one GEMM at a time by the backward pass (and its
//               segment-reduction mode for the weight gradients).
//   ffn_pair_kernel: the same CTA pairs running both GEMMs of the forward
//               expert FFN in one persistent launch (first-GEMM tiles, then
//               second-GEMM tiles gated by per-token-tile ready counts; the
//               second GEMM may split each tile's K in two halves when the
//               half tiles fill the last wave of pairs better).
//   grouped_gemm_tc (decode-sized batches, token tiles of up to 64 rows):
//               one CTA per SM, M = 128, eight stages; 8 epilogue warps;
//               output by 16-byte lane stores.
// The two TMEM accumulators let the epilogue of tile i overlap the MMAs of
// tile i+1.  Every wait is bounded: past the time limit the kernel records
// an error in the workspace, drains its in-flight copies and MMAs, frees TMEM
// and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int BM = 128;                      // weight rows per tile (MMA M)
constexpr int BK = 64;                       // K per stage: one 128-byte swizzle row
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int BOX_ROWS = 32;                 // token rows per TMA box
constexpr int BOX_BYTES = BOX_ROWS * BK * 2; // 4 KB
constexpr uint64_t kDrainNs = 2000000000ull; // drain waits on the error path

template <int BN_MAX, int STAGES, bool GEMM1>
struct Cfg {
    static constexpr int B_BYTES = BN_MAX * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int OUT_ES = GEMM1 ? 2 : 4;
    static constexpr int STAGING = kEpiWarps * 32 * 32 * OUT_ES;
    static constexpr int TMEM_COLS = 2 * BN_MAX;
    static constexpr int OFF_STAGING = STAGES * STAGE_BYTES;
    static constexpr int OFF_BARS = OFF_STAGING + STAGING;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
    static constexpr int OFF_TILES = OFF_MISC + 16;
    static constexpr int SMEM = OFF_TILES + (kMaxExperts + 1) * 4 + 1023;
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 512, "TMEM allocation");
};

struct Params {
    const int32_t* offsets;     // [E+1] segment starts (device)
    const __nv_bfloat16* bias;  // [E][n_out] or null (no bias)
    const float* row_w;         // [rows] routing weight per row (second GEMM) or null
    void* out;                  // first GEMM: bf16 [rows][n_out]; second: fp32 [rows][n_out]
    DeviceHeader* hdr;
    uint64_t timeout_ns;
    int E, n_out, K, rows_cap;
    int act;                    // first GEMM: 1 = GELU, 0 = none (the pre-activation)
    // Segment-reduction mode (CTA-pair kernel, second-GEMM epilogue;
    // seg_maps not null): out[e*tok_rows + i][n] = sum over the rows r of
    // expert e's segment (offsets) of TOK[r][i] * WT[r][n], both operands
    // row-major over the permuted rows ([rows][tok_rows], [rows][n_out]) and
    // read MN-major: the K dimension of the MMAs is the segment's rows.
    // seg_maps[2e] (WT) and seg_maps[2e + 1] (TOK) are tensor maps of that
    // segment alone (rows past its end read as zero), written on the device
    // by seg_maps_kernel.  An empty segment gives zeros.
    const CUtensorMap* seg_maps;
    int tok_rows;
    // CTA-pair kernel: 1 when the operand maps are the 3-D views of
    // make_map3 (one box covers a stage's ATOMS K atoms), 0 for 2-D maps
    // (one box per atom)
    int box3d;
    // fused expert FFN, second GEMM: per-tile counts of the first K half's
    // epilogue warps when it splits K (zero at launch), ksync_cap of them
    int32_t* ksync;
    int ksync_cap;
    // CTA-pair kernel, not segment reduction: 1 when the weight operand is
    // W [E][K][n_out] (the transpose of the usual [E][n_out][K]), read
    // MN-major through a map of 64-column x 128-row boxes over its E*K rows
    int a_mn;
    // first-GEMM epilogue: when not null, the pre-activation (acc + bias,
    // before the GELU) is also written, rounded to bf16, to pre_out
    // [rows][n_out] (the backward pass's U beside H = GELU)
    __nv_bfloat16* pre_out;
    // first-GEMM epilogue (bf16 out, no bias, no GELU): when not null, each
    // output element o[r][n], once rounded to bf16, is multiplied by
    // GELU'(gelu_u[r][n]) (the backward pass's dU = dH GELU'(U); gelu_u
    // [rows][n_out] bf16) and rounded again
    const __nv_bfloat16* gelu_u;
    // with gelu_u: when not null, also the dots of each output row with
    // GELU(gelu_u) over every 16 columns, before the GELU' scaling:
    // spart[r][n / 16] = sum over the 16 columns n of o[r][n] GELU(u[r][n])
    // (o rounded to bf16; ceil(n_out / 16) a row; the backward pass's slot
    // scores)
    float* spart;
};

// Rows of an expert's segment (offsets clamped to the buffers).
__device__ __forceinline__ int seg_rows(const Params& p, int e) {
    const int s0 = min(max(__ldg(p.offsets + e), 0), p.rows_cap);
    const int s1 = min(max(__ldg(p.offsets + e + 1), s0), p.rows_cap);
    return s1 - s0;
}


struct Tile {
    int e, r0, n, m0;
    int o0;  // first output row (r0 except in dense mode)
};

// Work item t of the single-CTA kernel: expert e, token tile (fastest) and
// 128-row weight tile.
__device__ __forceinline__ Tile decode_tile(int t, const int* s_tiles, const Params& p,
                                            int bn_max) {
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {  // last expert whose first item is <= t
        const int mid = (lo + hi + 1) >> 1;
        if (s_tiles[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Tile tl;
    tl.e = lo;
    const int local = t - s_tiles[lo];
    const int s0 = min(max(__ldg(p.offsets + lo), 0), p.rows_cap);
    const int s1 = min(max(__ldg(p.offsets + lo + 1), s0), p.rows_cap);
    const int nt = (s1 - s0 + bn_max - 1) / bn_max;
    const int ti = local % nt, gi = local / nt;  // token tile fastest
    tl.r0 = s0 + ti * bn_max;
    tl.o0 = tl.r0;
    tl.n = min(bn_max, s1 - tl.r0);
    tl.m0 = gi * BM;
    return tl;
}

// Wait for phase `parity` of `bar`; false if the kernel is aborting or the
// time limit passed (then the abort flag is raised and the error recorded).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         const Params& p, int where) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (tc::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p.hdr, kErrTimeout, where);
            return false;
        }
    }
    return true;
}

// Drain wait: bounded by a fixed limit only (used on the way out).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (tc::globaltimer() - t0 > kDrainNs) break;
    }
}

// Epilogue of one accumulator tile: this warp reads TMEM lanes 32q..32q+31
// (weight rows fbase + 32q + lane) and the token columns of its part (of
// nparts) of the COLS-wide tile (columns acc_col + c, c < n), applies bias + GELU (first
// GEMM, bf16 out) or bias x routing weight (second GEMM, fp32 out; the
// weight of input row r0 + c), and writes output rows o0 + c through a
// shared-memory transpose (stg: 32 x 32).
// With tm_out (second GEMM of the pair kernel) a full 32-row chunk leaves
// shared memory by a TMA tensor store issued by lane 0 (box 32 weight rows x
// 32 token rows of the output), so the warp neither reads the staging back
// nor issues the global stores; a partial chunk (the end of an expert's
// segment: the rows after it belong to the next segment) is stored by the
// lanes.
template <int COLS, bool GEMM1, bool ZERO_TILES = false>
__device__ __forceinline__ void epilogue_tile(const Params& p, int e, int r0, int o0, int n,
                                              int fbase,
                                              uint32_t tmem_base, int acc_col, int q, int part,
                                              int nparts, int lane, uint8_t* stg,
                                              const CUtensorMap* tm_out = nullptr,
                                              bool zero = false, bool accumulate = false) {
    const int f0 = fbase + q * 32;  // first weight row (output feature) of this warp
    const int f = f0 + lane;
    // accumulate (second GEMM, second K half): out += acc * w, the bias having
    // come with the first half; full chunks by TMA reduce-add, the others by a
    // plain load, add and store (a float atomic would flush subnormals)
    const float bias = f < p.n_out && p.bias != nullptr && !accumulate
                           ? __bfloat162float(p.bias[(size_t)e * p.n_out + f])
                           : 0.f;
    const int c_begin = part * (COLS / nparts), c_end = min(c_begin + COLS / nparts, n);
    for (int c = c_begin; c < c_end; c += 32) {
        float v[32];
        if constexpr (ZERO_TILES) {
            if (zero) {  // no MMA wrote this accumulator: its contents are undefined
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            } else {
                tc::tmem_ld_32cols(tmem_base + ((uint32_t)(q * 32) << 16) +
                                       (uint32_t)(acc_col + c),
                                   v);
            }
        } else {
            tc::tmem_ld_32cols(tmem_base + ((uint32_t)(q * 32) << 16) +
                                   (uint32_t)(acc_col + c),
                               v);
        }
        const int rows_here = min(32, n - c);
        if (GEMM1) {
            __nv_bfloat16* s16 = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 u = __fadd2_rn(make_float2(v[j], v[j + 1]), make_float2(bias, bias));
                const float2 g = p.act ? gelu2_as7126(u) : u;
                s16[j * 32 + lane] = __float2bfloat16_rn(g.x);
                s16[(j + 1) * 32 + lane] = __float2bfloat16_rn(g.y);
            }
            __syncwarp();
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int ci = lane + 32 * i, j = ci >> 2, part = ci & 3;
                const int fc = f0 + part * 8;
                if (j < rows_here && fc < p.n_out) {
                    const uint4 val = *reinterpret_cast<const uint4*>(stg + j * 64 + part * 16);
                    *reinterpret_cast<uint4*>(out + (size_t)(o0 + c + j) * p.n_out + fc) = val;
                }
            }
        } else {
            float wl = 1.f;
            if (p.row_w != nullptr && lane < rows_here) wl = __ldg(p.row_w + r0 + c + lane);
            if (zero) wl = 0.f;  // an empty segment's tile is zero whatever the bias
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (v[j] + bias) * __shfl_sync(0xffffffffu, wl, j);
            if (tm_out != nullptr) {  // the previous chunk's store has read the staging rows
                if (lane == 0) tc::bulk_wait_read_all();
                __syncwarp();
            }
            float* s32 = reinterpret_cast<float*>(stg);
#pragma unroll
            for (int j = 0; j < 32; ++j) s32[j * 32 + lane] = v[j];
            if (tm_out != nullptr && rows_here == 32 && f0 < p.n_out) {
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (accumulate)
                        tc::tma_reduce_add_2d(tm_out, stg, f0, o0 + c);
                    else
                        tc::tma_store_2d(tm_out, stg, f0, o0 + c);
                    tc::bulk_commit();
                }
                continue;
            }
            __syncwarp();
            float* out = reinterpret_cast<float*>(p.out);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ci = lane + 32 * i, j = ci >> 3, part = ci & 7;
                const int fc = f0 + part * 4;
                if (j < rows_here && fc < p.n_out) {
                    const float4 val = *reinterpret_cast<const float4*>(stg + j * 128 + part * 16);
                    float4* dst = reinterpret_cast<float4*>(out + (size_t)(o0 + c + j) * p.n_out + fc);
                    if (accumulate) {
                        const float4 o = __ldcg(dst);
                        *dst = make_float4(o.x + val.x, o.y + val.y, o.z + val.z, o.w + val.w);
                    } else {
                        *dst = val;
                    }
                }
            }
        }
        __syncwarp();
    }
}

template <int BN_MAX, int STAGES, bool GEMM1>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const Params p) {
    using C = Cfg<BN_MAX, STAGES, GEMM1>;
    const int cta = blockIdx.x, nctas = gridDim.x;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* s_tiles = reinterpret_cast<int*>(smem + C::OFF_TILES);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mt = (p.n_out + BM - 1) / BM;
    const int KB = (p.K + BK - 1) / BK;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], kEpiWarps);
        }
        tc::mbar_init(drain, 1);
        *s_abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
    }
    if (warp == 2) {
        tc::tmem_alloc(s_tmem, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    pdl_wait();  // offsets and the operands come from the previous kernel
    pdl_trigger();
    if (warp == 3) {  // exclusive prefix of tiles per expert
        int run = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            int nt = 0;
            if (e < p.E) {
                nt = ((seg_rows(p, e) + BN_MAX - 1) / BN_MAX) * mt;
            }
            int v = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (e < p.E) s_tiles[e] = run + v - nt;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_tiles[p.E] = run;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const int total = s_tiles[p.E];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int t = cta; t < total && ok; t += nctas) {
                const Tile tl = decode_tile(t, s_tiles, p, BN_MAX);
                const int nb = (tl.n + BOX_ROWS - 1) / BOX_ROWS;
                const uint32_t bytes = A_BYTES + nb * BOX_BYTES;
                const int arow = tl.e * p.n_out + tl.m0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(&empty[stage], phase ^ 1, s_abort, p, 1)) { ok = false; break; }
                    tc::mbar_expect_tx(&full[stage], bytes);
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    tc::tma_load_2d(sa, &tmA, &full[stage], kb * BK, arow);
                    for (int b = 0; b < nb; ++b)
                        tc::tma_load_2d(sb + b * BOX_BYTES, &tmB, &full[stage], kb * BK,
                                        tl.r0 + b * BOX_ROWS);
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            // every issued copy lands before the CTA can exit
            const long long last = fills < STAGES ? fills : STAGES;
            for (long long i = fills - last; i < fills; ++i)
                drain_bar(&full[i % STAGES], (uint32_t)((i / STAGES) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = cta; t < total && ok; t += nctas) {
                const Tile tl = decode_tile(t, s_tiles, p, BN_MAX);
                const uint32_t n_mma = (uint32_t)((tl.n + 15) / 16) * 16;
                const uint32_t idesc = tc::idesc_bf16_f32(BM, n_mma);
                if (!wait_bar(&tempty[acc], acc_phase ^ 1, s_abort, p, 2)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN_MAX);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(&full[stage], phase, s_abort, p, 3)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t sa = tc::smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc::mma_bf16(d_tmem, tc::sdesc_k128_sw128(sa + kk * 32),
                                     tc::sdesc_k128_sw128(sb + kk * 32), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            // every issued MMA completes before TMEM is freed
            tc::mma_commit(drain);
            drain_bar(drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int ew = warp - 4;
        const int q = warp & 3;        // TMEM lane quarter this warp may access
        const int half = ew >> 2;      // which half of the tile's columns
        uint8_t* stg = smem + C::OFF_STAGING + ew * 32 * 32 * C::OUT_ES;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = cta; t < total; t += nctas) {
            const Tile tl = decode_tile(t, s_tiles, p, BN_MAX);
            const bool ok = wait_bar(&tfull[acc], acc_phase, s_abort, p, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            epilogue_tile<BN_MAX, GEMM1>(p, tl.e, tl.r0, tl.o0, tl.n, tl.m0, tmem_base,
                                         acc * BN_MAX, q, half, 2, lane, stg);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_relaxed(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ===================================================================== dense decode FFN
// Both expert GEMMs of a decode-sized batch in one persistent kernel, each
// expert evaluated on all T <= 64 tokens (moe_forward's dense decode path;
// every (expert, token) row equals the sparse path's: the MMA's rows are
// independent).  Work
// items 0 .. N1-1 are the first GEMM's 128-row weight tiles (expert
// e = i / mt1: h_all[e*T + t] = GELU(x[t] W1_e^T + b1_e), bf16), items
// N1 .. N1+N2-1 the second's (e = (i - N1) / mt2: y_all[e*T + t] =
// h_all[e*T + t] W2_e^T + b2_e, fp32).  The producer claims items in order
// from a counter in the workspace (so every item is claimed only after all
// earlier ones, by a CTA that is running) and hands each to the MMA and
// epilogue warps through a small ring in shared memory.  A second-GEMM item of
// expert e loads its first weight stages, then waits (bounded) until every
// epilogue warp of every first-GEMM item of e has stored its rows of h_all and
// counted itself in ready[e]; so the second GEMM starts on the SMs the first
// one frees, expert by expert, with no launch boundary or tail in between.
// A first-GEMM item never waits on anything but its own pipeline, so the
// waits always end.
struct DenseFfn {
    Params g1, g2;    // the two GEMMs (bias, activation, output, sizes, error record)
    int32_t* sched;   // [0] claim counter, [1 + e] ready arrivals of expert e (zero at launch)
    int T, n1, n2, mt1, mt2;
};

constexpr int kRing = 4;  // claimed items in flight between the roles

struct DenseCfg {
    using C = Cfg<64, 8, false>;  // 8 stages of a 128 x 64 weight box + two 32 x 64 token boxes
    static constexpr int STAGES = 8;
    static constexpr int OFF_RING = C::OFF_MISC + 16;          // ring: kRing ints
    static constexpr int OFF_RBARS = OFF_RING + kRing * 4;     // kRing full + kRing empty barriers
    static constexpr int SMEM = OFF_RBARS + 2 * kRing * 8 + 1023;
    static_assert(OFF_RBARS % 8 == 0, "barrier alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// wait_bar for warps with nothing else to do until the barrier completes (the
// epilogue warps of the fused FFN, which outnumber the issuing threads): a
// short sleep between polls leaves the issue slots to the producer and MMA
// threads of the same SM sub-partitions.
__device__ __forceinline__ bool wait_bar_idle(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, const Params& p,
                                              int where) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (tc::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p.hdr, kErrTimeout, where);
            return false;
        }
        __nanosleep(256);
    }
    return true;
}

// Spin (bounded by the pipeline time-out) until *cnt >= target; a time-out
// records the error (where) and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_count(const int32_t* cnt, int target, volatile int* abort_flag,
                                           const Params& p, int where) {
    if (ld_acquire_gpu(cnt) >= target) return true;
    const uint64_t t0 = tc::globaltimer();
    while (ld_acquire_gpu(cnt) < target) {
        if (*abort_flag) return false;
        if (tc::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p.hdr, kErrTimeout, where);
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
dense_ffn_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                 const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                 const DenseFfn f) {
    using C = DenseCfg::C;
    constexpr int STAGES = DenseCfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* ring = reinterpret_cast<volatile int*>(smem + DenseCfg::OFF_RING);
    uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + DenseCfg::OFF_RBARS);
    uint64_t* rempty = rfull + kRing;
    const Params& P = f.g1;  // error record and time limit

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = f.n1 + f.n2;
    const int nb = (f.T + BOX_ROWS - 1) / BOX_ROWS;
    const uint32_t bytes = A_BYTES + nb * BOX_BYTES;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], kEpiWarps);
        }
        for (int r = 0; r < kRing; ++r) {
            tc::mbar_init(&rfull[r], 1);
            tc::mbar_init(&rempty[r], 1 + kEpiWarps);
        }
        tc::mbar_init(drain, 1);
        *s_abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA1);
        tc::tma_prefetch_desc(&tmB1);
        tc::tma_prefetch_desc(&tmA2);
        tc::tma_prefetch_desc(&tmB2);
    }
    if (warp == 2) {
        tc::tmem_alloc(s_tmem, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    pdl_trigger();  // the inputs are the layer's: nothing to wait for before starting
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ claims + TMA producer
        if (lane == 0) {
            int stage = 0, slot = 0;
            uint32_t phase = 0, rphase = 0;
            long long fills = 0;
            bool ok = true;
            while (ok) {
                const int item = atomicAdd(f.sched, 1);
                const int it = item < total ? item : -1;
                if (!wait_bar(&rempty[slot], rphase ^ 1, s_abort, P, 5)) break;
                ring[slot] = it;
                asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                                 tc::smem_u32(&rfull[slot]))
                             : "memory");
                if (++slot == kRing) { slot = 0; rphase ^= 1; }
                if (it < 0) break;
                const bool first = it < f.n1;
                const int e = first ? it / f.mt1 : (it - f.n1) / f.mt2;
                const int m0 = (first ? it % f.mt1 : (it - f.n1) % f.mt2) * BM;
                const CUtensorMap* tA = first ? &tmA1 : &tmA2;
                const CUtensorMap* tB = first ? &tmB1 : &tmB2;
                const int KB = ((first ? f.g1.K : f.g2.K) + BK - 1) / BK;
                const int arow = e * (first ? f.g1.n_out : f.g2.n_out) + m0;
                const int brow = first ? 0 : e * f.T;
                // a second-GEMM item issues up to STAGES weight boxes before it
                // waits for its expert's rows of h_all, then their token boxes
                int deferred = 0;
                const int target = kEpiWarps * f.mt1;
                bool ready = first || ld_acquire_gpu(f.sched + 1 + e) >= target;
                if (!first && ready) asm volatile("fence.proxy.async.global;" ::: "memory");
                for (int kb = 0; kb < KB && ok; ++kb) {
                    if (!ready && (deferred == STAGES || ld_acquire_gpu(f.sched + 1 + e) >= target)) {
                        const uint64_t t0 = tc::globaltimer();
                        while (ld_acquire_gpu(f.sched + 1 + e) < target) {
                            if (*s_abort) { ok = false; break; }
                            if (tc::globaltimer() - t0 > P.timeout_ns) {
                                *s_abort = 1;
                                record_error(P.hdr, kErrTimeout, 6);
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        ready = true;
                        for (int q = 0; q < deferred; ++q) {
                            const int kq = kb - deferred + q;
                            const int sq = (int)((fills - deferred + q) % STAGES);
                            uint8_t* sb = smem + sq * C::STAGE_BYTES + A_BYTES;
                            for (int b = 0; b < nb; ++b)
                                tc::tma_load_2d(sb + b * BOX_BYTES, tB, &full[sq], kq * BK,
                                                brow + b * BOX_ROWS);
                        }
                        deferred = 0;
                    }
                    if (!wait_bar(&empty[stage], phase ^ 1, s_abort, P, 1)) { ok = false; break; }
                    tc::mbar_expect_tx(&full[stage], bytes);
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    tc::tma_load_2d(sa, tA, &full[stage], kb * BK, arow);
                    if (ready) {
                        for (int b = 0; b < nb; ++b)
                            tc::tma_load_2d(sa + A_BYTES + b * BOX_BYTES, tB, &full[stage], kb * BK,
                                            brow + b * BOX_ROWS);
                    } else {
                        ++deferred;
                    }
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (ok && !ready) {  // a short item: every K step deferred
                    const uint64_t t0 = tc::globaltimer();
                    while (ld_acquire_gpu(f.sched + 1 + e) < target) {
                        if (*s_abort || tc::globaltimer() - t0 > P.timeout_ns) {
                            if (!*s_abort) record_error(P.hdr, kErrTimeout, 6);
                            *s_abort = 1;
                            ok = false;
                            break;
                        }
                    }
                    if (ok) {
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        for (int q = 0; q < deferred; ++q) {
                            const int kq = KB - deferred + q;
                            const int sq = (int)((fills - deferred + q) % STAGES);
                            uint8_t* sb = smem + sq * C::STAGE_BYTES + A_BYTES;
                            for (int b = 0; b < nb; ++b)
                                tc::tma_load_2d(sb + b * BOX_BYTES, tB, &full[sq], kq * BK,
                                                brow + b * BOX_ROWS);
                        }
                    }
                }
            }
            // every issued copy lands before the CTA can exit
            const long long last = fills < STAGES ? fills : STAGES;
            for (long long i = fills - last; i < fills; ++i)
                drain_bar(&full[i % STAGES], (uint32_t)((i / STAGES) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0, slot = 0;
            uint32_t phase = 0, acc_phase = 0, rphase = 0;
            const uint32_t idesc = tc::idesc_bf16_f32(BM, (uint32_t)((f.T + 15) / 16) * 16);
            bool ok = true;
            while (ok) {
                if (!wait_bar(&rfull[slot], rphase, s_abort, P, 7)) break;
                const int it = ring[slot];
                tc::mbar_arrive_relaxed(&rempty[slot]);
                if (++slot == kRing) { slot = 0; rphase ^= 1; }
                if (it < 0) break;
                const int KB = ((it < f.n1 ? f.g1.K : f.g2.K) + BK - 1) / BK;
                if (!wait_bar(&tempty[acc], acc_phase ^ 1, s_abort, P, 2)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 64);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(&full[stage], phase, s_abort, P, 3)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t sa = tc::smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc::mma_bf16(d_tmem, tc::sdesc_k128_sw128(sa + kk * 32),
                                     tc::sdesc_k128_sw128(sb + kk * 32), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                    tc::mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            tc::mma_commit(drain);
            drain_bar(drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int ew = warp - 4;
        const int q = warp & 3;
        const int half = ew >> 2;
        uint8_t* stg = smem + C::OFF_STAGING + ew * 32 * 32 * C::OUT_ES;
        int acc = 0, slot = 0;
        uint32_t acc_phase = 0, rphase = 0;
        while (true) {
            const bool okr = wait_bar(&rfull[slot], rphase, s_abort, P, 8);
            if (!__all_sync(0xffffffffu, okr)) break;
            const int it = ring[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_relaxed(&rempty[slot]);
            if (++slot == kRing) { slot = 0; rphase ^= 1; }
            if (it < 0) break;
            const bool ok = wait_bar(&tfull[acc], acc_phase, s_abort, P, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            if (it < f.n1) {
                const int e = it / f.mt1;
                epilogue_tile<64, true>(f.g1, e, 0, e * f.T, f.T, (it % f.mt1) * BM, tmem_base,
                                        acc * 64, q, half, 2, lane, stg);
                // this warp's rows of h_all are stored: count them for expert e
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(f.sched + 1 + e, 1);
            } else {
                const int e = (it - f.n1) / f.mt2;
                epilogue_tile<64, false>(f.g2, e, e * f.T, e * f.T, f.T, ((it - f.n1) % f.mt2) * BM,
                                         tmem_base, acc * 64, q, half, 2, lane, stg);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_relaxed(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    // the grid completes only after the previous kernel of its chain (the
    // router), which it never waited for
    if (threadIdx.x == 0) pdl_wait();
}

// First-GEMM epilogue of the CTA-pair kernel for this CTA's 128 weight rows x
// n tokens of one accumulator.  Work items are 16 TMEM lanes (weight rows) x
// 32 columns (tokens); the NPQ warps of lane quarter q take the quarter's
// items round robin.  Per item a warp loads the accumulator in the fragment
// layout (tcgen05.ld 16x256b), adds the bias, applies GELU two values per
// instruction, packs token pairs to bf16x2 and writes the transpose to its
// staging rows with stmatrix (32 token rows of 16 weight rows = 32 bytes; the
// two 16-byte halves of a row swap when bit 2 of the token is set, which is
// the 32-byte TMA swizzle and keeps each stored 8 x 8 matrix on distinct
// banks).  A full item then leaves by one TMA tensor store (box 16 x 32) from
// lane 0; a partial one (the end of an expert's segment) by lane stores.
// Compared with 32 scalar shared stores and a read-back per 32 x 32 chunk this
// halves the epilogue's shared-memory traffic, which competes with the MMA
// operand reads and the TMA fills.
// The first-GEMM epilogue of the forward pass: bias (+ GELU), bf16, each
// item (16 weight rows x 32 tokens) through the warp's staging and out by a
// TMA tensor store (lane stores for a partial item).
template <int NPQ>
__device__ __forceinline__ void epilogue_gelu(const Params& p, int e, int r0, int n, int fbase,
                                              uint32_t tmem_base, int acc_col, int q, int wq,
                                              int lane, uint8_t* stg, const CUtensorMap* tm_out) {
    const int g = lane >> 2;
    const int items = 2 * ((n + 31) / 32);
    const __nv_bfloat16* bias = p.bias != nullptr ? p.bias + (size_t)e * p.n_out : nullptr;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    const uint32_t stg_s = tc::smem_u32(stg);
    // this lane's stmatrix row address (matrix lane/8, row lane%8) for the two stores
    const int mi = lane >> 3, rr = lane & 7;
    uint32_t st_addr[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int b = 2 * k + (mi >> 1), sh = mi & 1, tok = 8 * b + rr;
        st_addr[k] = stg_s + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4);
    }
    for (int it = wq; it < items; it += NPQ) {
        const int h = it & 1, c = (it >> 1) * 32;
        const int fr = fbase + q * 32 + h * 16;  // first weight row of the item
        const float ba = bias != nullptr && fr + g < p.n_out ? __bfloat162float(bias[fr + g]) : 0.f;
        const float bb =
            bias != nullptr && fr + 8 + g < p.n_out ? __bfloat162float(bias[fr + 8 + g]) : 0.f;
        uint32_t r[16];
        tc::tmem_ld_16x32(tmem_base + ((uint32_t)(q * 32 + h * 16) << 16) + (uint32_t)(acc_col + c), r);
        uint32_t pk[8];  // pk[2b]: rows g, pk[2b+1]: rows g + 8; tokens 8b + 2(lane%4), +1
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float2 ga = __fadd2_rn(
                make_float2(__uint_as_float(r[4 * b]), __uint_as_float(r[4 * b + 1])), make_float2(ba, ba));
            float2 gb = __fadd2_rn(
                make_float2(__uint_as_float(r[4 * b + 2]), __uint_as_float(r[4 * b + 3])), make_float2(bb, bb));
            if (p.act) {
                ga = gelu2_as7126(ga);
                gb = gelu2_as7126(gb);
            }
            const __nv_bfloat162 pa = __floats2bfloat162_rn(ga.x, ga.y);
            const __nv_bfloat162 pb = __floats2bfloat162_rn(gb.x, gb.y);
            pk[2 * b] = *reinterpret_cast<const uint32_t*>(&pa);
            pk[2 * b + 1] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        if (lane == 0) tc::bulk_wait_read_all();  // the previous store has read the rows
        __syncwarp();
        tc::stmatrix_x4_trans(st_addr[0], pk[0], pk[1], pk[2], pk[3]);
        tc::stmatrix_x4_trans(st_addr[1], pk[4], pk[5], pk[6], pk[7]);
        const int rows_here = min(32, n - c);
        if (rows_here == 32 && fr < p.n_out) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::tma_store_2d(tm_out, stg, fr, r0 + c);
                tc::bulk_commit();
            }
            continue;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int ci = lane + 32 * j, tok = ci >> 1, sh = ci & 1;
            const int fc = fr + 8 * sh;
            if (c + tok < n && fc < p.n_out) {
                const uint4 val = *reinterpret_cast<const uint4*>(
                    stg + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4));
                *reinterpret_cast<uint4*>(out + (size_t)(r0 + c + tok) * p.n_out + fc) = val;
            }
        }
        __syncwarp();
    }
}

// The first-GEMM epilogue with the backward pass's extra work (Params
// gelu_u, spart, pre_out): the forward epilogue's steps plus the
// pre-activation output, the GELU' scaling and the partial dots.
template <int NPQ>
__device__ __forceinline__ void epilogue_gelu_bwd(const Params& p, int e, int r0, int n, int fbase,
                                              uint32_t tmem_base, int acc_col, int q, int wq,
                                              int lane, uint8_t* stg_w, const CUtensorMap* tm_out) {
    const int g = lane >> 2;
    const int items = 2 * ((n + 31) / 32);
    const __nv_bfloat16* bias = p.bias != nullptr ? p.bias + (size_t)e * p.n_out : nullptr;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    const uint32_t stg_s = tc::smem_u32(stg_w);
    // this lane's stmatrix row address (matrix lane/8, row lane%8) for the two stores
    const int mi = lane >> 3, rr = lane & 7;
    uint32_t st_addr[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int b = 2 * k + (mi >> 1), sh = mi & 1, tok = 8 * b + rr;
        st_addr[k] = stg_s + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4);
    }
    // With the backward pass's extra epilogue work (gelu_u, pre_out) the
    // warp's 2 KB of staging holds two items: item i stages in half i % 2
    // while the store of item i - 1 may still be reading the other half (the
    // previous tile's stores, in either half, have read theirs first).  The
    // forward pass's plain GELU epilogue keeps one half (measured faster).
    const bool dbl = p.gelu_u != nullptr || p.pre_out != nullptr;
    if (dbl) {
        if (lane == 0) tc::bulk_wait_read_all();
        __syncwarp();
    }
    for (int it = wq, nth = 0; it < items; it += NPQ, ++nth) {
        const int h = it & 1, c = (it >> 1) * 32;
        const int fr = fbase + q * 32 + h * 16;  // first weight row of the item
        const uint32_t half = dbl ? (uint32_t)(nth & 1) * 1024u : 0u;
        uint8_t* stg = stg_w + half;
        const float ba = bias != nullptr && fr + g < p.n_out ? __bfloat162float(bias[fr + g]) : 0.f;
        const float bb =
            bias != nullptr && fr + 8 + g < p.n_out ? __bfloat162float(bias[fr + 8 + g]) : 0.f;
        // GELU' operand (Params::gelu_u): this lane's two 8-column chunks of
        // the item's U, loaded before the accumulator so the load overlaps it
        uint4 uq[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (p.gelu_u != nullptr) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int ci = lane + 32 * j, tok = ci >> 1, fc = fr + 8 * (ci & 1);
                if (c + tok < n && fc < p.n_out)
                    uq[j] = __ldg(reinterpret_cast<const uint4*>(
                        p.gelu_u + (size_t)(r0 + c + tok) * p.n_out + fc));
            }
        }
        uint32_t r[16];
        tc::tmem_ld_16x32(tmem_base + ((uint32_t)(q * 32 + h * 16) << 16) + (uint32_t)(acc_col + c), r);
        float2 v[8];  // v[2b]: rows g, v[2b+1]: rows g + 8; tokens 8b + 2(lane%4), +1
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            v[2 * b] = __fadd2_rn(
                make_float2(__uint_as_float(r[4 * b]), __uint_as_float(r[4 * b + 1])), make_float2(ba, ba));
            v[2 * b + 1] = __fadd2_rn(
                make_float2(__uint_as_float(r[4 * b + 2]), __uint_as_float(r[4 * b + 3])), make_float2(bb, bb));
        }
        uint32_t pk[8];
        if (lane == 0) {  // the store that last used this half has read it
            if (dbl) tc::bulk_wait_read_1();
            else tc::bulk_wait_read_all();
        }
        __syncwarp();
        if (p.pre_out != nullptr) {  // the pre-activation through staging to pre_out
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 pv = __float22bfloat162_rn(v[i]);
                pk[i] = *reinterpret_cast<const uint32_t*>(&pv);
            }
            tc::stmatrix_x4_trans(st_addr[0] + half, pk[0], pk[1], pk[2], pk[3]);
            tc::stmatrix_x4_trans(st_addr[1] + half, pk[4], pk[5], pk[6], pk[7]);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int ci = lane + 32 * j, tok = ci >> 1, sh = ci & 1;
                const int fc = fr + 8 * sh;
                if (c + tok < n && fc < p.n_out)
                    *reinterpret_cast<uint4*>(p.pre_out + (size_t)(r0 + c + tok) * p.n_out + fc) =
                        *reinterpret_cast<const uint4*>(
                            stg + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4));
            }
            __syncwarp();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 o = p.act ? gelu2_as7126(v[i]) : v[i];
            const __nv_bfloat162 pv = __float22bfloat162_rn(o);
            pk[i] = *reinterpret_cast<const uint32_t*>(&pv);
        }
        tc::stmatrix_x4_trans(st_addr[0] + half, pk[0], pk[1], pk[2], pk[3]);
        tc::stmatrix_x4_trans(st_addr[1] + half, pk[4], pk[5], pk[6], pk[7]);
        if (p.gelu_u != nullptr) {
            // staging holds the item's [32 tokens][16 columns] in bf16; each
            // lane scales two 8-column chunks by GELU' of the same U chunk
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int ci = lane + 32 * j, tok = ci >> 1, sh = ci & 1;
                const int fc = fr + 8 * sh;
                float part = 0.f;  // this chunk's dot with GELU(u) (Params::spart)
                if (c + tok < n && fc < p.n_out) {
                    uint4* chunk = reinterpret_cast<uint4*>(
                        stg + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4));
                    uint4 dq = *chunk;
                    const __nv_bfloat162* uh = reinterpret_cast<const __nv_bfloat162*>(&uq[j]);
                    __nv_bfloat162* dh = reinterpret_cast<__nv_bfloat162*>(&dq);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 uf = __bfloat1622float2(uh[i]);
                        const float2 df = __bfloat1622float2(dh[i]);
                        float2 gr;
                        if (p.spart != nullptr) {
                            float2 hg;
                            gr = gelu_and_grad2(uf, &hg);
                            part = fmaf(df.x, hg.x, fmaf(df.y, hg.y, part));
                        } else {
                            gr = gelu_grad2(uf);
                        }
                        dh[i] = __float22bfloat162_rn(__fmul2_rn(df, gr));
                    }
                    *chunk = dq;
                }
                if (p.spart != nullptr) {  // the token's two chunks: lanes 2t, 2t + 1
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    if (sh == 0 && c + tok < n && fr < p.n_out)
                        p.spart[(size_t)(r0 + c + tok) * ((p.n_out + 15) >> 4) + (fr >> 4)] = part;
                }
            }
        }
        const int rows_here = min(32, n - c);
        if (rows_here == 32 && fr < p.n_out) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::tma_store_2d(tm_out, stg, fr, r0 + c);
                tc::bulk_commit();
            }
            continue;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int ci = lane + 32 * j, tok = ci >> 1, sh = ci & 1;
            const int fc = fr + 8 * sh;
            if (c + tok < n && fc < p.n_out) {
                const uint4 val = *reinterpret_cast<const uint4*>(
                    stg + tok * 32 + ((sh ^ ((tok >> 2) & 1)) << 4));
                *reinterpret_cast<uint4*>(out + (size_t)(r0 + c + tok) * p.n_out + fc) = val;
            }
        }
        __syncwarp();
    }
}

// The GELU' operand of a first-GEMM-epilogue tile (Params::gelu_u) fetched
// into L2 by one epilogue warp ahead of its use: for each of the warp's
// items (as epilogue_gelu deals them), lane l takes token row l's 32 bytes.
template <int NPQ>
__device__ __forceinline__ void prefetch_gelu_u(const Params& p, int r0, int n, int fbase, int q,
                                                int wq, int lane) {
    const int items = 2 * ((n + 31) / 32);
    for (int it = wq; it < items; it += NPQ) {
        const int c = (it >> 1) * 32, fr = fbase + q * 32 + (it & 1) * 16;
        if (c + lane < n && fr < p.n_out)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(
                p.gelu_u + (size_t)(r0 + c + lane) * p.n_out + fr));
    }
}

// ===================================================================== CTA-pair kernel
// cta_group::2: a cluster of two CTAs (two SMs) computes a 256 x 256 tile
// D[f][j] (256 weight rows x up to 256 token rows) with one tcgen05.mma of
// M = 256 per K = 16 step.  CTA r holds weight rows 128r .. 128r+127 (its A)
// and token rows r*N/2 .. (r+1)*N/2-1 (its half of B) in its own shared
// memory, and rows 128r .. of the accumulator in its own TMEM.  Per SM and
// K-step this moves 16 KB of A and 16 KB of B (the single-CTA 128 x 256 tile
// moves 48 KB).  Each CTA fetches its operands as two whole boxes per K-step
// (128 x 64 each); rows past a segment's end belong to the next segment or
// read as zero, and the MMA's N covers only the segment's rows.  Only CTA 0
// issues MMAs; both CTAs' TMA copies signal CTA 0's full barrier, and CTA 0's
// commits arrive on both CTAs' barriers (multicast).  Both epilogues arrive
// on CTA 0's TMEM-empty barrier.
constexpr int BN2 = 256;  // tokens per pair tile (MMA N, max)

// The token operand of the CTA-pair kernel as four tensor maps whose boxes are
// 128, 64, 32 and 16 rows high (64 columns): each tile loads, per CTA, the
// smallest box that holds its half of the tile's rows, so a tile of few
// tokens (a small expert's segment, the end of a segment) does not move a
// whole 128-row box per K step.
struct BMaps {
    CUtensorMap m[4];
};

// A stage holds the ATOMS weight atoms (A_BYTES each) and then the ATOMS
// token atoms, each as many 128-byte rows as the tile's token box (at most
// BN2 / 2), packed one after another.
template <int STAGES, bool GEMM1, int EW, int ATOMS>
struct Cfg2 {
    static constexpr int THREADS = (4 + EW) * 32;       // 4 role warps + EW epilogue warps
    static constexpr int B_BYTES = (BN2 / 2) * BK * 2;  // 16 KB: this CTA's half of B per atom (max)
    static constexpr int STAGE_BYTES = ATOMS * (A_BYTES + B_BYTES);  // ATOMS x 64 columns of K
    static constexpr int OUT_ES = GEMM1 ? 2 : 4;
    static constexpr int STAGING = EW * 32 * 32 * OUT_ES;
    static constexpr int TMEM_COLS = 2 * BN2;
    static constexpr int OFF_STAGING = STAGES * STAGE_BYTES;
    static constexpr int OFF_BARS = OFF_STAGING + STAGING;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
    static constexpr int OFF_TILES = OFF_MISC + 16;
    static constexpr int SMEM = OFF_TILES + (kMaxExperts + 1) * 4 + 1023;
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// The CTA-pair token box for half_rows rows a CTA: the smallest of the 128-,
// 64-, 32- and 16-row boxes that holds them (index into BMaps).
__device__ __forceinline__ int pair_bsel_rows(int half_rows) {
    return half_rows <= 16 ? 3 : half_rows <= 32 ? 2 : half_rows <= 64 ? 1 : 0;
}

// Token rows of operand bytes one group of token tiles may hold (see
// decode_pair_tile): about half the 126 MB L2.
constexpr long long kGroupBytes = 64ll << 20;

// Pair tile t: expert e (binary search over the per-expert tile prefix),
// then token tile fastest and 256-row weight tile, so the token tiles that
// share a weight tile run at about the same time and re-read it from L2.
// When an expert's token operand (rows x K) is larger than kGroupBytes, its
// token tiles are taken in groups of GT that fit: within a group, token tile
// fastest, then weight tile, so a group's token rows stay in L2 while every
// weight tile passes over them (each weight tile is read once per group,
// each token row about once) instead of the token rows being read again by
// every wave of weight tiles.
// s_tiles[e] * mul is expert e's first tile (mul = 1: a table of tiles;
// mul = mt2: a table of token tiles, which both GEMMs of one layer share).
__device__ __forceinline__ Tile decode_pair_tile(int t, const int* s_tiles, const Params& p,
                                                 int mt2, int mul = 1) {
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {  // last expert whose first tile is <= t
        const int mid = (lo + hi + 1) >> 1;
        if (s_tiles[mid] * mul <= t) lo = mid; else hi = mid - 1;
    }
    int s0, s1;
    if (p.seg_maps != nullptr) {  // segment reduction: tok_rows output rows per expert
        s0 = lo * p.tok_rows;
        s1 = s0 + p.tok_rows;
    } else {
        s0 = min(max(__ldg(p.offsets + lo), 0), p.rows_cap);
        s1 = min(max(__ldg(p.offsets + lo + 1), s0), p.rows_cap);
    }
    const int nt = (s1 - s0 + BN2 - 1) / BN2;
    const int local = t - s_tiles[lo] * mul;
    int gt = nt;  // token tiles per group
    if (p.seg_maps == nullptr && (long long)nt * BN2 * p.K * 2 > kGroupBytes)
        gt = max(1, (int)(kGroupBytes / ((long long)BN2 * p.K * 2)));
    const int g = local / (gt * mt2);               // group (all but the last are full)
    const int gsize = min(gt, nt - g * gt);
    const int lg = local - g * gt * mt2;
    Tile tl;
    tl.e = lo;
    tl.r0 = s0 + (g * gt + lg % gsize) * BN2;
    tl.o0 = tl.r0;
    tl.n = min(BN2, s1 - tl.r0);
    tl.m0 = (lg / gsize) * 2 * BM;
    return tl;
}

// OPS, the operand forms and epilogue work (fixed at compile time, so the
// forward pass's kernels carry none of the backward pass's cases):
//   0  both operands K-major, the forward epilogues;
//   1  both K-major, the backward first-GEMM epilogue (Params::pre_out);
//   2  the weight operand MN-major (Params::a_mn), the backward first-GEMM
//      epilogue (Params::gelu_u, spart) or the second-GEMM one;
//   3  segment reduction, both operands MN-major (Params::seg_maps).
template <int STAGES, bool GEMM1, int EW, int ATOMS, int OPS>
__global__ void __launch_bounds__(Cfg2<STAGES, GEMM1, EW, ATOMS>::THREADS, 1)
grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ BMaps tmB,
                  const __grid_constant__ CUtensorMap tmO, const Params p) {
    using C = Cfg2<STAGES, GEMM1, EW, ATOMS>;
    constexpr bool kRed = OPS == 3, kAmn = OPS >= 2, kBwdEpi = OPS == 1 || OPS == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* s_tiles = reinterpret_cast<int*>(smem + C::OFF_TILES);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)tc::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
    const int mt2 = (p.n_out + 2 * BM - 1) / (2 * BM);  // 256-row weight tiles
    const int KB = (p.K + ATOMS * BK - 1) / (ATOMS * BK);  // stages per tile
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], 2 * EW);
        }
        tc::mbar_init(drain, 1);
        *s_abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA);
        for (int i = 0; i < 4; ++i) tc::tma_prefetch_desc(&tmB.m[i]);
    }
    if (warp == 2) {
        tc::tmem_alloc_pair(s_tmem, C::TMEM_COLS);
        tc::tmem_relinquish_pair();
    }
    pdl_wait();  // offsets and the operands come from the previous kernel
    pdl_trigger();
    if (warp == 3) {  // exclusive prefix of pair tiles per expert
        int run = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            int nt = 0;
            if (e < p.E) {
                const int rows_e = p.seg_maps != nullptr ? p.tok_rows : seg_rows(p, e);
                nt = ((rows_e + BN2 - 1) / BN2) * mt2;
            }
            int v = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (e < p.E) s_tiles[e] = run + v - nt;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_tiles[p.E] = run;
    }
    tc::fence_before_sync();
    tc::cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc::fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const int total = s_tiles[p.E];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            int last_e = -1;
            for (int t = pair; t < total && ok; t += npairs) {
                const Tile tl = decode_pair_tile(t, s_tiles, p, mt2);
                const int m0 = tl.m0;  // pair tile base row
                // segment reduction: both operands MN-major through the
                // segment's own maps, the whole 256-token MMA N (128 a CTA)
                constexpr bool red = kRed, amn = kAmn;
                const int half_rows = red ? BN2 / 2 : ((tl.n + 31) & ~31) / 2;
                // the smallest token box that holds this CTA's half_rows rows
                const int bsel = half_rows <= 16 ? 3 : half_rows <= 32 ? 2 : half_rows <= 64 ? 1 : 0;
                const CUtensorMap* ta = red ? p.seg_maps + 2 * tl.e : &tmA;
                const CUtensorMap* tb = red ? p.seg_maps + 2 * tl.e + 1 : &tmB.m[bsel];
                if (red && tl.e != last_e) {  // the maps were written by the previous kernel
                    tc::tensormap_acquire(ta);
                    tc::tensormap_acquire(tb);
                    last_e = tl.e;
                }
                const uint32_t bytes = 2 * ATOMS * (A_BYTES + (BN2 / 2 >> bsel) * BK * 2);
                const int batom = (BN2 / 2 >> bsel) * BK * 2;  // bytes of one token atom
                // K-major weight rows / MN-major weight columns of this CTA
                const int arow = (amn ? 0 : tl.e * p.n_out) + m0 + rank * BM;
                const int brow = (red ? tl.r0 - tl.e * p.tok_rows : tl.r0) + rank * half_rows;
                const int krow0 = red ? 0 : tl.e * p.K;  // MN-major: the expert's first K row
                const int KBt = red ? (seg_rows(p, tl.e) + ATOMS * BK - 1) / (ATOMS * BK) : KB;
                for (int kb = 0; kb < KBt; ++kb) {
                    if (!wait_bar(&empty[stage], phase ^ 1, s_abort, p, 1)) { ok = false; break; }
                    if (leader) tc::mbar_expect_tx(&full[stage], bytes);
                    const uint32_t full_l = tc::cluster_addr(&full[stage], 0);
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    uint8_t* sb = sa + ATOMS * A_BYTES;
                    const int kr = krow0 + kb * ATOMS * BK;  // MN-major: first K row of the stage
                    if (p.box3d) {  // one box per operand: 64 columns x rows x ATOMS atoms
                        const int kc = kb * ATOMS;
                        if (amn)  // 64 MN columns x 128 K rows x 2 column chunks
                            tc::tma_load_3d_pair(sa, ta, full_l, 0, kr, arow / BK);
                        else
                            tc::tma_load_3d_pair(sa, ta, full_l, 0, arow, kc);
                        if (red)
                            tc::tma_load_3d_pair(sb, tb, full_l, 0, kr, brow / BK);
                        else
                            tc::tma_load_3d_pair(sb, tb, full_l, 0, brow, kc);
                    } else {
#pragma unroll
                        for (int at = 0; at < ATOMS; ++at) {
                            const int kc = (kb * ATOMS + at) * BK;
                            if (amn)
                                tc::tma_load_2d_pair(sa + at * A_BYTES, ta, full_l, arow + at * BK, kr);
                            else
                                tc::tma_load_2d_pair(sa + at * A_BYTES, ta, full_l, kc, arow);
                            if (red)
                                tc::tma_load_2d_pair(sb + at * batom, tb, full_l, brow + at * BK, kr);
                            else
                                tc::tma_load_2d_pair(sb + at * batom, tb, full_l, kc, brow);
                        }
                    }
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            // the copies of fill i have landed once its stage was released
            const long long last = fills < STAGES ? fills : STAGES;
            for (long long i = fills - last; i < fills; ++i)
                drain_bar(&empty[i % STAGES], (uint32_t)((i / STAGES) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (CTA 0)
        if (lane == 0 && leader) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                const Tile tl = decode_pair_tile(t, s_tiles, p, mt2);
                constexpr bool red = kRed, amn = kAmn;  // red: both operands MN-major
                const uint32_t N = red ? (uint32_t)BN2 : (uint32_t)((tl.n + 31) & ~31);
                const uint32_t idesc = tc::idesc_bf16_f32(2 * BM, N) | (amn ? tc::kIdescAMn : 0u) |
                                       (red ? tc::kIdescBMn : 0u);
                const int half_rows = (int)N / 2;  // the producer's token box for this tile
                const int bsel = half_rows <= 16 ? 3 : half_rows <= 32 ? 2 : half_rows <= 64 ? 1 : 0;
                const uint32_t batom = (uint32_t)((BN2 / 2 >> bsel) * BK * 2);
                if (!wait_bar(&tempty[acc], acc_phase ^ 1, s_abort, p, 2)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN2);
                const int KBt = red ? (seg_rows(p, tl.e) + ATOMS * BK - 1) / (ATOMS * BK) : KB;
                for (int kb = 0; kb < KBt; ++kb) {
                    if (!wait_bar(&full[stage], phase, s_abort, p, 3)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t s0 = tc::smem_u32(smem + stage * C::STAGE_BYTES);
#pragma unroll
                    for (int at = 0; at < ATOMS; ++at) {
                        const uint32_t sa = s0 + at * A_BYTES;
                        const uint32_t sb = s0 + ATOMS * A_BYTES + at * batom;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            // MN-major: K step at * 4 + kk is 16 rows of 128 bytes
                            // into the first box; the second box (the next 64
                            // MN columns) lies A_BYTES / batom further on
                            const uint32_t kmn = (uint32_t)(at * (BK / 16) + kk) * 2048u;
                            const uint64_t ad = amn ? tc::sdesc_mn_sw128(s0 + kmn, A_BYTES)
                                                    : tc::sdesc_k128_sw128(sa + kk * 32);
                            const uint64_t bd =
                                red ? tc::sdesc_mn_sw128(s0 + ATOMS * A_BYTES + kmn, batom)
                                    : tc::sdesc_k128_sw128(sb + kk * 32);
                            tc::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | at | kk) != 0 ? 1u : 0u);
                        }
                    }
                    tc::mma_commit_pair_mc(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit_pair_mc(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            // every issued MMA completes before either CTA frees its TMEM
            tc::mma_commit_pair_mc(drain, 0x3);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int ew = warp - 4;
        const int q = warp & 3;
        const int part = ew >> 2;  // which of the EW/4 column parts of the tile
        uint8_t* stg = smem + C::OFF_STAGING + ew * 32 * 32 * C::OUT_ES;
        int acc = 0;
        uint32_t acc_phase = 0;
        if (GEMM1 && kBwdEpi && p.gelu_u != nullptr && pair < total) {
            const Tile t0 = decode_pair_tile(pair, s_tiles, p, mt2);
            prefetch_gelu_u<EW / 4>(p, t0.r0, t0.n, t0.m0 + rank * BM, q, part, lane);
        }
        for (int t = pair; t < total; t += npairs) {
            const Tile tl = decode_pair_tile(t, s_tiles, p, mt2);
            const int m0 = tl.m0;
            if (GEMM1 && kBwdEpi && p.gelu_u != nullptr && t + npairs < total) {  // next tile's U
                const Tile tn = decode_pair_tile(t + npairs, s_tiles, p, mt2);
                prefetch_gelu_u<EW / 4>(p, tn.r0, tn.n, tn.m0 + rank * BM, q, part, lane);
            }
            const bool ok = wait_bar(&tfull[acc], acc_phase, s_abort, p, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            if constexpr (GEMM1 && kBwdEpi)
                epilogue_gelu_bwd<EW / 4>(p, tl.e, tl.r0, tl.n, m0 + rank * BM, tmem_base,
                                          acc * BN2, q, part, lane, stg, &tmO);
            else if constexpr (GEMM1)
                epilogue_gelu<EW / 4>(p, tl.e, tl.r0, tl.n, m0 + rank * BM, tmem_base, acc * BN2,
                                      q, part, lane, stg, &tmO);
            else
                epilogue_tile<BN2, GEMM1, kRed>(p, tl.e, tl.r0, tl.r0, tl.n, m0 + rank * BM,
                                                tmem_base, acc * BN2, q, part, EW / 4, lane, stg,
                                                &tmO,
                                                p.seg_maps != nullptr && seg_rows(p, tl.e) == 0);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster_relaxed(tc::cluster_addr(&tempty[acc], 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    if (warp >= 4 && lane == 0) tc::bulk_wait_all();  // the output is written before exit
    if (warp == 1 && lane == 0) drain_bar(drain, 0);
    tc::fence_before_sync();
    tc::cluster_sync();  // no cross-CTA arrive or MMA write is still pending
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------
// The expert FFN's two GEMMs in one persistent launch of CTA pairs.
//
// Work items: every first-GEMM tile (h = GELU(x_perm W1^T + b1)), then every
// second-GEMM tile (y_perm = (h W2^T + b2) w), dealt round robin to the CTA
// pairs.  When the second GEMM's w = tiles / pairs waves end better in half
// tiles (2w / ceil(2w) > w / ceil(w) + 0.05) its K is split in two: the first
// halves come before all second halves, a first half stores (acc + b2) w and
// the second adds acc w once ksync[tile] counts the first half's 16 epilogue
// warps (a fixed order, so the result repeats bit for bit).  A pair that runs out of first-GEMM tiles
// goes on to second-GEMM tiles while the others finish theirs, where two
// launches make the whole second GEMM wait for the slowest pair's last
// first-GEMM tile and for the launch boundary.  A second-GEMM tile reads the
// h rows of one 256-token tile: its producer waits until every first-GEMM
// tile of those rows has counted its 32 epilogue warps (2 CTAs x 16) in
// ready[token tile], each after its h stores completed.  Every pair takes its
// items in increasing order and all first-GEMM items come before all
// second-GEMM items, so a wait is only ever on items that wait on nothing.
//
// 16 epilogue warps: all of them run a first-GEMM tile's GELU epilogue (2 KB
// of staging each), the first 8 a second-GEMM tile's epilogue (4 KB each, TMA
// stores of fp32 y_perm, as in the second-GEMM kernel).  The two layouts
// overlap, so before its first second-GEMM tile each warp waits until all 16
// have finished staging first-GEMM output (a bounded barrier; items come in
// the same order to every warp, and all first-GEMM items come first).
struct FfnPair {
    Params g1, g2;   // g1: n_out = d_ff, K = d, GELU, bf16 h; g2: n_out = d, K = d_ff
    int32_t* ready;  // [ready_cap] first-GEMM arrivals per token tile, zero at launch
    int ready_cap;
};

// One work item of the fused kernel.
struct FfnItem {
    Tile tl;
    int g;   // 0: first GEMM, 1: second
    int kh;  // second GEMM split in K: 0 first half (or whole), 1 second half
    int tb;  // the whole tile's index within its GEMM
    int tt;  // token tile (index of its ready counter)
};

__device__ __forceinline__ FfnItem decode_ffn_item(int t, int n1, int n2, const int* s_tt,
                                                   const FfnPair& f, int mt1, int mt2) {
    FfnItem it;
    if (t < n1) {
        it.g = 0;
        it.kh = 0;
        it.tb = t;
        it.tl = decode_pair_tile(t, s_tt, f.g1, mt1, mt1);
    } else {
        const int u = t - n1;
        it.g = 1;
        it.kh = u >= n2 ? 1 : 0;
        it.tb = u - it.kh * n2;
        it.tl = decode_pair_tile(it.tb, s_tt, f.g2, mt2, mt2);
    }
    const int s0 = min(max(__ldg(f.g1.offsets + it.tl.e), 0), f.g1.rows_cap);
    it.tt = s_tt[it.tl.e] + (it.tl.r0 - s0) / BN2;
    return it;
}

// Publish this warp's output of a finished item: its tensor stores complete,
// its plain stores fenced, then one count.
__device__ __forceinline__ void publish_count(int32_t* cnt, int lane) {
    if (lane == 0) {
        tc::bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        atomicAdd(cnt, 1);
    }
}

template <int STAGES, int ATOMS>
__global__ void __launch_bounds__(Cfg2<STAGES, true, 16, ATOMS>::THREADS, 1)
ffn_pair_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ BMaps tmB1,
                const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ BMaps tmB2, const __grid_constant__ CUtensorMap tmO2,
                const FfnPair f) {
    constexpr int EW = 16, EW2 = 8;  // epilogue warps of a first / second-GEMM tile
    using C = Cfg2<STAGES, true, EW, ATOMS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* s_split = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
    int* s_tt = reinterpret_cast<int*>(smem + C::OFF_TILES);  // token-tile prefix per expert
    __shared__ uint64_t s_xfer;  // the epilogue warps' hand-over of the staging memory
    const Params& P = f.g1;      // time-out and error record

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)tc::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
    const int mt1 = (f.g1.n_out + 2 * BM - 1) / (2 * BM), mt2 = (f.g2.n_out + 2 * BM - 1) / (2 * BM);
    const int KB1 = (f.g1.K + ATOMS * BK - 1) / (ATOMS * BK);
    const int KB2 = (f.g2.K + ATOMS * BK - 1) / (ATOMS * BK);
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], 2 * EW);
        }
        tc::mbar_init(drain, 1);
        tc::mbar_init(&s_xfer, EW);
        *s_abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA1);
        tc::tma_prefetch_desc(&tmA2);
        for (int i = 0; i < 4; ++i) {
            tc::tma_prefetch_desc(&tmB1.m[i]);
            tc::tma_prefetch_desc(&tmB2.m[i]);
        }
    }
    if (warp == 2) {
        tc::tmem_alloc_pair(s_tmem, C::TMEM_COLS);
        tc::tmem_relinquish_pair();
    }
    pdl_wait();  // offsets and x_perm come from the previous kernel
    pdl_trigger();
    if (warp == 3) {  // exclusive prefix of token tiles per expert
        int run = 0;
        for (int e0 = 0; e0 < f.g1.E; e0 += 32) {
            const int e = e0 + lane;
            const int nt = e < f.g1.E ? (seg_rows(f.g1, e) + BN2 - 1) / BN2 : 0;
            int v = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (e < f.g1.E) s_tt[e] = run + v - nt;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            s_tt[f.g1.E] = run;
            // the second GEMM's split in K (see above)
            const int n2 = run * mt2;
            int split = 0;
            if (n2 > 0 && n2 <= f.g2.ksync_cap && f.g2.K % (2 * ATOMS * BK) == 0) {
                const float w = (float)n2 / (float)npairs;
                split = 2.0f * w / ceilf(2.0f * w) > w / ceilf(w) + 0.05f;
            }
            *s_split = split;
        }
    }
    tc::fence_before_sync();
    tc::cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc::fence_after_sync();
    const uint32_t tmem_base = *s_tmem;
    const int TT = s_tt[f.g1.E];
    const int n1 = TT * mt1, n2 = TT * mt2;
    const int split = *s_split;
    const int total = n1 + (n2 << split);
    const int KB2h = KB2 >> split;
    const int ready_target = mt1 * 2 * EW;  // arrivals of a token tile's first-GEMM items

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                const FfnItem it = decode_ffn_item(t, n1, n2, s_tt, f, mt1, mt2);
                const Params& p = it.g ? f.g2 : f.g1;
                const CUtensorMap* tA = it.g ? &tmA2 : &tmA1;
                if (it.g == 1) {  // the h rows of this token tile are complete
                    if (it.tt >= f.ready_cap ||
                        !wait_count(f.ready + it.tt, ready_target, s_abort, P, 7)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const int m0 = it.tl.m0;
                const int half_rows = ((it.tl.n + 31) & ~31) / 2;
                const int bsel = pair_bsel_rows(half_rows);
                const CUtensorMap* tb = it.g ? &tmB2.m[bsel] : &tmB1.m[bsel];
                const uint32_t bytes = 2 * ATOMS * (A_BYTES + (BN2 / 2 >> bsel) * BK * 2);
                const int batom = (BN2 / 2 >> bsel) * BK * 2;
                const int arow = it.tl.e * p.n_out + m0 + rank * BM;
                const int brow = it.tl.r0 + rank * half_rows;
                const int KBt = it.g ? KB2h : KB1;
                const int k0 = it.kh * KB2h * ATOMS * BK;
                for (int kb = 0; kb < KBt; ++kb) {
                    if (!wait_bar(&empty[stage], phase ^ 1, s_abort, P, 1)) { ok = false; break; }
                    if (leader) tc::mbar_expect_tx(&full[stage], bytes);
                    const uint32_t full_l = tc::cluster_addr(&full[stage], 0);
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    uint8_t* sb = sa + ATOMS * A_BYTES;
                    if (p.box3d) {
                        const int kc = k0 / BK + kb * ATOMS;
                        tc::tma_load_3d_pair(sa, tA, full_l, 0, arow, kc);
                        tc::tma_load_3d_pair(sb, tb, full_l, 0, brow, kc);
                    } else {
#pragma unroll
                        for (int at = 0; at < ATOMS; ++at) {
                            const int kc = k0 + (kb * ATOMS + at) * BK;
                            tc::tma_load_2d_pair(sa + at * A_BYTES, tA, full_l, kc, arow);
                            tc::tma_load_2d_pair(sb + at * batom, tb, full_l, kc, brow);
                        }
                    }
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            const long long last = fills < STAGES ? fills : STAGES;
            for (long long i = fills - last; i < fills; ++i)
                drain_bar(&empty[i % STAGES], (uint32_t)((i / STAGES) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (CTA 0)
        if (lane == 0 && leader) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                const FfnItem it = decode_ffn_item(t, n1, n2, s_tt, f, mt1, mt2);
                const uint32_t N = (uint32_t)((it.tl.n + 31) & ~31);
                const uint32_t idesc = tc::idesc_bf16_f32(2 * BM, N);
                const int bsel = pair_bsel_rows((int)N / 2);
                const uint32_t batom = (uint32_t)((BN2 / 2 >> bsel) * BK * 2);
                if (!wait_bar(&tempty[acc], acc_phase ^ 1, s_abort, P, 2)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN2);
                const int KBt = it.g ? KB2h : KB1;
                for (int kb = 0; kb < KBt; ++kb) {
                    if (!wait_bar(&full[stage], phase, s_abort, P, 3)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t s0 = tc::smem_u32(smem + stage * C::STAGE_BYTES);
#pragma unroll
                    for (int at = 0; at < ATOMS; ++at) {
                        const uint32_t sa = s0 + at * A_BYTES;
                        const uint32_t sb = s0 + ATOMS * A_BYTES + at * batom;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            tc::mma_bf16_pair(d_tmem, tc::sdesc_k128_sw128(sa + kk * 32),
                                              tc::sdesc_k128_sw128(sb + kk * 32), idesc,
                                              (kb | at | kk) != 0 ? 1u : 0u);
                    }
                    tc::mma_commit_pair_mc(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit_pair_mc(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            tc::mma_commit_pair_mc(drain, 0x3);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int ew = warp - 4;
        const int q = warp & 3;
        const int part = ew >> 2;  // which of the column parts of the tile
        uint8_t* stg1 = smem + C::OFF_STAGING + ew * 32 * 32 * 2;
        uint8_t* stg2 = smem + C::OFF_STAGING + ew * 32 * 32 * 4;
        static_assert(EW2 * 32 * 32 * 4 <= C::STAGING, "second-GEMM staging");
        int acc = 0;
        uint32_t acc_phase = 0;
        bool staged2 = false;  // this warp has handed over to second-GEMM staging
        for (int t = pair; t < total; t += npairs) {
            const FfnItem it = decode_ffn_item(t, n1, n2, s_tt, f, mt1, mt2);
            const int fb = it.tl.m0 + rank * BM;
            if (it.g == 1 && !staged2) {
                // this warp's first-GEMM tensor stores have read its staging rows;
                // once all 16 warps say so the second-GEMM layout may be written
                if (lane == 0) {
                    tc::bulk_wait_read_all();
                    tc::mbar_arrive(&s_xfer);
                }
                __syncwarp();
                const bool okx = wait_bar_idle(&s_xfer, 0, s_abort, P, 8);
                if (!__all_sync(0xffffffffu, okx)) break;
                staged2 = true;
            }
            const bool ok = wait_bar_idle(&tfull[acc], acc_phase, s_abort, P, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            if (it.kh == 1 && ew < EW2) {  // the first K half of this tile is in y_perm
                bool okw = true;
                if (lane == 0) okw = wait_count(f.g2.ksync + it.tb, 2 * EW2, s_abort, P, 5);
                if (!__all_sync(0xffffffffu, __shfl_sync(0xffffffffu, okw, 0))) break;
                (void)ld_acquire_gpu(f.g2.ksync + it.tb);  // every lane acquires
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            if (it.g == 0)
                epilogue_gelu<EW / 4>(f.g1, it.tl.e, it.tl.r0, it.tl.n, fb, tmem_base, acc * BN2,
                                      q, part, lane, stg1, &tmO1);
            else if (ew < EW2)
                epilogue_tile<BN2, false>(f.g2, it.tl.e, it.tl.r0, it.tl.r0, it.tl.n, fb,
                                          tmem_base, acc * BN2, q, part, EW2 / 4, lane, stg2,
                                          &tmO2, false, it.kh == 1);
            // the accumulator is read: hand it back before waiting on the stores
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster_relaxed(tc::cluster_addr(&tempty[acc], 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
            if (it.g == 0) {
                if (it.tt < f.ready_cap) publish_count(f.ready + it.tt, lane);
            } else if (split && it.kh == 0 && ew < EW2) {
                publish_count(f.g2.ksync + it.tb, lane);
            }
        }
    }

    if (warp >= 4 && lane == 0) tc::bulk_wait_all();  // the output is written before exit
    if (warp == 1 && lane == 0) drain_bar(drain, 0);
    tc::fence_before_sync();
    tc::cluster_sync();  // no cross-CTA arrive or MMA write is still pending
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// One bounded pipeline wait on a barrier nothing arrives on: gives up after
// timeout_ns and records the time-out (where = 900) like a stalled pipeline.
__global__ void __launch_bounds__(32) wait_timeout_probe(DeviceHeader* hdr, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
    Params p{};
    p.hdr = hdr;
    p.timeout_ns = timeout_ns;
    wait_bar(&bar, 0, &abort_flag, p, 900);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major bf16 matrix [outer][inner] as a 2-D TMA map with 128-byte swizzle
// and boxes of box_outer rows x 64 columns; out-of-range elements read as 0.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_outer) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four token-operand maps of the CTA-pair kernel (BMaps).
bool make_b_maps(BMaps* m, const void* base, uint64_t inner, uint64_t outer) {
    for (int i = 0; i < 4; ++i)
        if (!make_map(&m->m[i], base, inner, outer, (uint32_t)(BN2 / 2) >> i)) return false;
    return true;
}

// Row-major bf16 matrix [outer][inner] (inner a multiple of 64) viewed in 3-D
// as [inner / 64][outer][64]: the innermost dimension is 64 columns (one
// 128-byte swizzle row), the next the rows, the outermost the 64-column
// chunks of K.  A box of 64 x box_outer x atoms then lands in shared memory as
// `atoms` consecutive 128-byte-swizzled [box_outer][64] tiles - the layout two
// (or more) 2-D boxes would give - in one TMA operation, which halves the box
// count per stage (the TMA issue rate per SM, not bytes, bounds a stage of
// 16 KB boxes).  Chunks past the end read as zero, like columns past K.
bool make_map3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
               uint32_t box_outer, uint32_t atoms) {
    auto fn = encode_fn();
    if (fn == nullptr || inner % BK != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)BK, outer, inner / BK};
    cuuint64_t strides[2] = {inner * 2, (cuuint64_t)BK * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, box_outer, atoms};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kPairAtoms = 2;  // K atoms per stage of the CTA-pair kernel

// The fused expert FFN (ffn_pair_kernel) for layers whose GEMMs are at most
// this many multiply-adds (T k d d_ff; upper bound on the kept rows).  A/B
// on one B300, expert FFN alone (uniform segments, L2 flushed), fused vs two
// launches: (T k, d, d_ff) = (8192, 1024, 4096) 114.7 vs 118.8 us; (16384,
// 2048, 8192) 682 vs 682 us; (16384, 4096, 14336) 2.30 vs 2.26 ms; (32768,
// 4096, 14336) 5.46-5.71 vs 5.46-5.57 ms.  In the full layer the Switch
// layer (32768 x 2048 x 8192 = 2^39) went from 334 to 327 us.
constexpr double kFusedFfnMaxWork = 549755813888.0;  // 2^39

// The CTA-pair kernel's operand maps: 3-D (one box per operand and stage)
// when K is a multiple of 64 and the driver takes the 3-D view, else 2-D.
// Returns the Params::box3d value.
bool make_pair_maps(CUtensorMap* a, const void* W, uint64_t K, uint64_t w_rows, BMaps* b,
                    const void* T, uint64_t t_rows, int* box3d) {
    bool ok3 = K % BK == 0 && make_map3(a, W, K, w_rows, BM, kPairAtoms);
    for (int i = 0; ok3 && i < 4; ++i)
        ok3 = make_map3(&b->m[i], T, K, t_rows, (uint32_t)(BN2 / 2) >> i, kPairAtoms);
    if (ok3) {
        *box3d = 1;
        return true;
    }
    *box3d = 0;
    return make_map(a, W, K, w_rows, BM) && make_b_maps(b, T, K, t_rows);
}

// Row-major bf16 matrix [outer][inner] as the destination of 16 x 32 tensor
// stores from staging rows in the 32-byte swizzle.
bool make_store_map_sw32(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major fp32 matrix [outer][inner] as the destination of 32 x 32 tensor
// stores (no swizzle: the staging rows are plain 128-byte rows).
bool make_store_map_f32(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of CS CTAs that can be resident at once (one CTA per SM).
template <auto Kern>
int resident_clusters(int cs, int smem, int threads = kThreads) {
    static int cache[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = num_sms() / cs;
    if (cs > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * n, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = cs;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int q = 0;
        if (cudaOccupancyMaxActiveClusters(&q, Kern, &cfg) == cudaSuccess && q > 0 && q < n) n = q;
        cudaGetLastError();
    }
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

template <int BN_MAX, int STAGES, bool GEMM1>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                       cudaStream_t s) {
    using C = Cfg<BN_MAX, STAGES, GEMM1>;
    constexpr auto kern = grouped_gemm_tc<BN_MAX, STAGES, GEMM1>;
    cudaError_t err = ensure_smem<kern>(C::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(num_sms()), dim3(kThreads), C::SMEM, s, 1, true, a, b, p);
}

template <int STAGES, bool GEMM1, int EW, int ATOMS, int OPS = 0>
cudaError_t launch_one_pair(const CUtensorMap& a, const BMaps& b, const CUtensorMap& o,
                            const Params& p, cudaStream_t s) {
    using C = Cfg2<STAGES, GEMM1, EW, ATOMS>;
    constexpr auto kern = grouped_gemm_pair<STAGES, GEMM1, EW, ATOMS, OPS>;
    cudaError_t err = ensure_smem<kern>(C::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(2 * resident_clusters<kern>(2, C::SMEM, C::THREADS)),
                         dim3(C::THREADS), C::SMEM, s, 2, true, a, b, o, p);
}

template <int STAGES, int ATOMS>
cudaError_t launch_ffn_pair(const CUtensorMap& a1, const BMaps& b1, const CUtensorMap& o1,
                            const CUtensorMap& a2, const BMaps& b2, const CUtensorMap& o2,
                            const FfnPair& f, cudaStream_t s) {
    using C = Cfg2<STAGES, true, 16, ATOMS>;
    constexpr auto kern = ffn_pair_kernel<STAGES, ATOMS>;
    cudaError_t err = ensure_smem<kern>(C::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(2 * resident_clusters<kern>(2, C::SMEM, C::THREADS)),
                         dim3(C::THREADS), C::SMEM, s, 2, true, a1, b1, o1, a2, b2, o2, f);
}

template <int BN_MAX, int STAGES>
cudaError_t launch_pair(const CUtensorMap* maps, const Params& p1, const Params& p2,
                        cudaStream_t s) {
    cudaError_t err = launch_one<BN_MAX, STAGES, true>(maps[0], maps[1], p1, s);
    if (err != cudaSuccess) return err;
    return launch_one<BN_MAX, STAGES, false>(maps[2], maps[3], p2, s);
}

}  // namespace

uint64_t g_tc_timeout_ns = 2000000000ull;

cudaError_t launch_wait_timeout_probe(DeviceHeader* hdr, uint64_t timeout_ns, cudaStream_t s) {
    wait_timeout_probe<<<1, 32, 0, s>>>(hdr, timeout_ns);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_expert_ffn_tc(const moe_config& c, const void* x_perm, int64_t x_rows,
                                 const int32_t* offsets, const void* W1, const void* b1,
                                 const void* W2, const void* b2, const float* perm_w,
                                 float* y_perm, void* h, int64_t h_rows, DeviceHeader* hdr,
                                 int32_t* ksync, int32_t* ready, cudaStream_t s) {
    if (h_rows == 0) return cudaSuccess;
    // tokens per expert on average decides the widest token tile
    const bool wide = (int64_t)c.T * c.k >= 96LL * c.E;
    CUtensorMap maps[4];
    const uint32_t box_w = BM, box_x = BOX_ROWS;
    if (!make_map(&maps[0], W1, c.d, (uint64_t)c.E * c.d_ff, box_w) ||
        !make_map(&maps[1], x_perm, c.d, (uint64_t)x_rows, box_x) ||
        !make_map(&maps[2], W2, c.d_ff, (uint64_t)c.E * c.d, box_w) ||
        !make_map(&maps[3], h, c.d_ff, (uint64_t)h_rows, box_x))
        return cudaErrorInvalidValue;
    Params p1{offsets, reinterpret_cast<const __nv_bfloat16*>(b1), nullptr, h, hdr,
              g_tc_timeout_ns, c.E, c.d_ff, c.d, (int)h_rows, 1, nullptr, 0};
    Params p2{offsets, reinterpret_cast<const __nv_bfloat16*>(b2), perm_w, y_perm, hdr,
              g_tc_timeout_ns, c.E, c.d, c.d_ff, (int)h_rows, 0, nullptr, 0};
    if (wide) {
        // operand maps for the pair kernel; h and y_perm as store targets
        CUtensorMap a1, a2, so[2];
        BMaps bx, bh;
        if (!make_pair_maps(&a1, W1, c.d, (uint64_t)c.E * c.d_ff, &bx, x_perm, (uint64_t)x_rows,
                            &p1.box3d) ||
            !make_pair_maps(&a2, W2, c.d_ff, (uint64_t)c.E * c.d, &bh, h, (uint64_t)h_rows,
                            &p2.box3d) ||
            !make_store_map_sw32(&so[0], h, c.d_ff, (uint64_t)h_rows) ||
            !make_store_map_f32(&so[1], y_perm, c.d, (uint64_t)h_rows))
            return cudaErrorInvalidValue;
        // Layers up to kFusedFfnMaxWork multiply-adds a GEMM run both GEMMs in
        // one launch (its counters, ready and ksync, are zero); larger ones as
        // two launches, where the boundary is a small share of the time.
        if ((double)c.T * c.k * c.d * c.d_ff <= kFusedFfnMaxWork) {
            p2.ksync = ksync;
            p2.ksync_cap = kKsyncCap;
            const FfnPair f{p1, p2, ready, ready_tiles(h_rows, c.E)};
            return launch_ffn_pair<3, kPairAtoms>(a1, bx, so[0], a2, bh, so[1], f, s);
        }
        cudaError_t err = launch_one_pair<3, true, 16, kPairAtoms>(a1, bx, so[0], p1, s);
        if (err != cudaSuccess) return err;
        return launch_one_pair<3, false, 8, kPairAtoms>(a2, bh, so[1], p2, s);
    }
    return launch_pair<64, 8>(maps, p1, p2, s);
}

// Both GEMMs of the dense decode FFN in one persistent launch
// (dense_ffn_kernel).  sched: 1 + E int32 in the workspace, zero at launch.
cudaError_t launch_dense_ffn(const moe_config& c, const void* x, const void* W1, const void* b1,
                             const void* W2, const void* b2, void* h_all, float* y_all,
                             int32_t* sched, DeviceHeader* hdr, cudaStream_t s) {
    CUtensorMap a1, bx, a2, bh;
    if (!make_map(&a1, W1, c.d, (uint64_t)c.E * c.d_ff, BM) ||
        !make_map(&bx, x, c.d, (uint64_t)c.T, BOX_ROWS) ||
        !make_map(&a2, W2, c.d_ff, (uint64_t)c.E * c.d, BM) ||
        !make_map(&bh, h_all, c.d_ff, (uint64_t)c.E * c.T, BOX_ROWS))
        return cudaErrorInvalidValue;
    DenseFfn f;
    f.g1 = Params{nullptr, reinterpret_cast<const __nv_bfloat16*>(b1), nullptr, h_all, hdr,
                  g_tc_timeout_ns, c.E, c.d_ff, c.d, c.E * c.T, 1, nullptr, 0};
    f.g2 = Params{nullptr, reinterpret_cast<const __nv_bfloat16*>(b2), nullptr, y_all, hdr,
                  g_tc_timeout_ns, c.E, c.d, c.d_ff, c.E * c.T, 0, nullptr, 0};
    f.sched = sched;
    f.T = c.T;
    f.mt1 = (c.d_ff + BM - 1) / BM;
    f.mt2 = (c.d + BM - 1) / BM;
    f.n1 = c.E * f.mt1;
    f.n2 = c.E * f.mt2;
    constexpr auto kern = dense_ffn_kernel;
    cudaError_t err = ensure_smem<kern>(DenseCfg::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(num_sms()), dim3(kThreads), DenseCfg::SMEM, s, 1, true, a1, bx,
                         a2, bh, f);
}

// One grouped GEMM out[r][n] = sum_k A[r][k] W_e[n][k] (+ bias_e[n]) over the
// expert segments of A (the forward pass's kernels, for the backward pass):
// bf16_out: bf16 out, optional GELU (act), and with pre_out also the
// pre-activation (Params::pre_out; CTA-pair kernel); else fp32 out times
// row_w[r] (row_w null: 1).  A: [a_rows][K] bf16, W: [E][n_out][K] bf16, out:
// [out_rows][n_out].  `wide` picks the CTA-pair kernel (as the forward does).
cudaError_t launch_grouped_gemm_tc(const moe_config& c, bool bf16_out, bool act, const void* A,
                                   int64_t a_rows, const int32_t* offsets, const void* W,
                                   const void* bias, const float* row_w, void* out,
                                   int64_t out_rows, int n_out, int K, DeviceHeader* hdr,
                                   cudaStream_t s, void* pre_out) {
    if (out_rows == 0) return cudaSuccess;
    if (pre_out != nullptr && !bf16_out) return cudaErrorInvalidValue;
    // (the pre-activation output is a CTA-pair kernel epilogue mode)
    const bool wide = (int64_t)c.T * c.k >= 96LL * c.E || pre_out != nullptr;
    Params p{offsets, reinterpret_cast<const __nv_bfloat16*>(bias), bf16_out ? nullptr : row_w,
             out, hdr, g_tc_timeout_ns, c.E, n_out, K, (int)out_rows, act ? 1 : 0, nullptr, 0};
    p.pre_out = static_cast<__nv_bfloat16*>(pre_out);
    CUtensorMap mw;
    if (wide) {
        BMaps ma;
        CUtensorMap mo;
        if (!make_pair_maps(&mw, W, (uint64_t)K, (uint64_t)c.E * n_out, &ma, A, (uint64_t)a_rows,
                            &p.box3d))
            return cudaErrorInvalidValue;
        if (bf16_out) {
            if (!make_store_map_sw32(&mo, out, (uint64_t)n_out, (uint64_t)out_rows))
                return cudaErrorInvalidValue;
            return pre_out != nullptr
                       ? launch_one_pair<3, true, 16, kPairAtoms, 1>(mw, ma, mo, p, s)
                       : launch_one_pair<3, true, 16, kPairAtoms>(mw, ma, mo, p, s);
        }
        if (!make_store_map_f32(&mo, out, (uint64_t)n_out, (uint64_t)out_rows))
            return cudaErrorInvalidValue;
        return launch_one_pair<3, false, 8, kPairAtoms>(mw, ma, mo, p, s);
    }
    if (!make_map(&mw, W, (uint64_t)K, (uint64_t)c.E * n_out, BM)) return cudaErrorInvalidValue;
    CUtensorMap ma;
    if (!make_map(&ma, A, (uint64_t)K, (uint64_t)a_rows, BOX_ROWS)) return cudaErrorInvalidValue;
    return bf16_out ? launch_one<64, 8, true>(mw, ma, p, s) : launch_one<64, 8, false>(mw, ma, p, s);
}

// One grouped GEMM out[r][n] = sum_k A[r][k] W[e][k][n] over the expert
// segments of A with the weight stored K rows by n_out columns, W [E][K][n_out]
// (the backward pass's dH = dY_perm W2 and dX_perm = dU W1 read W2 [E][d][d_ff]
// and W1 [E][d_ff][d] as they are): the CTA-pair kernel with its weight
// operand read MN-major.  bf16_out: bf16 out (no bias), times GELU'(gelu_u)
// when gelu_u is not null (Params::gelu_u), with the partial dots spart
// ([out_rows][ceil(n_out / 16)]) when that is not null; else fp32.
cudaError_t launch_grouped_gemm_mn(const moe_config& c, bool bf16_out, const void* A,
                                   int64_t a_rows, const int32_t* offsets, const void* W,
                                   const void* gelu_u, float* spart, void* out, int64_t out_rows,
                                   int n_out, int K, DeviceHeader* hdr, cudaStream_t s) {
    if (out_rows == 0) return cudaSuccess;
    if ((gelu_u != nullptr && !bf16_out) || (spart != nullptr && gelu_u == nullptr))
        return cudaErrorInvalidValue;
    Params p{offsets, nullptr, nullptr, out, hdr, g_tc_timeout_ns, c.E, n_out, K, (int)out_rows,
             0, nullptr, 0};
    p.a_mn = 1;
    p.gelu_u = static_cast<const __nv_bfloat16*>(gelu_u);
    p.spart = spart;
    CUtensorMap mw, mo;
    BMaps ma;
    const uint64_t w_rows = (uint64_t)c.E * K;
    // 3-D boxes when both the weight's n_out and the tokens' K allow them
    bool ok = n_out % BK == 0 && K % BK == 0 &&
              make_map3(&mw, W, (uint64_t)n_out, w_rows, kPairAtoms * BK, kPairAtoms);
    for (int i = 0; ok && i < 4; ++i)
        ok = make_map3(&ma.m[i], A, (uint64_t)K, (uint64_t)a_rows, (uint32_t)(BN2 / 2) >> i,
                       kPairAtoms);
    p.box3d = ok ? 1 : 0;
    if (!ok && !(make_map(&mw, W, (uint64_t)n_out, w_rows, kPairAtoms * BK) &&
                 make_b_maps(&ma, A, (uint64_t)K, (uint64_t)a_rows)))
        return cudaErrorInvalidValue;
    if (bf16_out) {
        if (!make_store_map_sw32(&mo, out, (uint64_t)n_out, (uint64_t)out_rows))
            return cudaErrorInvalidValue;
        return launch_one_pair<3, true, 16, kPairAtoms, 2>(mw, ma, mo, p, s);
    }
    if (!make_store_map_f32(&mo, out, (uint64_t)n_out, (uint64_t)out_rows))
        return cudaErrorInvalidValue;
    return launch_one_pair<3, false, 8, kPairAtoms, 2>(mw, ma, mo, p, s);
}

namespace {

// Tensor maps of a row-major bf16 [rows][inner] buffer read MN-major by the
// segment reduction: boxes of 64 columns x 128 rows (a stage's K), in the
// 3-D view (two column chunks a box) when inner is a multiple of 64.
bool make_seg_template(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                       bool box3d) {
    return box3d ? make_map3(m, base, inner, rows, kPairAtoms * BK, kPairAtoms)
                 : make_map(m, base, inner, rows, kPairAtoms * BK);
}

// For each expert e, out[2e] (WT) and out[2e + 1] (TOK): copies of the
// whole-buffer maps whose base is the segment's first row and whose row
// extent is the segment's length, so that a box reaching past the segment's
// end reads zeros there instead of the next segment's rows.
__global__ void __launch_bounds__(128) seg_maps_kernel(
    const __grid_constant__ CUtensorMap wt, const __grid_constant__ CUtensorMap tok,
    const int32_t* __restrict__ offsets, int E, int rows_cap, const uint8_t* wt_base,
    int64_t wt_row_bytes, const uint8_t* tok_base, int64_t tok_row_bytes, CUtensorMap* out) {
    pdl_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) {
        const int s0 = min(max(__ldg(offsets + e), 0), rows_cap);
        const int s1 = min(max(__ldg(offsets + e + 1), s0), rows_cap);
        const int n = max(s1 - s0, 1);  // (an empty segment's maps are never read)
        const CUtensorMap* src[2] = {&wt, &tok};
        const uint8_t* base[2] = {wt_base + s0 * wt_row_bytes, tok_base + s0 * tok_row_bytes};
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            CUtensorMap* m = out + 2 * e + o;
            const uint4* from = reinterpret_cast<const uint4*>(src[o]);
            uint4* to = reinterpret_cast<uint4*>(m);
#pragma unroll
            for (int i = 0; i < (int)(sizeof(CUtensorMap) / sizeof(uint4)); ++i) to[i] = from[i];
            tc::tensormap_set_address(m, base[o]);
            tc::tensormap_set_dim1(m, n);
        }
        tc::tensormap_release();
    }
    pdl_trigger();
}

cudaError_t launch_seg_maps(const CUtensorMap& wt, const CUtensorMap& tok, const int32_t* offsets,
                            int E, int64_t rows_cap, const void* WT, int n_out, const void* TOK,
                            int tok_rows, CUtensorMap* maps, cudaStream_t s) {
    return launch_kernel(seg_maps_kernel, dim3((E + 127) / 128), dim3(128), 0, s, 1, true, wt, tok,
                         offsets, E, (int)rows_cap, static_cast<const uint8_t*>(WT),
                         (int64_t)n_out * 2, static_cast<const uint8_t*>(TOK),
                         (int64_t)tok_rows * 2, maps);
}

}  // namespace

// Segment reduction on the CTA-pair kernel (see Params::seg_maps): out fp32
// [E*tok_rows][n_out] = per expert TOK_e^T WT_e over the segment's rows, TOK
// [rows_cap][tok_rows] and WT [rows_cap][n_out] bf16 row-major over the
// permuted rows.  maps: 2E tensor maps of workspace (128-byte aligned),
// written here by seg_maps_kernel and read by the GEMM.
cudaError_t launch_segment_reduction_tc(int E, const int32_t* offsets, int64_t rows_cap,
                                        const void* TOK, int tok_rows, const void* WT, int n_out,
                                        float* out, CUtensorMap* maps, DeviceHeader* hdr,
                                        cudaStream_t s) {
    Params p{offsets, nullptr, nullptr, out, hdr, g_tc_timeout_ns, E, n_out, 0, (int)rows_cap, 0,
             maps, tok_rows};
    const bool box3d = n_out % BK == 0 && tok_rows % BK == 0;
    CUtensorMap mw, mt, mo;
    if (!make_seg_template(&mw, WT, (uint64_t)n_out, (uint64_t)rows_cap, box3d) ||
        !make_seg_template(&mt, TOK, (uint64_t)tok_rows, (uint64_t)rows_cap, box3d) ||
        !make_store_map_f32(&mo, out, (uint64_t)n_out, (uint64_t)E * tok_rows))
        return cudaErrorInvalidValue;
    p.box3d = box3d ? 1 : 0;
    cudaError_t err = launch_seg_maps(mw, mt, offsets, E, rows_cap, WT, n_out, TOK, tok_rows,
                                      maps, s);
    if (err != cudaSuccess) return err;
    BMaps mb;  // (the kernel loads through the segment maps in this mode)
    for (int i = 0; i < 4; ++i) mb.m[i] = mt;
    return launch_one_pair<3, false, 8, kPairAtoms, 3>(mw, mb, mo, p, s);
}

// The device-side map edits of launch_segment_reduction_tc checked against
// the driver's own encoding (moe_check_segment_maps).
moe_status check_segment_maps(void* ws, size_t ws_bytes, cudaStream_t s) {
    constexpr int E = 3;
    constexpr size_t kMaps = 256;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < kSegMapCheckBytes) return MOE_ERR_WORKSPACE;
    const int32_t offs[E + 1] = {0, 37, 37, 301};  // a ragged, an empty and a long segment
    const int64_t rows_cap = 320;
    uint8_t* base = static_cast<uint8_t*>(ws);
    int32_t* d_offs = reinterpret_cast<int32_t*>(base);
    CUtensorMap* d_maps = reinterpret_cast<CUtensorMap*>(base + kMaps);
    // buffers that are never read (no copy runs): WT [rows][192], TOK [rows][136]
    const void* WT = base + (1 << 20);
    const void* TOK = base + (2 << 20);
    const int n_out = 192, tok_rows = 136;
    for (int v = 0; v < 2; ++v) {  // the 3-D and the 2-D views
        const bool box3d = v == 0;
        const int tr = box3d ? 128 : tok_rows;  // the 3-D view wants multiples of 64
        CUtensorMap mw, mt;
        if (!make_seg_template(&mw, WT, n_out, rows_cap, box3d) ||
            !make_seg_template(&mt, TOK, tr, rows_cap, box3d))
            return MOE_ERR_CUDA;
        if (cudaMemcpyAsync(d_offs, offs, sizeof(offs), cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemsetAsync(d_maps, 0, 2 * E * sizeof(CUtensorMap), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        chain_begin();  // the launch follows a memset: no programmatic overlap
        if (launch_seg_maps(mw, mt, d_offs, E, rows_cap, WT, n_out, TOK, tr, d_maps, s) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        CUtensorMap got[2 * E];
        if (cudaMemcpyAsync(got, d_maps, sizeof(got), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return MOE_ERR_CUDA;
        for (int e = 0; e < E; ++e) {
            const int n = offs[e + 1] - offs[e] > 0 ? offs[e + 1] - offs[e] : 1;
            CUtensorMap want[2];
            if (!make_seg_template(&want[0], static_cast<const uint8_t*>(WT) + offs[e] * n_out * 2,
                                   n_out, n, box3d) ||
                !make_seg_template(&want[1], static_cast<const uint8_t*>(TOK) + offs[e] * tr * 2,
                                   tr, n, box3d))
                return MOE_ERR_CUDA;
            for (int o = 0; o < 2; ++o) {
                if (memcmp(&want[o], &got[2 * e + o], sizeof(CUtensorMap)) == 0) continue;
                const uint8_t* w = reinterpret_cast<const uint8_t*>(&want[o]);
                const uint8_t* g = reinterpret_cast<const uint8_t*>(&got[2 * e + o]);
                fprintf(stderr, "segment map %d.%d (%s view) differs at bytes:", e, o,
                        box3d ? "3-D" : "2-D");
                for (int b = 0; b < (int)sizeof(CUtensorMap); ++b)
                    if (w[b] != g[b]) fprintf(stderr, " %d (%02x, edited %02x)", b, w[b], g[b]);
                fprintf(stderr, "\n");
                return MOE_ERR_UNSUPPORTED;
            }
        }
    }
    return MOE_OK;
}

}  // namespace moe
