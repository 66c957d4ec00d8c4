// Router logits on the 5th-generation tensor cores (tcgen05 + TMEM, TMA-fed)
// for bf16 token batches, followed by the same softmax / top-k / statistics
// as the other router kernels.
//
// "Mixture of Experts: Scaling Parameters Without Scaling Compute", section
// "The MoE layer", step 1: g = W_r x, p = softmax(g).
//
// Each CTA owns 128 tokens (the MMA's M).  W_r (fp32) is split beforehand
// into three bf16 parts hi + mid + lo that add up to W_r exactly; the three
// MMAs of a K = 16 step accumulate x.hi^T + x.mid^T + x.lo^T into one fp32
// TMEM accumulator of NP columns (NP = E rounded up), so every product is
// exact and only the fp32 accumulation rounds.  Warp 0 streams 64-column
// slices of x (128 x 64) and of the three parts (one 3 NP x 64 box: the
// parts are consecutive rows of one tensor) into a 2-deep ring, with the
// x slices prefetched into L2 a few stages ahead; warp 1 issues the MMAs; warps 4-7 read the accumulator back
// (TMEM lane = token) into shared memory.  Then one thread per token does the
// softmax and top-k, and the block finishes like the other router kernels.
// A small batch (too few 128-token tiles to fill the SMs) splits each tile's
// K over a cluster of 2 or 4 CTAs: each accumulates its share of the
// 64-column slices, rank 0 adds the other ranks' partial logits from their
// shared memory (in rank order, so the sum repeats bit for bit) and
// finishes the tile.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>

#include "route_common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace rt;

constexpr int TM = 128;                  // tokens per CTA
constexpr int RBK = 64;                  // K per stage
constexpr int RA_BYTES = TM * RBK * 2;   // 16 KB
// Two stages, and the logits tile reuses the ring once the MMAs are done, so
// two CTAs fit on an SM: a batch of T / 128 CTAs then runs in one wave on the
// 148 SMs (T = 32768: 256 CTAs) instead of 1.7 waves of one CTA per SM, with
// the same bytes in flight per SM.
constexpr int RSTAGES = 2;
constexpr uint64_t kRouteTimeoutNs = 2000000000ull;
// Stages of x prefetched into L2 ahead of the loads (measured on the Switch
// batch: 4 -> 3 us less than none; 8 and 16 slower).
constexpr int kXPrefetch = 4;

template <int NP>
struct RCfg {
    static constexpr int PART_BYTES = NP * RBK * 2;
    static constexpr int STAGE_BYTES = RA_BYTES + 3 * PART_BYTES;
    static constexpr int LDS = NP + 1;
    static constexpr int OFF_P = 0;  // logits tile [TM][LDS] fp32, over the stage ring
    static constexpr int RING = RSTAGES * STAGE_BYTES;
    static constexpr int P_BYTES = ((TM * LDS * 4 + 1023) / 1024) * 1024;
    static constexpr int OFF_BARS = RING > P_BYTES ? RING : P_BYTES;
    static constexpr int NUM_BARS = 2 * RSTAGES + 2;
    static constexpr int SMEM = OFF_BARS + NUM_BARS * 8 + 1023;
    static constexpr int TMEM_COLS = NP < 32 ? 32 : NP;
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(2 * (SMEM + 8192) <= 233472, "two CTAs per SM");
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              DeviceHeader* hdr, int where) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (tc::globaltimer() - t0 > kRouteTimeoutNs) {
            *abort_flag = 1;
            record_error(hdr, kErrTimeout, 100 + where);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity))
        if (tc::globaltimer() - t0 > kRouteTimeoutNs) break;
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 2)
route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                RouteArgs a, int ks) {
    using C = RCfg<NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* s_p = reinterpret_cast<float*>(smem + C::OFF_P);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* empty = full + RSTAGES;
    uint64_t* tfull = empty + RSTAGES;
    uint64_t* drain = tfull + 1;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_idx[TM * kMaxTopK];
    __shared__ int s_cnt[NP], s_top1[NP], carry[NP];
    __shared__ int wh[kWarps][NP];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // ks > 1: a cluster of ks CTAs shares the tile, each summing its share of
    // K; rank 0 adds the others' partial logits and finishes the tile
    const int rank = ks > 1 ? (int)tc::cluster_ctarank() : 0;
    const int tile = blockIdx.x / ks;
    const int t0 = tile * TM;
    const int KB = (a.d + RBK - 1) / RBK;
    const int kb0 = rank * KB / ks, kb1 = (rank + 1) * KB / ks;  // this CTA's K steps
    const bool gemm = a.logits_in == nullptr;

    if (tid < NP) { s_cnt[tid] = 0; s_top1[tid] = 0; }
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < RSTAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(tfull, 1);
        tc::mbar_init(drain, 1);
        s_abort = 0;
        tc::fence_barrier_init();
        if (gemm) {
            tc::tma_prefetch_desc(&tmX);
            tc::tma_prefetch_desc(&tmW);
            // x is the caller's input, written before this call's first
            // kernel started: its first slices can head for L2 while the
            // previous kernel (the router-weight split) finishes
            for (int j = kb0; j < kb0 + kXPrefetch && j < kb1; ++j)
                tc::tma_prefetch_l2_2d(&tmX, j * RBK, t0);
        }
    }
    if (warp == 2) {
        tc::tmem_alloc(&s_tmem, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem_base = s_tmem;
    volatile int* abort_flag = &s_abort;

    if (!gemm) {
        for (int i = tid; i < TM * NP; i += kThreads) {
            const int tok = i / NP, e = i % NP;
            const int t = t0 + tok;
            s_p[tok * C::LDS + e] =
                (t < a.T && e < a.E) ? __ldg(a.logits_in + (size_t)t * a.E + e) : 0.f;
        }
    } else if (warp == 0) {
        if (lane == 0) {  // ---------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int fills = 0;
            // x is read once: its boxes go to L2 kXPrefetch stages ahead of
            // their loads, so more of the batch is in flight than the ring
            // holds (the first ones before the programmatic wait, above)
            for (int kb = kb0; kb < kb1; ++kb) {
                if (kb + kXPrefetch < kb1) tc::tma_prefetch_l2_2d(&tmX, (kb + kXPrefetch) * RBK, t0);
                if (!wait_or_abort(&empty[stage], phase ^ 1, abort_flag, a.hdr, 1)) break;
                tc::mbar_expect_tx(&full[stage], C::STAGE_BYTES);
                uint8_t* sa = smem + stage * C::STAGE_BYTES;
                tc::tma_load_2d(sa, &tmX, &full[stage], kb * RBK, t0);
                // the three parts are consecutive rows of one tensor: one box
                tc::tma_load_2d(sa + RA_BYTES, &tmW, &full[stage], kb * RBK, 0);
                ++fills;
                if (++stage == RSTAGES) { stage = 0; phase ^= 1; }
            }
            const int last = fills < RSTAGES ? fills : RSTAGES;
            for (int i = fills - last; i < fills; ++i)
                drain_wait(&full[i % RSTAGES], (uint32_t)((i / RSTAGES) & 1));
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------------------------------- MMA issuer
            const uint32_t idesc = tc::idesc_bf16_f32(TM, NP);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1 && ok; ++kb) {
                if (!wait_or_abort(&full[stage], phase, abort_flag, a.hdr, 2)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t sa = tc::smem_u32(smem + stage * C::STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < RBK / 16; ++kk)
#pragma unroll
                    for (int part = 0; part < 3; ++part)
                        tc::mma_bf16(tmem_base, tc::sdesc_k128_sw128(sa + kk * 32),
                                     tc::sdesc_k128_sw128(sa + RA_BYTES + part * C::PART_BYTES +
                                                          kk * 32),
                                     idesc, (kb != kb0 || kk != 0 || part != 0) ? 1u : 0u);
                tc::mma_commit(&empty[stage]);
                if (++stage == RSTAGES) { stage = 0; phase ^= 1; }
            }
            if (ok) tc::mma_commit(tfull);
            tc::mma_commit(drain);
            drain_wait(drain, 0);
        }
    } else if (warp >= 4) {  // ------------------------------------ accumulator -> smem
        // s_p overlays the stage ring: written only after tfull, when every
        // TMA fill has been consumed by the MMAs
        const int q = warp & 3;
        const int tok = q * 32 + lane;
        const bool ok = wait_or_abort(tfull, 0, abort_flag, a.hdr, 3);
        if (__all_sync(0xffffffffu, ok)) {
            tc::fence_after_sync();
#pragma unroll
            for (int c0 = 0; c0 < NP; c0 += 32) {
                float v[32];
                tc::tmem_ld_32cols(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int e = c0 + j;
                    if (e < NP) {
                        float g = v[j];
                        if (a.bias != nullptr && e < a.E && rank == 0) g += __ldg(a.bias + e);
                        s_p[tok * C::LDS + e] = g;
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (ks > 1) {
        tc::cluster_sync();  // every rank's partial logits are in its shared memory
        if (rank == 0) {
            // 8 elements a round: their remote loads are all issued before the
            // adds wait on any of them
            uint32_t rbase[3];
#pragma unroll
            for (int r = 1; r < 4; ++r) rbase[r - 1] = r < ks ? tc::cluster_addr(s_p, (uint32_t)r) : 0u;
            constexpr int PER = TM * NP / kThreads;
            static_assert(PER % 8 == 0, "8-element rounds");
#pragma unroll 1
            for (int j0 = 0; j0 < PER; j0 += 8) {
                int off[8];
                float part[3][8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int i = tid + (j0 + q) * kThreads;
                    off[q] = (i / NP) * C::LDS + i % NP;
                }
#pragma unroll
                for (int r = 1; r < 4; ++r)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        part[r - 1][q] = r < ks ? tc::ld_shared_cluster_f32(rbase[r - 1] + 4u * off[q])
                                                : 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float acc = s_p[off[q]];
#pragma unroll
                    for (int r = 1; r < 4; ++r)  // fixed order: rank 0 + 1 + 2 + 3
                        if (r < ks) acc += part[r - 1][q];
                    s_p[off[q]] = acc;
                }
            }
        }
        tc::cluster_sync();  // rank 0 has read the partials: the others leave
        if (rank != 0) return;
    }
    stage_logits<NP>(a, s_p, C::LDS, TM, t0);
    __syncthreads();
    if constexpr (NP == 64) {  // two threads per token (all 256)
        static_assert(kThreads == 2 * TM, "a thread pair per token");
        token_epilogue_pair<NP>(a, s_p + (tid >> 1) * C::LDS, t0 + (tid >> 1), tid >> 1, tid & 1,
                                s_idx, s_cnt, s_top1);
    } else if (tid < TM) {
        token_epilogue<NP>(a, s_p + tid * C::LDS, t0 + tid, tid, s_idx, s_cnt, s_top1);
    }
    __syncthreads();
    finish_block<NP>(a, s_p, C::LDS, TM, s_idx, s_cnt, s_top1, wh, carry, tile);
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

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_outer) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)RBK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NP>
cudaError_t launch_np(const RouteArgs& a, const __nv_bfloat16* wsplit, cudaStream_t s) {
    using C = RCfg<NP>;
    CUtensorMap mx, mw;
    if (a.logits_in == nullptr) {
        if (!make_map(&mx, a.x, (uint64_t)a.d, (uint64_t)a.T, TM) ||
            !make_map(&mw, wsplit, (uint64_t)a.d, (uint64_t)3 * NP, 3 * NP))
            return cudaErrorInvalidValue;
    } else {
        memset(&mx, 0, sizeof(mx));
        memset(&mw, 0, sizeof(mw));
    }
    // few tiles (a small batch): split K over a cluster of 2 or 4 CTAs per
    // tile while all the CTAs still fit one per SM, at least 4 K steps each
    int ks = 1;
    const int KB = (a.d + RBK - 1) / RBK;
    while (a.logits_in == nullptr && ks < 4 && (int64_t)a.nblk * (2 * ks) <= num_sms() &&
           KB >= 4 * (2 * ks))
        ks *= 2;
    constexpr auto kern = route_tc_kernel<NP>;
    cudaError_t err = ensure_smem<kern>(C::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(a.nblk * ks), dim3(kThreads), C::SMEM, s, ks, true, mx, mw, a,
                         ks);
}

}  // namespace

namespace rt {
cudaError_t launch_route_tc(const RouteArgs& a, const __nv_bfloat16* wsplit, int np,
                            cudaStream_t s) {
    if (np <= 16) return launch_np<16>(a, wsplit, s);
    if (np <= 32) return launch_np<32>(a, wsplit, s);
    return launch_np<64>(a, wsplit, s);
}
}  // namespace rt

}  // namespace moe
