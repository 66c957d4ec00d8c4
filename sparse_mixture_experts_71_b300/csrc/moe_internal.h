// Internal declarations shared by the kernels and the C-ABI layer of libmoe.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
// assignments covered by one block of the counting kernel
constexpr int kCountBlock = 256;

// Device error record at the start of every workspace.
struct DeviceHeader {
    int32_t err_code;   // first error recorded (0 = none)
    int32_t err_info;
    uint32_t route_done;  // blocks of the route kernel that finished (reset per call)
    int32_t pad[61];
};
static_assert(sizeof(DeviceHeader) == 256, "header is one 256-byte line");

enum DeviceError : int32_t { kErrExpertRange = 1, kErrTimeout = 2 };

// Byte offsets of the workspace regions for one configuration.
struct WsLayout {
    size_t header;       // DeviceHeader
    size_t counts;       // int32 [E]   assignments per expert (all slots)
    size_t top1;         // int32 [E]   first-slot choices per expert
    size_t blk_p;        // fp32 [route_blocks][E] per-block sums of p
    size_t blk_hist;     // int32 [count_blocks][E]
    size_t blk_base;     // int32 [count_blocks][E]
    size_t local_rank;   // int32 [T*k]
    size_t topk_idx;     // int32 [T*k]     (moe_forward)
    size_t topk_w;       // fp32  [T*k]     (moe_forward)
    size_t offsets;      // int32 [E+1]     (moe_forward)
    size_t slot_of;      // int32 [T*k]     (moe_forward)
    size_t perm_token;   // int32 [T*k]     (moe_forward)
    size_t perm_w;       // fp32  [T*k]     (moe_forward)
    size_t x_perm;       // dtype [rows][d] (moe_forward)
    size_t h;            // dtype [rows][d_ff]
    size_t y_perm;       // fp32  [rows][d] (moe_forward)
    size_t total;
    int route_blocks;
    int count_blocks;
    int64_t rows;        // upper bound of kept assignments
};

WsLayout ws_layout(const moe_config& c);
int route_tokens_per_block(int E);

// Kernel launches enqueued so far (moe_launch_count).
void count_launches(int n);

template <typename T> __host__ __device__ inline T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(base) + off);
}

// ---- launchers (kernels live in route.cu, dispatch.cu, gemm_simt.cu, combine.cu)
cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r,
                         const float* logit_bias, const float* logits_in, float* logits_out,
                         int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                         float* aux_out, void* ws, const WsLayout& L, cudaStream_t s);

cudaError_t launch_dispatch(const moe_config& c, const void* x, const int32_t* topk_idx,
                            const float* topk_w, int32_t* offsets, int32_t* slot_of,
                            int32_t* perm_token, float* perm_w, void* x_perm, void* ws,
                            const WsLayout& L, cudaStream_t s);

cudaError_t launch_expert_ffn(const moe_config& c, const void* x_perm, int64_t x_rows,
                              const int32_t* offsets, const void* W1, const void* b1,
                              const void* W2, const void* b2, const float* perm_w, float* y_perm,
                              void* ws, const WsLayout& L, cudaStream_t s);

cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* slot_of,
                           void* y, cudaStream_t s);

}  // namespace moe
