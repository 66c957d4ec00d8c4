// moe_dispatch_noalloc: moe_dispatch with its scratch memory in a fixed
// device array owned by the library instead of a caller-provided workspace.
//
// Some callers cannot hand the library a workspace: a host program whose GPU
// memory is carved up once at start-up by another component (a serving
// engine's fixed pool, a plugin host that owns every allocation) has no
// allocator to call, and must not trigger one behind its back.  For them the
// dispatch step - the only part of the layer whose scratch is small and
// bounded by the batch - can run on this statically sized array.
//
// The array lives in this file as a __device__ variable, so every GPU that
// loads the library holds it until the process exits.  Host code cannot use
// its name as a device address; the device address is looked up with
// cudaGetSymbolAddress once per device (on the first call made while that
// device is current) and passed to the kernels.

#include <cuda_runtime.h>

#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// Scratch bound: T * k <= kNoAllocMaxAssignments and E <= kMaxExperts.
constexpr int kNoAllocMaxAssignments = 65536;
constexpr int kNoAllocMaxBlocks = kNoAllocMaxAssignments / kCountBlock;  // 256
constexpr size_t kHistBytes = sizeof(int32_t) * (size_t)kNoAllocMaxBlocks * kMaxExperts;
constexpr size_t kScratchBytes = sizeof(DeviceHeader) + 2 * kHistBytes +
                                 sizeof(int32_t) * (size_t)kNoAllocMaxAssignments;  // 768.25 KB

static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once
// per device), or null if the lookup failed.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* x,
                                           const int32_t* topk_idx, const float* topk_w,
                                           int32_t* offsets, int32_t* slot_of,
                                           int32_t* perm_token, float* perm_w, void* x_perm,
                                           void* stream) {
    const moe_status cs = config_status(cfg);
    if (cs != MOE_OK) return cs;
    const moe_config& c = *cfg;
    if (c.routing != MOE_TOKEN_CHOICE || c.overflow != MOE_DROP)
        return MOE_ERR_UNSUPPORTED;  // a token-choice step that drops on overflow
    if (c.T < 0 || c.d <= 0 || c.d_ff <= 0 || c.E <= 0 || c.k <= 0 ||
        (c.dtype != MOE_F32 && c.dtype != MOE_BF16) || (c.renormalize != 0 && c.renormalize != 1) ||
        c.n_shared < 0 || c.n_shared >= c.E || c.k > c.E - c.n_shared)
        return MOE_ERR_INVALID_ARG;
    if (c.E > kMaxExperts || c.k + c.n_shared > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (c.d % 8 != 0 || c.d_ff % 8 != 0) return MOE_ERR_ALIGNMENT;
    const moe_config cd = dispatch_config(c);  // K = k + n_shared assignments per token
    if ((int64_t)cd.T * cd.k > kNoAllocMaxAssignments) return MOE_ERR_UNSUPPORTED;  // scratch bound
    if (offsets == nullptr) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c.T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), s) == cudaSuccess
                             ? MOE_OK : MOE_ERR_CUDA;
    if (x == nullptr || topk_idx == nullptr || slot_of == nullptr || perm_token == nullptr ||
        x_perm == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (perm_w != nullptr && topk_w == nullptr) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(x_perm) & 15u) != 0)
        return MOE_ERR_ALIGNMENT;

    void* scratch = scratch_for_current_device();
    if (scratch == nullptr) return MOE_ERR_CUDA;
    // The scratch regions the dispatch kernels use, laid out in the array.
    WsLayout L = ws_layout(c);
    L.header = 0;
    L.blk_hist = sizeof(DeviceHeader);
    L.blk_base = L.blk_hist + kHistBytes;
    L.local_rank = L.blk_base + kHistBytes;
    // The error record must start at zero; the kernels overwrite everything
    // else they read.
    if (cudaMemsetAsync(scratch, 0, sizeof(DeviceHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
    chain_begin();  // the first kernel follows the memset
    cudaError_t e = launch_count(cd, topk_idx, scratch, L, s);
    if (e == cudaSuccess)
        e = launch_scan_permute(cd, x, topk_idx, topk_w, kCountBlock, L.count_blocks, offsets,
                                slot_of, perm_token, perm_w, x_perm, scratch, L, LossArgs{}, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
