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
// cudaGetSymbolAddress once per CUDA context (on the first call made while
// that context is current) and passed to the kernels.  A module symbol's
// address belongs to a context, not to a device ordinal: a host that creates
// its own driver-API contexts, switches between several on one device, or
// resets the device (which replaces the primary context) gets a lookup of its
// own, keyed on the context's process-unique ID.

#include <cuda.h>
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

// Symbol addresses already looked up, keyed on the context's unique ID (a
// context that is destroyed never has its ID reused).  Sixteen entries; the
// oldest is replaced when a seventeenth context calls.
constexpr int kCacheEntries = 16;
struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
};
ScratchEntry g_scratch_cache[kCacheEntries] = {};
int g_scratch_next = 0;
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(ptr);
}

// ID of the calling thread's current context, or 0 if there is none or the
// driver does not say.
unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current context, or null if the
// lookup failed.  Looked up once per context; without a context ID (no
// context current yet: the lookup itself makes the device's primary context
// current) the result is cached under the ID of the context the lookup left
// current.
void* scratch_for_current_context() {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = current_context_id();
    if (id != 0)
        for (const ScratchEntry& en : g_scratch_cache)
            if (en.ctx_id == id) return en.ptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (id == 0) id = current_context_id();
    if (id != 0) {
        g_scratch_cache[g_scratch_next] = ScratchEntry{id, p};
        g_scratch_next = (g_scratch_next + 1) % kCacheEntries;
    }
    return p;
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

    void* scratch = scratch_for_current_context();
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
