// ar_noalloc.cu -- ar_residual_rmsnorm_noalloc: the two-shot fused call with
// its scratch (one fp32 sum of squares per row chunk) in an array that the
// library itself holds in device memory, for callers that may not allocate.
//
// The array is a file-scope __device__ variable: every device that loads the
// library gets its own copy when the library's code is loaded into a context
// there, and keeps it until the context is destroyed (at process exit, or by
// cudaDeviceReset).  On the host, `g_scratch` names only a host-side stand-in
// for that symbol, never a device address, so it is never handed to a kernel.
// The device address is looked up with cudaGetSymbolAddress (with the device
// current) and cached per device together with the id of the context it was
// looked up in; a call from another context (after a device reset, or under a
// context the caller made current) looks it up again, so a cached address
// never outlives the context that holds the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ar.h"

namespace {

constexpr size_t kScratchFloats = AR_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

struct ScratchEntry {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void* addr;                 // device address of g_scratch in that context
};

std::mutex g_mutex;
ScratchEntry g_scratch_cache[kMaxDevices];

// The driver's cuCtxGetCurrent and cuCtxGetId, reached through the runtime
// (the library links the static runtime only, not libcuda).
using CtxGetCurrentFn = CUresult(CUDAAPI*)(CUcontext*);
using CtxGetIdFn = CUresult(CUDAAPI*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Id of the calling thread's current context: unique among all contexts the
// process creates, so a context created after a reset never repeats it.
// 0 when no context is current yet.  Called with g_mutex held.
bool current_context_id(unsigned long long* id)
{
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || f1 == nullptr || f2 == nullptr)
            return false;
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS)
        return false;
    *id = 0;
    return ctx == nullptr || g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current
// context, looked up on the first call from that context.
int scratch_on_current_device(void** addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return AR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return AR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx))
        return AR_ERR_CUDA;
    ScratchEntry& e = g_scratch_cache[dev];
    if (ctx == 0 || e.ctx_id != ctx || e.addr == nullptr) {
        // The look-up makes the runtime's context current if none was yet.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return AR_ERR_CUDA;
        if (ctx == 0 && !current_context_id(&ctx))
            return AR_ERR_CUDA;
        e.ctx_id = ctx;
        e.addr = p;
    }
    *addr = e.addr;
    return AR_OK;
}

}  // namespace

extern "C" int ar_residual_rmsnorm_noalloc(const void* const* partials, int R, const void* bias,
                                           const void* residual, const void* weight, float eps,
                                           int hidden, int tokens, void* out, void* residual_out,
                                           int dtype, ar_stream_t stream)
{
    // Shapes whose scratch could exceed the array are refused before the
    // device is touched.  ar_workspace_size_rows is the bound for either
    // path (packed or element-wise); it is 0 for shapes the fused call
    // itself rejects, which then fail its own checks below.
    if (tokens > 0 && ar_workspace_size_rows(R, hidden, tokens, dtype) > AR_NOALLOC_SCRATCH_BYTES)
        return AR_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (int st = scratch_on_current_device(&scratch))
        return st;
    // Phase 1 of the two-shot path writes every (row, chunk) entry that
    // phase 2 then reads, so what an earlier call left in the array is never
    // read and nothing needs clearing.
    return ar_residual_rmsnorm(partials, R, bias, residual, weight, eps, hidden, tokens, out, residual_out,
                               scratch, AR_NOALLOC_SCRATCH_BYTES, dtype, AR_TWOSHOT, stream);
}
