// ar_noalloc.cu -- ar_residual_rmsnorm_noalloc: the two-shot fused call with
// its scratch (one fp32 sum of squares per row chunk) in an array that the
// library itself holds in device memory, for callers that may not allocate.
//
// The array is a file-scope __device__ variable: every device that loads the
// library gets its own copy when the library's code is loaded there, and
// keeps it until the process exits.  On the host, `g_scratch` names only a
// host-side stand-in for that symbol, never a device address, so it is never
// handed to a kernel.  The device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached here.
#include <cuda_runtime.h>

#include <mutex>

#include "ar.h"

namespace {

constexpr size_t kScratchFloats = AR_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch per device, null until looked up

// Device address of the scratch array on the current device (looked up on
// the first call for that device).
int scratch_on_current_device(void** addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return AR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return AR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return AR_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
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
