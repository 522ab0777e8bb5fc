// ar_host.cu -- ar_residual_rmsnorm_host: the fused call on tensors that live
// in host memory, with the host<->device copies pipelined against the
// kernels.  Host code only; it calls the public entry points of ar_api.cu.
//
// The rows are cut into chunks of `chunk_tokens` rows.  Chunk i goes through
// three stages on three streams, in a ring of kBuffers device staging buffers:
//   copy-in stream   R partial chunks + the residual chunk, host -> device
//   caller's stream  ar_residual_rmsnorm on the staged chunk
//   copy-out stream  out and residual_out chunks, device -> host
// so chunk i+1 is copied in while chunk i is computed and chunk i-1 copied
// out.  The last chunk_tokens rows (or fewer) go in shrinking pieces, halves
// until at most 2 x kMinTailRows rows are left, so that what runs after the
// last copy in (the drain: a piece's kernel and its copy out) is a small
// piece's, not a whole chunk's.  Events order each buffer's reuse after its
// previous copy-out.  Work
// queued on the caller's stream before the call is ordered before every copy
// of the call, and work queued after the call sees the outputs in host memory.
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "ar.h"

namespace {

constexpr int kBuffers = 2;      // staging buffers in the ring
constexpr int kMinTailRows = 64; // pieces of the shrinking tail stop halving at 2x this
constexpr int kMaxDevices = 64;

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int esize_of(int dtype)
{
    switch (dtype) {
    case AR_FP32: return 4;
    case AR_FP16: return 2;
    case AR_BF16: return 2;
    default: return 0;
    }
}

// Helper streams and events of one device, made on first use and kept for
// the life of the process.
struct Pipeline {
    bool ready = false;
    cudaStream_t copy_in = nullptr;
    cudaStream_t copy_out = nullptr;
    cudaEvent_t entry = nullptr;                 // the caller's stream reached the call
    cudaEvent_t staged[kBuffers] = {};           // inputs of the buffer's chunk are on the device
    cudaEvent_t computed[kBuffers] = {};         // the buffer's chunk is computed
    cudaEvent_t drained[kBuffers] = {};          // the buffer's outputs are back on the host
    cudaEvent_t consts = nullptr;                // weight and bias are on the device
};

std::mutex g_mutex;  // one call issues its work at a time (the events are shared)
Pipeline g_pipe[kMaxDevices];

int pipeline_of_current_device(Pipeline** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return AR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return AR_ERR_UNSUPPORTED;
    Pipeline& p = g_pipe[dev];
    if (!p.ready) {
        const unsigned fl = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&p.copy_in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.copy_out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.entry, fl) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.consts, fl) == cudaSuccess;
        for (int b = 0; ok && b < kBuffers; ++b)
            ok = cudaEventCreateWithFlags(&p.staged[b], fl) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.computed[b], fl) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.drained[b], fl) == cudaSuccess;
        if (!ok)
            return AR_ERR_CUDA;
        p.ready = true;
    }
    *out = &p;
    return AR_OK;
}

// Byte offsets of one staging buffer's parts (each 256-byte aligned).
struct Layout {
    size_t chunk_bytes;  // one [chunk_tokens, hidden] tensor
    size_t ws_bytes;     // two-shot workspace of one chunk
    size_t buffer;       // one buffer: R partials, residual, out, residual_out, workspace
    size_t consts;       // weight then bias, after the buffers
    size_t total;
};

Layout layout_of(int R, int hidden, int chunk_tokens, int dtype)
{
    Layout L{};
    const size_t row = static_cast<size_t>(hidden) * esize_of(dtype);
    L.chunk_bytes = round256(row * static_cast<size_t>(chunk_tokens));
    L.ws_bytes = round256(ar_workspace_size_rows(R, hidden, chunk_tokens, dtype));
    L.buffer = static_cast<size_t>(R + 3) * L.chunk_bytes + L.ws_bytes;
    L.consts = kBuffers * L.buffer;
    L.total = L.consts + 2 * round256(row);
    return L;
}

}  // namespace

extern "C" size_t ar_host_staging_size(int R, int hidden, int chunk_tokens, int dtype)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || chunk_tokens < 1 || esize_of(dtype) == 0)
        return 0;
    return layout_of(R, hidden, chunk_tokens, dtype).total;
}

extern "C" int ar_residual_rmsnorm_host(const void* const* partials, int R, const void* bias,
                                        const void* residual, const void* weight, float eps, int hidden,
                                        int tokens, void* out, void* residual_out, void* staging,
                                        size_t staging_bytes, int chunk_tokens, int dtype, int strategy,
                                        ar_stream_t stream)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0 || chunk_tokens < 1)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (tokens == 0)
        return AR_OK;
    if (partials == nullptr || residual == nullptr || weight == nullptr || out == nullptr ||
        residual_out == nullptr || staging == nullptr || out == residual_out)
        return AR_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        if (partials[r] == nullptr)
            return AR_ERR_INVALID_ARG;
    if (chunk_tokens > tokens)
        chunk_tokens = tokens;
    const Layout L = layout_of(R, hidden, chunk_tokens, dtype);
    if (staging_bytes < L.total || (reinterpret_cast<uintptr_t>(staging) & 255u) != 0)
        return AR_ERR_WORKSPACE;

    std::lock_guard<std::mutex> lock(g_mutex);
    Pipeline* P = nullptr;
    if (int st = pipeline_of_current_device(&P))
        return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(staging);
    const size_t row = static_cast<size_t>(hidden) * esize;
    void* d_weight = base + L.consts;
    void* d_bias = bias != nullptr ? base + L.consts + round256(row) : nullptr;

#define AR_TRY(call)                       \
    do {                                   \
        if ((call) != cudaSuccess)         \
            return AR_ERR_CUDA;            \
    } while (0)

    // Everything of this call comes after what the caller queued before it.
    AR_TRY(cudaEventRecord(P->entry, cs));
    AR_TRY(cudaStreamWaitEvent(P->copy_in, P->entry, 0));
    AR_TRY(cudaStreamWaitEvent(P->copy_out, P->entry, 0));
    AR_TRY(cudaMemcpyAsync(d_weight, weight, row, cudaMemcpyHostToDevice, P->copy_in));
    if (bias != nullptr)
        AR_TRY(cudaMemcpyAsync(d_bias, bias, row, cudaMemcpyHostToDevice, P->copy_in));
    AR_TRY(cudaEventRecord(P->consts, P->copy_in));
    AR_TRY(cudaStreamWaitEvent(cs, P->consts, 0));

    // (first row, rows) of every piece: whole chunks, then the shrinking tail.
    std::vector<std::pair<int, int>> pieces;
    int next = 0;
    while (tokens - next > chunk_tokens) {
        pieces.emplace_back(next, chunk_tokens);
        next += chunk_tokens;
    }
    for (int rem = tokens - next; rem > 0;) {
        const int p = rem > 2 * kMinTailRows ? (rem + 1) / 2 : rem;
        pieces.emplace_back(next, p);
        next += p;
        rem -= p;
    }
    const int nchunks = static_cast<int>(pieces.size());
    for (int i = 0; i < nchunks; ++i) {
        const int b = i % kBuffers;
        const int t0 = pieces[i].first;
        const int rows = pieces[i].second;
        const size_t off = static_cast<size_t>(t0) * row;
        const size_t bytes = static_cast<size_t>(rows) * row;
        char* buf = base + b * L.buffer;
        const void* d_parts[AR_MAX_RANKS];
        for (int r = 0; r < R; ++r)
            d_parts[r] = buf + r * L.chunk_bytes;
        char* d_res = buf + R * L.chunk_bytes;
        char* d_out = buf + (R + 1) * L.chunk_bytes;
        char* d_rout = buf + (R + 2) * L.chunk_bytes;
        char* d_ws = buf + (R + 3) * L.chunk_bytes;

        // The buffer is free once its previous chunk's outputs are back home
        // (which also means that chunk's kernel has read its inputs).
        if (i >= kBuffers)
            AR_TRY(cudaStreamWaitEvent(P->copy_in, P->drained[b], 0));
        for (int r = 0; r < R; ++r)
            AR_TRY(cudaMemcpyAsync(buf + r * L.chunk_bytes, static_cast<const char*>(partials[r]) + off, bytes,
                                   cudaMemcpyHostToDevice, P->copy_in));
        AR_TRY(cudaMemcpyAsync(d_res, static_cast<const char*>(residual) + off, bytes, cudaMemcpyHostToDevice,
                               P->copy_in));
        AR_TRY(cudaEventRecord(P->staged[b], P->copy_in));

        AR_TRY(cudaStreamWaitEvent(cs, P->staged[b], 0));
        const int st = ar_residual_rmsnorm(d_parts, R, d_bias, d_res, d_weight, eps, hidden, rows, d_out, d_rout,
                                           d_ws, L.ws_bytes, dtype, strategy, stream);
        if (st != AR_OK)
            return st;
        AR_TRY(cudaEventRecord(P->computed[b], cs));

        AR_TRY(cudaStreamWaitEvent(P->copy_out, P->computed[b], 0));
        AR_TRY(cudaMemcpyAsync(static_cast<char*>(out) + off, d_out, bytes, cudaMemcpyDeviceToHost, P->copy_out));
        AR_TRY(cudaMemcpyAsync(static_cast<char*>(residual_out) + off, d_rout, bytes, cudaMemcpyDeviceToHost,
                               P->copy_out));
        AR_TRY(cudaEventRecord(P->drained[b], P->copy_out));
    }
    // Work queued on the caller's stream after this call sees the outputs.
    for (int b = 0; b < kBuffers && b < nchunks; ++b)
        AR_TRY(cudaStreamWaitEvent(cs, P->drained[b], 0));
#undef AR_TRY
    return AR_OK;
}
