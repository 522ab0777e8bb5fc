// ar_internal.h -- kernel argument blocks and launcher declarations shared by
// the host dispatch (ar_api.cu) and the per-dtype kernel translation units.
//
// The argument blocks are passed BY VALUE as kernel parameters (well under
// the 4 KB parameter limit), the way AllReduceParams carries
// peer_comm_buffer_ptrs[MAX_RANKS_PER_NODE] into the kernels ("type.d2",
// AllReduceParams): the R partial pointers travel with the launch, so the
// library needs no device-side pointer table and no allocation.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ar {

constexpr int kMaxRanks = 16;

// Threads per block of the flat kernels (reduce-only, two-shot phases).
constexpr int kFlatThreads = 256;

// Units each thread of the reduce-only kernel sums per launch (R * UNROLL
// loads in flight per thread): fewer for more partials, to bound registers.
__host__ __device__ constexpr int sum_unroll(int R, bool packed)
{
    return !packed ? 4 : (R <= 2 ? 8 : (R <= 4 ? 4 : 2));
}

// Two-shot fused path: vectors per thread per chunk.  A chunk is
// kFlatThreads * kChunkVPT packed vectors of one row.
constexpr int kChunkVPT = 2;

// One-shot fused path: the largest number of packed vectors (or scalar
// elements on the element-wise path) a thread keeps in registers, and the
// largest number of threads cooperating on one row.
constexpr int kMaxVPTVec = 8;
constexpr int kMaxVPTScalar = 16;
constexpr int kMaxTPR = 1024;

// Largest block of the one-shot fused kernel for a thread that holds
// `values` fp32 values of its row (units per thread * lanes per unit): they
// stay live across the row reduction, so more values need more registers
// per thread and hence fewer threads per block.
__host__ __device__ constexpr int oneshot_max_threads(int values)
{
    return values <= 16 ? 1024 : (values <= 32 ? 512 : 256);
}

// Largest block of the Lamport-style fused kernel for a thread that holds
// `values` fp32 values of its row: half the one-shot kernel's, because it
// also holds the R slot vectors of the unit it is polling.
__host__ __device__ constexpr int lamport_max_threads(int values)
{
    return values <= 16 ? 512 : 256;
}

// Largest block of the norm kernel k_rmsnorm for `vpt` units per thread: 8
// packed vectors (32 registers of row data) need a 512-thread cap to stay
// out of local memory; 4 packed vectors run in blocks of at most 256
// threads, norm_min_blocks of them per SM (40 registers a thread, against 60
// without the hint: 6 rows in flight per SM instead of 4); everything else
// fits 1024 threads.
__host__ __device__ constexpr int norm_max_threads(bool packed, int vpt)
{
    return packed && vpt >= 8 ? 512 : (packed && vpt == 4 ? 256 : kMaxTPR);
}
__host__ __device__ constexpr int norm_min_blocks(bool packed, int vpt)
{
    return packed && vpt == 4 ? 6 : 1;
}

struct SumArgs {
    const void* partials[kMaxRanks];
    void* out;
    int R;
    uint32_t tail;      // elements after the last full vector (packed path only)
    uint64_t nunits;    // full 16-byte vectors (packed path) or elements (element-wise path)
    uint64_t slice;     // units per slice: nunits (one-shot) or ~nunits/R (two-shot)
};

struct FusedArgs {
    const void* partials[kMaxRanks];
    const void* bias;      // nullable
    const void* residual;  // nullable for the norm on its own
    const void* weight;
    void* out;
    void* residual_out;    // nullable for the norm on its own
    float* sumsq;          // two-shot workspace: [tokens, nchunk] fp32
    int R;
    int hidden;
    int tokens;
    int units_row;         // packed vectors per row (packed path) or hidden (element-wise)
    int nchunk;            // two-shot chunks per row
    int chunk_units;       // two-shot units per chunk
    float eps;
    int early_residual;    // one-shot: write residual_out before the row barrier
    int stall_stage;       // test build only: the bulk-copy producer leaves stage (stall_stage - 1)
                           // of every block unarmed; always 0 (none) in the product library
};

// Where the one-shot fused kernel keeps a row's fp32 sums between the sum and
// the normalisation.
enum OneShotMode {
    kRegisters = 0,   // registers, one block per `rows` rows
    kStaged = 1,      // shared memory, one block per `rows` rows
    kPersistent = 2,  // shared memory, persistent blocks striding over rows
    kTma = 3,         // registers, persistent blocks fed by bulk copies into a shared-memory ring
    kCluster = 4      // registers, each row split across a thread-block cluster
};

// Cluster sizes the row-split one-shot kernel may use (portable limit 8).
constexpr int kMaxCluster = 8;

// One-shot fused launch shape: `tpr` threads per row (a power of two),
// `vpt` units per thread, `rows` rows per block, the mode, the dynamic
// shared memory of the staged modes, and when residual_out is written.
struct OneShotShape {
    int tpr;
    int vpt;
    int rows;
    int mode;
    int smem_bytes;
    int early_residual;  // write residual_out before the row barrier
    int stages;          // kTma: ring slots per block; Lamport call: ring depth in grid steps
    int blocks_per_sm;   // kTma: resident blocks per SM
    int cluster;         // kCluster: blocks per row (the cluster size); tpr is then threads per block
    int roles;           // Lamport call: 1 = separate push and reduce warps (k_fused_lamport_ws)
};

// Largest block of the persistent one-shot kernel (it keeps the next row's
// first units in registers across the row barrier, so it needs more of them).
constexpr int kMaxPersistThreads = 512;

// Largest dynamic shared memory a staged one-shot block may use.
constexpr int kMaxStageBytes = 96 * 1024;

// One-shot fused path fed by bulk copies (mode kTma): consumer threads per
// block for `cpr` chunks per row (each keeps cpr * lanes fp32 values of its
// row in registers, so longer rows per thread allow fewer threads), the ring
// depth limits, and the shared memory one block may use.
__host__ __device__ constexpr int tma_max_consumers(int cpr)
{
    return cpr <= 2 ? 512 : (cpr == 4 ? 256 : 128);
}
constexpr int kTmaMinStages = 2;
constexpr int kTmaMaxStages = 16;
constexpr int kSmemPerBlockMax = 227 * 1024;  // opt-in dynamic shared memory of one block
constexpr int kSmemPerSM = 228 * 1024;        // shared memory of one SM
constexpr int kSmemReservedPerBlock = 1024;   // taken by the runtime from each resident block

// Shared memory of one kTma block: `stages` ring slots of `inputs` * nc
// 16-byte vectors (inputs = the R partials, plus the residual when there is
// one), then a full and an empty barrier per slot (8 bytes each), then the
// row-reduction scratch, [2][32] floats.
__host__ __device__ constexpr size_t tma_smem_bytes(int inputs, int nc, int stages)
{
    return static_cast<size_t>(stages) * inputs * nc * 16 + static_cast<size_t>(stages) * 16 + 2 * 32 * 4;
}

// Whether launches carry the programmatic-stream-serialization attribute
// (defined in ar_api.cu: always in the product library).
bool pdl_enabled();

// Launchers, explicitly instantiated for float, __half and __nv_bfloat16 in
// the per-dtype translation units.  Each returns the cudaError_t of the launch.
template <typename T>
cudaError_t launch_sum(const SumArgs& a, bool packed, int nslices, cudaStream_t s);

template <typename T>
cudaError_t launch_fused_oneshot(const FusedArgs& a, bool packed, OneShotShape shape, cudaStream_t s);

template <typename T>
cudaError_t launch_fused_twoshot(const FusedArgs& a, bool packed, cudaStream_t s);

// RMSNorm of a.partials[0] rows into a.out (register-resident rows, shape.mode
// must be kRegisters).
template <typename T>
cudaError_t launch_rmsnorm(const FusedArgs& a, bool packed, OneShotShape shape, cudaStream_t s);

// The same through the bulk-copy-fed persistent kernel (shape.mode == kTma):
// a.partials[0] is x, a.R == 1, no bias, residual or residual_out.
template <typename T>
cudaError_t launch_rmsnorm_tma(const FusedArgs& a, OneShotShape shape, cudaStream_t s);

// Lamport-style fused call.  Buffer: one 64-bit progress word per block
// (kLamportProgressBytes), then R slots of slot_rows * units_row 16-byte
// vectors (a ring: row k of the call in ring row k mod ring_rows), then an
// exchange area of kLamportRowWords 32-bit words per token for rows split
// over up to kLamportMaxSplit blocks.
constexpr int kLamportMaxSplit = 8;
constexpr int kLamportRowWords = 16;

// The ring is ring_steps (2 .. kLamportMaxRingSteps, the launch shape's
// `stages`) steps of the launch's row groups deep; a slot holds at most
// kLamportRingGroups groups, so the launch takes at most that many over
// ring_steps blocks.  Rows one rank's slot holds for `tokens` rows of `rows_per_group`
// rows a group, or of rows split over `csize` > 1 blocks.
constexpr int kLamportRingGroups = 1024;
constexpr int kLamportMaxRingSteps = 4;
constexpr int kLamportProgressBytes = kLamportRingGroups / 2 * 8;
inline int lamport_slot_rows(int tokens, int rows_per_group, int csize)
{
    const long long cap = csize > 1 ? kLamportRingGroups / csize : static_cast<long long>(kLamportRingGroups) * rows_per_group;
    return tokens < cap ? tokens : static_cast<int>(cap);
}

// Pushes the R partials into the marker-filled buffer `lam`, then reduces
// from it in the same cooperative launch.  shape.mode == kRegisters: tpr
// threads a row; shape.mode == kCluster: each row split over shape.cluster
// blocks of shape.tpr threads.  skip_rank >= 0 leaves that rank's pushes out
// (tests).
// `epoch`: this call's own value in [1, 2^31), which its blocks' progress
// words carry.
template <typename T>
cudaError_t launch_fused_lamport(const FusedArgs& a, void* lam, OneShotShape shape, int skip_rank, uint32_t epoch,
                                 cudaStream_t s);

// Fills `bytes` of `buf` (16-byte aligned, bytes even) with T's empty marker.
template <typename T>
cudaError_t launch_lamport_fill(void* buf, size_t bytes, cudaStream_t s);

// Number of bounded waits that gave up in the kernels of element type T since
// the last call, which resets it.  Synchronous (reads device memory).
template <typename T>
cudaError_t take_wait_timeouts(unsigned int* count);

// The same for the multi-GPU peer kernels (ar_peer.cu).
cudaError_t take_peer_wait_timeouts(unsigned int* count);

}  // namespace ar
