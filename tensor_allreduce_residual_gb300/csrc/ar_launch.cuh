// ar_launch.cuh -- launchers: pick the compile-time specialisation (rank
// count, units per thread) and the grid, then launch on the caller's stream.
// Included once per element type by ar_kern_{f32,f16,bf16}.cu.
//
// Specialisations: the rank count R is a template parameter for 1..8 on the
// reduce-only path and for 1, 2, 4 and 8 on the fused paths (the rank counts
// of a tensor-parallel node; other R use a runtime loop), after the
// AllReduceDispatchType -> AllReduceDispatchRanksPerNode templates of
// "allreduce.d2".
#pragma once

#include <climits>
#include <utility>

#include "ar_kernels.cuh"
#include "ar_lamport.cuh"
#include "ar_tma.cuh"

namespace ar {

// Launches `kernel` on `s` with the programmatic-stream-serialization
// attribute (see pdl_enter in ar_kernels.cuh); returns the launch status.
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename T, bool PACKED, int R_CT, int UNROLL>
static cudaError_t run_sum(const SumArgs& a, int nslices, cudaStream_t s)
{
    const uint64_t per_block = static_cast<uint64_t>(kFlatThreads) * UNROLL;
    uint64_t gx = (a.slice + per_block - 1) / per_block;
    if (gx == 0)
        gx = 1;  // a tail-only launch still needs one block
    if (gx > static_cast<uint64_t>(INT_MAX))
        return cudaErrorInvalidConfiguration;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(nslices));
    return launch_k(k_sum<T, PACKED, R_CT, UNROLL>, grid, dim3(kFlatThreads), 0, s, a);
}

template <typename T>
cudaError_t launch_sum(const SumArgs& a, bool packed, int nslices, cudaStream_t s)
{
    if (!packed)
        return run_sum<T, false, 0, sum_unroll(0, false)>(a, nslices, s);
    switch (a.R) {
    case 1: return run_sum<T, true, 1, sum_unroll(1, true)>(a, nslices, s);
    case 2: return run_sum<T, true, 2, sum_unroll(2, true)>(a, nslices, s);
    case 3: return run_sum<T, true, 3, sum_unroll(3, true)>(a, nslices, s);
    case 4: return run_sum<T, true, 4, sum_unroll(4, true)>(a, nslices, s);
    case 5: return run_sum<T, true, 5, sum_unroll(5, true)>(a, nslices, s);
    case 6: return run_sum<T, true, 6, sum_unroll(6, true)>(a, nslices, s);
    case 7: return run_sum<T, true, 7, sum_unroll(7, true)>(a, nslices, s);
    case 8: return run_sum<T, true, 8, sum_unroll(8, true)>(a, nslices, s);
    default: return run_sum<T, true, 0, sum_unroll(16, true)>(a, nslices, s);
    }
}

// Same as launch_k, with the blocks grouped into clusters of `cluster_x`.
template <typename... KArgs, typename... Args>
static cudaError_t launch_k_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    unsigned cluster_x, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// One row per cluster of sh.cluster blocks of sh.tpr threads.
template <typename T, int R_CT, int VPT>
static cudaError_t run_cluster(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    const long long blocks = static_cast<long long>(a.tokens) * sh.cluster;
    if (blocks > INT_MAX || sh.cluster < 1 || sh.cluster > kMaxCluster)
        return cudaErrorInvalidConfiguration;
    return launch_k_cluster(k_fused_oneshot_cluster<T, R_CT, VPT>, dim3(static_cast<unsigned>(blocks)),
                            dim3(sh.tpr), 0, s, static_cast<unsigned>(sh.cluster), a, sh.cluster);
}

template <typename T, bool PACKED, int R_CT, int VPT, bool STAGE, bool EARLY>
static cudaError_t run_oneshot(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    auto kernel = k_fused_oneshot<T, PACKED, R_CT, VPT, STAGE, EARLY>;
    if (STAGE && sh.smem_bytes > 48 * 1024) {
        // Beyond 48 KB of dynamic shared memory a kernel must opt in (per device).
        const cudaError_t attr = cudaFuncSetAttribute(
            kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxStageBytes);
        if (attr != cudaSuccess)
            return attr;
    }
    const int threads = sh.tpr * sh.rows;
    const unsigned grid = static_cast<unsigned>((a.tokens + sh.rows - 1) / sh.rows);
    return launch_k(kernel, dim3(grid), dim3(threads), STAGE ? sh.smem_bytes : 0, s, a, sh.tpr);
}

template <typename T, bool PACKED, int R_CT, bool STAGE, bool EARLY>
static cudaError_t oneshot_vpt(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    switch (sh.vpt) {
    case 1: return run_oneshot<T, PACKED, R_CT, 1, STAGE, EARLY>(a, sh, s);
    case 2: return run_oneshot<T, PACKED, R_CT, 2, STAGE, EARLY>(a, sh, s);
    case 4: return run_oneshot<T, PACKED, R_CT, 4, STAGE, EARLY>(a, sh, s);
    case 8: return run_oneshot<T, PACKED, R_CT, 8, STAGE, EARLY>(a, sh, s);
    case 16:
        if constexpr (!PACKED && !STAGE)
            return run_oneshot<T, PACKED, R_CT, 16, STAGE, EARLY>(a, sh, s);
        return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool PACKED, int R_CT, bool STAGE>
static cudaError_t oneshot_order(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    return sh.early_residual ? oneshot_vpt<T, PACKED, R_CT, STAGE, true>(a, sh, s)
                             : oneshot_vpt<T, PACKED, R_CT, STAGE, false>(a, sh, s);
}

template <typename T, int R_CT, int VPT>
static cudaError_t run_persist(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    auto kernel = k_fused_oneshot_persist<T, R_CT, VPT>;
    if (sh.smem_bytes > 48 * 1024) {
        const cudaError_t attr = cudaFuncSetAttribute(
            kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxStageBytes);
        if (attr != cudaSuccess)
            return attr;
    }
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, sh.tpr, sh.smem_bytes);
    if (e != cudaSuccess)
        return e;
    const long long resident = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = static_cast<unsigned>(a.tokens < resident ? a.tokens : resident);
    return launch_k(kernel, dim3(grid), dim3(sh.tpr), sh.smem_bytes, s, a);
}

// Persistent blocks fed by bulk copies: sh.tpr consumer threads plus one
// producer warp, sh.stages ring slots, sh.blocks_per_sm blocks per SM.
template <typename T, int R_CT, int CPR>
static cudaError_t run_tma(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    auto kernel = k_fused_oneshot_tma<T, R_CT, CPR>;
    if (sh.tpr > tma_max_consumers(CPR))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem_bytes);
    int dev = 0, sms = 0;
    if (e == cudaSuccess)
        e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const long long slots = static_cast<long long>(sms) * sh.blocks_per_sm;
    const unsigned grid = static_cast<unsigned>(a.tokens < slots ? a.tokens : slots);
    return launch_k(kernel, dim3(grid), dim3(sh.tpr + 32), sh.smem_bytes, s, a, sh.stages);
}

template <typename T, int R_CT>
static cudaError_t oneshot_packed(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    if (sh.mode == kCluster) {
        switch (sh.vpt) {
        case 1: return run_cluster<T, R_CT, 1>(a, sh, s);
        case 2: return run_cluster<T, R_CT, 2>(a, sh, s);
        case 4: return run_cluster<T, R_CT, 4>(a, sh, s);
        case 8: return run_cluster<T, R_CT, 8>(a, sh, s);
        default: return cudaErrorInvalidValue;
        }
    }
    if (sh.mode == kTma) {
        switch (sh.vpt) {
        case 1: return run_tma<T, R_CT, 1>(a, sh, s);
        case 2: return run_tma<T, R_CT, 2>(a, sh, s);
        case 4: return run_tma<T, R_CT, 4>(a, sh, s);
        case 8: return run_tma<T, R_CT, 8>(a, sh, s);
        default: return cudaErrorInvalidValue;
        }
    }
    if constexpr (R_CT > 0) {
        if (sh.mode == kPersistent) {
            switch (sh.vpt) {
            case 1: return run_persist<T, R_CT, 1>(a, sh, s);
            case 2: return run_persist<T, R_CT, 2>(a, sh, s);
            case 4: return run_persist<T, R_CT, 4>(a, sh, s);
            case 8: return run_persist<T, R_CT, 8>(a, sh, s);
            default: return cudaErrorInvalidValue;
            }
        }
    }
    return sh.mode != kRegisters ? oneshot_order<T, true, R_CT, true>(a, sh, s)
                                 : oneshot_order<T, true, R_CT, false>(a, sh, s);
}

template <typename T>
cudaError_t launch_fused_oneshot(const FusedArgs& a, bool packed, OneShotShape sh, cudaStream_t s)
{
    if (!packed)
        return oneshot_vpt<T, false, 0, false, true>(a, sh, s);
    switch (a.R) {
    case 1: return oneshot_packed<T, 1>(a, sh, s);
    case 2: return oneshot_packed<T, 2>(a, sh, s);
    case 4: return oneshot_packed<T, 4>(a, sh, s);
    case 8: return oneshot_packed<T, 8>(a, sh, s);
    default: return oneshot_packed<T, 0>(a, sh, s);
    }
}

template <typename T, bool PACKED, int VPT>
static cudaError_t run_rmsnorm(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    const unsigned grid = static_cast<unsigned>((a.tokens + sh.rows - 1) / sh.rows);
    return launch_k(k_rmsnorm<T, PACKED, VPT>, dim3(grid), dim3(sh.tpr * sh.rows), 0, s, a, sh.tpr);
}

template <typename T, bool PACKED>
static cudaError_t rmsnorm_vpt(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    switch (sh.vpt) {
    case 1: return run_rmsnorm<T, PACKED, 1>(a, sh, s);
    case 2: return run_rmsnorm<T, PACKED, 2>(a, sh, s);
    case 4: return run_rmsnorm<T, PACKED, 4>(a, sh, s);
    case 8: return run_rmsnorm<T, PACKED, 8>(a, sh, s);
    case 16:
        if constexpr (!PACKED)
            return run_rmsnorm<T, PACKED, 16>(a, sh, s);
        return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_rmsnorm(const FusedArgs& a, bool packed, OneShotShape sh, cudaStream_t s)
{
    return packed ? rmsnorm_vpt<T, true>(a, sh, s) : rmsnorm_vpt<T, false>(a, sh, s);
}

template <typename T>
cudaError_t launch_rmsnorm_tma(const FusedArgs& a, OneShotShape sh, cudaStream_t s)
{
    switch (sh.vpt) {
    case 1: return run_tma<T, 1, 1>(a, sh, s);
    case 2: return run_tma<T, 1, 2>(a, sh, s);
    case 4: return run_tma<T, 1, 4>(a, sh, s);
    case 8: return run_tma<T, 1, 8>(a, sh, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, bool PACKED, int R_CT>
static cudaError_t run_twoshot(const FusedArgs& a, cudaStream_t s)
{
    const uint64_t blocks = static_cast<uint64_t>(a.tokens) * a.nchunk;
    if (blocks > static_cast<uint64_t>(INT_MAX))
        return cudaErrorInvalidConfiguration;
    const cudaError_t e = launch_k(k_twoshot_phase1<T, PACKED, R_CT>, dim3(static_cast<unsigned>(blocks)),
                                   dim3(kFlatThreads), 0, s, a);
    if (e != cudaSuccess)
        return e;
    return launch_k(k_twoshot_phase2<T, PACKED>, dim3(static_cast<unsigned>(blocks)), dim3(kFlatThreads), 0, s, a);
}

template <typename T>
cudaError_t launch_fused_twoshot(const FusedArgs& a, bool packed, cudaStream_t s)
{
    if (!packed)
        return run_twoshot<T, false, 0>(a, s);
    switch (a.R) {
    case 1: return run_twoshot<T, true, 1>(a, s);
    case 2: return run_twoshot<T, true, 2>(a, s);
    case 4: return run_twoshot<T, true, 4>(a, s);
    case 8: return run_twoshot<T, true, 8>(a, s);
    default: return run_twoshot<T, true, 0>(a, s);
    }
}

// Lamport-style fused kernel: one cooperative launch (all blocks resident at
// once, which its blocks' waits on one another need).  One block per row
// group (rows, or row slices when rows are split), capped at the blocks that
// fit on the device at once and at half the ring's groups (rounded down to
// whole split rows); blocks take the groups in steps of the grid.
template <typename T, int R_CT, int VPT>
static cudaError_t run_lamport(const FusedArgs& a, void* lam, OneShotShape sh, int skip_rank, uint32_t epoch,
                               cudaStream_t s)
{
    auto kernel = k_fused_lamport<T, R_CT, VPT>;
    const int threads = sh.tpr * sh.rows;
    const int ring_steps = sh.stages;
    if (ring_steps < 2 || ring_steps > kLamportMaxRingSteps)
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int csize = sh.mode == kCluster ? sh.cluster : 1;
    const long long groups = csize > 1 ? static_cast<long long>(a.tokens) * csize
                                       : (static_cast<long long>(a.tokens) + sh.rows - 1) / sh.rows;
    if (groups > INT_MAX || (csize > 1 && sh.rows != 1))
        return cudaErrorInvalidConfiguration;
    // Whole steps of split rows: the grid is a multiple of csize.
    long long cap = static_cast<long long>(sms) * per_sm;
    if (cap > kLamportRingGroups / ring_steps)
        cap = kLamportRingGroups / ring_steps;
    cap = cap / csize * csize;
    if (cap < csize)
        return cudaErrorInvalidConfiguration;
    const long long grid = groups < cap ? groups : cap;
    const int slot_rows = lamport_slot_rows(a.tokens, sh.rows, csize);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, a, static_cast<uint4*>(lam), sh.tpr, csize, skip_rank, slot_rows, epoch,
                              ring_steps);
}

// The same with separate push and reduce warps: blocks of 2 x tpr x rows
// threads, rows never split.
template <typename T, int R_CT, int VPT>
static cudaError_t run_lamport_ws(const FusedArgs& a, void* lam, OneShotShape sh, int skip_rank, uint32_t epoch,
                                  cudaStream_t s)
{
    const int threads = 2 * sh.tpr * sh.rows;
    auto kernel = k_fused_lamport_ws<T, R_CT, VPT, 512>;
    if constexpr (VPT <= 2) {
        if (threads > 512)
            kernel = k_fused_lamport_ws<T, R_CT, VPT, 1024>;
    }
    const int ring_steps = sh.stages;
    if (ring_steps < 2 || ring_steps > kLamportMaxRingSteps)
        return cudaErrorInvalidValue;
    if (sh.mode == kCluster || threads > (VPT <= 2 ? 1024 : 512))
        return cudaErrorInvalidConfiguration;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const long long groups = (static_cast<long long>(a.tokens) + sh.rows - 1) / sh.rows;
    if (groups > INT_MAX)
        return cudaErrorInvalidConfiguration;
    long long cap = static_cast<long long>(sms) * per_sm;
    if (cap > kLamportRingGroups / ring_steps)
        cap = kLamportRingGroups / ring_steps;
    const long long grid = groups < cap ? groups : cap;
    const int slot_rows = lamport_slot_rows(a.tokens, sh.rows, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, a, static_cast<uint4*>(lam), sh.tpr, skip_rank, slot_rows, epoch,
                              ring_steps);
}

template <typename T, int R_CT>
static cudaError_t lamport_vpt(const FusedArgs& a, void* lam, OneShotShape sh, int skip_rank, uint32_t epoch,
                               cudaStream_t s)
{
    if (sh.roles) {
        switch (sh.vpt) {
        case 1: return run_lamport_ws<T, R_CT, 1>(a, lam, sh, skip_rank, epoch, s);
        case 2: return run_lamport_ws<T, R_CT, 2>(a, lam, sh, skip_rank, epoch, s);
        case 4: return run_lamport_ws<T, R_CT, 4>(a, lam, sh, skip_rank, epoch, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (sh.vpt) {
    case 1: return run_lamport<T, R_CT, 1>(a, lam, sh, skip_rank, epoch, s);
    case 2: return run_lamport<T, R_CT, 2>(a, lam, sh, skip_rank, epoch, s);
    case 4: return run_lamport<T, R_CT, 4>(a, lam, sh, skip_rank, epoch, s);
    case 8: return run_lamport<T, R_CT, 8>(a, lam, sh, skip_rank, epoch, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_fused_lamport(const FusedArgs& a, void* lam, OneShotShape sh, int skip_rank, uint32_t epoch,
                                 cudaStream_t s)
{
    switch (a.R) {
    case 1: return lamport_vpt<T, 1>(a, lam, sh, skip_rank, epoch, s);
    case 2: return lamport_vpt<T, 2>(a, lam, sh, skip_rank, epoch, s);
    case 4: return lamport_vpt<T, 4>(a, lam, sh, skip_rank, epoch, s);
    case 8: return lamport_vpt<T, 8>(a, lam, sh, skip_rank, epoch, s);
    default: return lamport_vpt<T, 0>(a, lam, sh, skip_rank, epoch, s);
    }
}

template <typename T>
cudaError_t launch_lamport_fill(void* buf, size_t bytes, cudaStream_t s)
{
    const uint64_t nvec = bytes / 16;
    const uint32_t tail_halves = static_cast<uint32_t>((bytes % 16) / 2);
    uint64_t blocks = (nvec + kFlatThreads - 1) / kFlatThreads;
    if (blocks > 4096)
        blocks = 4096;
    if (blocks == 0)
        blocks = 1;
    return launch_k(k_lamport_fill<T>, dim3(static_cast<unsigned>(blocks)), dim3(kFlatThreads), 0, s,
                    static_cast<uint4*>(buf), nvec, tail_halves);
}

template <typename T>
cudaError_t take_wait_timeouts(unsigned int* count)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v));
    if (e == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
    }
    *count = v;
    return e;
}

}  // namespace ar

#define AR_INSTANTIATE_LAUNCHERS(T)                                                                   \
    template cudaError_t ar::launch_sum<T>(const ar::SumArgs&, bool, int, cudaStream_t);              \
    template cudaError_t ar::launch_fused_oneshot<T>(const ar::FusedArgs&, bool, ar::OneShotShape,    \
                                                     cudaStream_t);                                   \
    template cudaError_t ar::launch_fused_twoshot<T>(const ar::FusedArgs&, bool, cudaStream_t);     \
    template cudaError_t ar::take_wait_timeouts<T>(unsigned int*);                                  \
    template cudaError_t ar::launch_rmsnorm<T>(const ar::FusedArgs&, bool, ar::OneShotShape, cudaStream_t);      \
    template cudaError_t ar::launch_rmsnorm_tma<T>(const ar::FusedArgs&, ar::OneShotShape, cudaStream_t);     \
    template cudaError_t ar::launch_fused_lamport<T>(const ar::FusedArgs&, void*, ar::OneShotShape, int,       \
                                                     uint32_t, cudaStream_t);                                \
    template cudaError_t ar::launch_lamport_fill<T>(void*, size_t, cudaStream_t);
