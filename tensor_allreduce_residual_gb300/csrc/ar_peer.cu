// ar_peer.cu -- the all-reduce across the GPUs of one node: one process per
// GPU, each rank's partial in its own GPU, every rank reading its peers'
// buffers directly (the peer_comm_buffer_ptrs[MAX_RANKS_PER_NODE] of
// AllReduceParams, "type.d2"; oneShotAllReduceKernel and
// twoShotAllReduceKernel with their barriers, "allreduce.d2").  Host code
// and kernels for all three element types.
//
// Each rank registers one device buffer:
//   [flags]  2 barriers x kPeerBlocks blocks x AR_MAX_RANKS sources, uint32:
//            word (ph, b, src) of rank r's buffer is the last call (epoch)
//            in which block b of rank src reached barrier ph;
//   [data 0] [data 1]  two areas of round256(max_bytes): call e uses area
//            e & 1, so a call never writes an area a peer may still read
//            for the call before it (see the barrier below).
// Peers' buffers are mapped with CUDA IPC (cudaIpcOpenMemHandle).  Loads
// and stores to them are plain peer accesses; no multicast.
//
// Per-block barrier ph of call e, block b of rank r:
//   __syncthreads(); thread t < world stores e (release, system scope) into
//   word (ph, b, r) of rank t's flags; thread t < world waits (acquire,
//   bounded) until word (ph, b, t) of its own flags is >= e; __syncthreads().
// A block only reads, from every rank, the elements that block b of that
// rank wrote before the same barrier, so a per-block barrier is enough.
// The epochs grow by one per call on every rank (all ranks make the same
// calls), so flags never need resetting; ">=" accepts a peer that has
// already signalled the next call.  Reuse of a data area: block b of rank r
// writes area e & 1 again in call e + 2 only after passing barrier 0 of call
// e + 1, which every rank's block b reaches only after finishing call e.
//
// Every wait gives up after kPeerWaitNs of %globaltimer time, counts the
// event for ar_device_status and lets the block finish without the data it
// waited for.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <new>

#include "ar.h"
#include "ar_kernels.cuh"

namespace ar {

constexpr int kPeerBlocks = 128;
constexpr int kPeerThreads = 512;
constexpr int kPeerUnroll = 4;
constexpr size_t kPeerFlagBytes = 2ull * kPeerBlocks * AR_MAX_RANKS * sizeof(uint32_t);
constexpr unsigned long long kPeerWaitNs = 1000000000ull;

static __device__ unsigned int g_peer_wait_timeouts;

struct PeerArgs {
    const void* in;
    void* out;
    void* data[AR_MAX_RANKS];       // this call's data area of every rank
    uint32_t* flags[AR_MAX_RANKS];  // every rank's flag words
    uint64_t nunits;                // 16-byte vectors
    uint32_t tail;                  // elements after the last vector
    int rank;
    int world;
    uint32_t epoch;
};

__device__ __forceinline__ unsigned long long peer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v)
{
    asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A peer's element or vector, read from L2 (not kept in L1).
__device__ __forceinline__ uint4 ld_peer16(const void* p) { return __ldcg(static_cast<const uint4*>(p)); }

// Barrier ph of this call among block blockIdx.x of every rank.  False if a
// wait gave up (the block then carries on without the data).
__device__ bool peer_barrier(const PeerArgs& a, int ph)
{
    __shared__ int gave_up_at[2];  // one per barrier, so a reset never races a read of the other
    int& gave_up = gave_up_at[ph];
    if (threadIdx.x == 0)
        gave_up = 0;
    __syncthreads();
    const int t = static_cast<int>(threadIdx.x);
    const size_t word = (static_cast<size_t>(ph) * kPeerBlocks + blockIdx.x) * AR_MAX_RANKS;
    if (t < a.world)
        st_release_sys(a.flags[t] + word + a.rank, a.epoch);
    if (t < a.world) {
        const uint32_t* w = a.flags[a.rank] + word + t;
        if (static_cast<int32_t>(ld_acquire_sys(w) - a.epoch) < 0) {
            const unsigned long long t0 = peer_ns();
            bool ok = false;
            do {
                __nanosleep(64);
                ok = static_cast<int32_t>(ld_acquire_sys(w) - a.epoch) >= 0;
            } while (!ok && peer_ns() - t0 <= kPeerWaitNs);
            if (!ok) {
                atomicAdd(&g_peer_wait_timeouts, 1u);
                gave_up = 1;
            }
        }
    }
    __syncthreads();
    return gave_up == 0;
}

// This block's share [u0, u1) of n units, in kPeerBlocks-independent pieces:
// block b of every rank gets the same range (the barrier relies on it).
__device__ __forceinline__ void block_range(uint64_t n, uint64_t* u0, uint64_t* u1)
{
    const uint64_t per = (n + gridDim.x - 1) / gridDim.x;
    *u0 = min(n, static_cast<uint64_t>(blockIdx.x) * per);
    *u1 = min(n, *u0 + per);
}

// dst[u] (and dst2[u] if not null) = sum over ranks (rank order, fp32) of
// data[r][u], rounded once, for u in [u0, u1).
template <typename T>
__device__ void peer_sum_range(const PeerArgs& a, uint64_t u0, uint64_t u1, void* dst, void* dst2)
{
    using U = Unit<T, true>;
    constexpr int L = U::L;
    for (uint64_t u = u0 + threadIdx.x; u < u1; u += blockDim.x) {
        float acc[L], t[L];
        U::to_float(ld_peer16(static_cast<const uint4*>(a.data[0]) + u), acc);
        for (int r = 1; r < a.world; ++r) {
            U::to_float(ld_peer16(static_cast<const uint4*>(a.data[r]) + u), t);
            add_lanes<L>(acc, t);
        }
        U::store(dst, u, acc);
        if (dst2 != nullptr)
            U::store(dst2, u, acc);
    }
}

// The elements after the last vector: block 0 copies its rank's (phase
// "copy") or sums every rank's into out (phase "sum").
template <typename T>
__device__ void peer_tail(const PeerArgs& a, bool sum)
{
    if (blockIdx.x != 0 || a.tail == 0)
        return;
    const uint64_t e0 = a.nunits * Lanes<T>::V;
    for (uint32_t i = threadIdx.x; i < a.tail; i += blockDim.x) {
        if (!sum) {
            static_cast<T*>(a.data[a.rank])[e0 + i] = static_cast<const T*>(a.in)[e0 + i];
        } else {
            float acc = Lanes<T>::to_f(static_cast<const T*>(a.data[0])[e0 + i]);
            for (int r = 1; r < a.world; ++r)
                acc += Lanes<T>::to_f(static_cast<const T*>(a.data[r])[e0 + i]);
            static_cast<T*>(a.out)[e0 + i] = Lanes<T>::from_f(acc);
        }
    }
}

// One-shot: copy this block's range of the input into this rank's area,
// barrier, then sum every rank's range.
template <typename T>
__global__ void __launch_bounds__(kPeerThreads) k_peer_oneshot(const PeerArgs a)
{
    uint64_t u0, u1;
    block_range(a.nunits, &u0, &u1);
    for (uint64_t u = u0 + threadIdx.x; u < u1; u += blockDim.x)
        static_cast<uint4*>(a.data[a.rank])[u] = __ldcs(static_cast<const uint4*>(a.in) + u);
    peer_tail<T>(a, false);
    if (!peer_barrier(a, 0))
        return;
    peer_sum_range<T>(a, u0, u1, a.out, nullptr);
    peer_tail<T>(a, true);
}

// Two-shot: the vectors are cut into `world` rank slices; block b owns part b
// of every slice.  Copy part b of every slice into this rank's area,
// barrier; reduce part b of this rank's slice over every rank (written back
// into this rank's area and into out: the reduce-scatter); barrier; copy
// part b of every other slice from its rank's area (the all-gather).
template <typename T>
__global__ void __launch_bounds__(kPeerThreads) k_peer_twoshot(const PeerArgs a)
{
    const uint64_t slice = (a.nunits + a.world - 1) / a.world;
    auto part = [&](int s, uint64_t* p0, uint64_t* p1) {
        const uint64_t s0 = min(a.nunits, static_cast<uint64_t>(s) * slice);
        const uint64_t s1 = min(a.nunits, s0 + slice);
        const uint64_t per = (s1 - s0 + gridDim.x - 1) / gridDim.x;
        *p0 = min(s1, s0 + static_cast<uint64_t>(blockIdx.x) * per);
        *p1 = min(s1, *p0 + per);
    };
    uint64_t p0, p1;
    for (int s = 0; s < a.world; ++s) {
        part(s, &p0, &p1);
        for (uint64_t u = p0 + threadIdx.x; u < p1; u += blockDim.x)
            static_cast<uint4*>(a.data[a.rank])[u] = __ldcs(static_cast<const uint4*>(a.in) + u);
    }
    peer_tail<T>(a, false);
    if (!peer_barrier(a, 0))
        return;
    // The reduced part goes to out and back into this rank's area, where the
    // peers gather it from.
    part(a.rank, &p0, &p1);
    peer_sum_range<T>(a, p0, p1, a.out, a.data[a.rank]);
    peer_tail<T>(a, true);
    if (!peer_barrier(a, 1))
        return;
    for (int s = 0; s < a.world; ++s) {
        if (s == a.rank)
            continue;
        part(s, &p0, &p1);
        for (uint64_t u = p0 + threadIdx.x; u < p1; u += blockDim.x)
            static_cast<uint4*>(a.out)[u] = ld_peer16(static_cast<const uint4*>(a.data[s]) + u);
    }
}

template <typename T>
cudaError_t launch_peer(const PeerArgs& a, bool twoshot, cudaStream_t s)
{
    const uint64_t work = twoshot ? (a.nunits + a.world - 1) / a.world : a.nunits;
    uint64_t blocks = (work + static_cast<uint64_t>(kPeerThreads) * kPeerUnroll - 1) /
                      (static_cast<uint64_t>(kPeerThreads) * kPeerUnroll);
    if (blocks < 1)
        blocks = 1;
    if (blocks > kPeerBlocks)
        blocks = kPeerBlocks;
    if (twoshot)
        k_peer_twoshot<T><<<static_cast<unsigned>(blocks), kPeerThreads, 0, s>>>(a);
    else
        k_peer_oneshot<T><<<static_cast<unsigned>(blocks), kPeerThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ar

struct ar_comm {
    int rank;
    int world;
    int device;
    size_t max_bytes;
    size_t area_bytes;
    void* base[AR_MAX_RANKS];    // every rank's registered buffer, mapped here
    bool opened[AR_MAX_RANKS];   // mapped with cudaIpcOpenMemHandle (closed on destroy)
    uint32_t epoch;
};

namespace {

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int peer_esize(int dtype)
{
    switch (dtype) {
    case AR_FP32: return 4;
    case AR_FP16: return 2;
    case AR_BF16: return 2;
    default: return 0;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Zeroes this rank's flag words (synchronous: done before the caller's
// host barrier that precedes the first call).
int init_flags(void* buffer)
{
    return cudaMemset(buffer, 0, ar::kPeerFlagBytes) == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

int check_create(int rank, int world, const void* buffer, size_t buffer_bytes, size_t max_bytes, ar_comm** comm)
{
    if (comm == nullptr || world < 1 || world > AR_MAX_RANKS || rank < 0 || rank >= world || buffer == nullptr ||
        !aligned16(buffer) || max_bytes == 0)
        return AR_ERR_INVALID_ARG;
    if (buffer_bytes < ar_comm_buffer_size(world, max_bytes))
        return AR_ERR_WORKSPACE;
    return AR_OK;
}

ar_comm* new_comm(int rank, int world, size_t max_bytes)
{
    ar_comm* c = new (std::nothrow) ar_comm{};
    if (c == nullptr)
        return nullptr;
    c->rank = rank;
    c->world = world;
    c->max_bytes = max_bytes;
    c->area_bytes = round256(max_bytes);
    c->epoch = 0;
    cudaGetDevice(&c->device);
    return c;
}

}  // namespace

extern "C" {

size_t ar_comm_buffer_size(int world, size_t max_bytes)
{
    if (world < 1 || world > AR_MAX_RANKS || max_bytes == 0)
        return 0;
    return ar::kPeerFlagBytes + 2 * round256(max_bytes);
}

int ar_comm_export(const void* buffer, void* handle)
{
    if (buffer == nullptr || handle == nullptr)
        return AR_ERR_INVALID_ARG;
    cudaIpcMemHandle_t h;
    if (cudaIpcGetMemHandle(&h, const_cast<void*>(buffer)) != cudaSuccess)
        return AR_ERR_CUDA;
    static_assert(sizeof(h) == AR_IPC_HANDLE_BYTES, "IPC handle size");
    const char* src = reinterpret_cast<const char*>(&h);
    char* dst = static_cast<char*>(handle);
    for (int i = 0; i < AR_IPC_HANDLE_BYTES; ++i)
        dst[i] = src[i];
    return AR_OK;
}

int ar_comm_create(int rank, int world, void* buffer, size_t buffer_bytes, size_t max_bytes, const void* handles,
                   ar_comm** comm)
{
    if (int st = check_create(rank, world, buffer, buffer_bytes, max_bytes, comm))
        return st;
    if (world > 1 && handles == nullptr)
        return AR_ERR_INVALID_ARG;
    ar_comm* c = new_comm(rank, world, max_bytes);
    if (c == nullptr)
        return AR_ERR_CUDA;
    c->base[rank] = buffer;
    int st = init_flags(buffer);
    for (int q = 0; q < world && st == AR_OK; ++q) {
        if (q == rank)
            continue;
        cudaIpcMemHandle_t h;
        const char* src = static_cast<const char*>(handles) + static_cast<size_t>(q) * AR_IPC_HANDLE_BYTES;
        char* dst = reinterpret_cast<char*>(&h);
        for (int i = 0; i < AR_IPC_HANDLE_BYTES; ++i)
            dst[i] = src[i];
        void* p = nullptr;
        if (cudaIpcOpenMemHandle(&p, h, cudaIpcMemLazyEnablePeerAccess) != cudaSuccess || p == nullptr) {
            st = AR_ERR_CUDA;
            break;
        }
        c->base[q] = p;
        c->opened[q] = true;
    }
    if (st != AR_OK) {
        ar_comm_destroy(c);
        return st;
    }
    *comm = c;
    return AR_OK;
}

int ar_comm_destroy(ar_comm* comm)
{
    if (comm == nullptr)
        return AR_ERR_INVALID_ARG;
    int st = AR_OK;
    for (int q = 0; q < comm->world; ++q)
        if (comm->opened[q] && cudaIpcCloseMemHandle(comm->base[q]) != cudaSuccess)
            st = AR_ERR_CUDA;
    delete comm;
    return st;
}

int ar_allreduce_peer(ar_comm* comm, const void* input, void* out, size_t n, int dtype, int strategy,
                      ar_stream_t stream)
{
    if (comm == nullptr)
        return AR_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return AR_ERR_CUDA;
    if (dev != comm->device)  // its peers' mappings belong to that device
        return AR_ERR_INVALID_ARG;
    const int esize = peer_esize(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (strategy != AR_ONESHOT && strategy != AR_TWOSHOT && strategy != AR_AUTO)
        return AR_ERR_UNSUPPORTED;
    if (n == 0)
        return AR_OK;
    if (input == nullptr || out == nullptr)
        return AR_ERR_INVALID_ARG;
    if (!aligned16(input) || !aligned16(out))
        return AR_ERR_UNSUPPORTED;
    if (n > comm->max_bytes / static_cast<size_t>(esize))
        return AR_ERR_WORKSPACE;
    // AUTO: one-shot moves world x n elements into every rank, two-shot
    // about 2 n; one-shot while a rank's share is small (latency), two-shot
    // beyond.  A size rule: every box this was built on has one GPU, so it is
    // not measured.
    const bool twoshot = strategy == AR_TWOSHOT ||
                         (strategy == AR_AUTO && comm->world > 2 && n * static_cast<size_t>(esize) >= (1u << 20));
    ar::PeerArgs a{};
    a.in = input;
    a.out = out;
    a.rank = comm->rank;
    a.world = comm->world;
    a.epoch = ++comm->epoch;
    const size_t area = ar::kPeerFlagBytes + static_cast<size_t>(a.epoch & 1u) * comm->area_bytes;
    for (int r = 0; r < comm->world; ++r) {
        a.flags[r] = static_cast<uint32_t*>(comm->base[r]);
        a.data[r] = static_cast<char*>(comm->base[r]) + area;
    }
    const int lanes = 16 / esize;
    a.nunits = n / static_cast<size_t>(lanes);
    a.tail = static_cast<uint32_t>(n % static_cast<size_t>(lanes));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (dtype) {
    case AR_FP32: e = ar::launch_peer<float>(a, twoshot, s); break;
    case AR_FP16: e = ar::launch_peer<__half>(a, twoshot, s); break;
    default: e = ar::launch_peer<__nv_bfloat16>(a, twoshot, s); break;
    }
    return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

#ifdef AR_TEST_HOOKS
// Test build only: a communicator whose ranks' buffers are all local device
// pointers (no IPC).  Its one use is a rank whose peers never run: its
// barrier waits then run out, which is how the bounded waits are tested on
// one GPU without anything waiting on another kernel.
int ar_comm_create_local(int rank, int world, void* const* buffers, size_t buffer_bytes, size_t max_bytes,
                         ar_comm** comm)
{
    if (buffers == nullptr)
        return AR_ERR_INVALID_ARG;
    if (int st = check_create(rank, world, buffers[rank], buffer_bytes, max_bytes, comm))
        return st;
    ar_comm* c = new_comm(rank, world, max_bytes);
    if (c == nullptr)
        return AR_ERR_CUDA;
    for (int q = 0; q < world; ++q) {
        if (buffers[q] == nullptr || init_flags(buffers[q]) != AR_OK) {
            delete c;
            return buffers[q] == nullptr ? AR_ERR_INVALID_ARG : AR_ERR_CUDA;
        }
        c->base[q] = buffers[q];
    }
    *comm = c;
    return AR_OK;
}
#endif

}  // extern "C"

namespace ar {

// Bounded waits of the peer kernels that gave up since the last call (which
// resets the count).  Synchronous.
cudaError_t take_peer_wait_timeouts(unsigned int* count)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_peer_wait_timeouts, sizeof(v));
    if (e == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_peer_wait_timeouts, &zero, sizeof(zero));
    }
    *count = v;
    return e;
}

}  // namespace ar
