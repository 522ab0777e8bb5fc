// ar_kernels.cuh -- device code of the single-GPU R-way sum and the fused
// sum + bias + residual + RMSNorm, for sm_103a.
//
// Every kernel here is bound by HBM bandwidth: about one fp32 add per
// element read, far below any ALU or tensor-core ridge, so the design goals
// are (1) 16-byte coalesced loads with many independent loads in flight per
// thread, (2) every input byte read once and every output byte written once,
// (3) fp32 accumulation in a fixed order for bit-reproducible results.
//
// Data views.  A "unit" is either a 16-byte packed vector (4 fp32 lanes, or
// 8 fp16 / bf16 lanes: the PackedOn16Bytes<T> int4 / float[4] / half2[4]
// unions of "type.d2") or, on the element-wise path taken for misaligned
// pointers, a single element.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ar_internal.h"

#ifndef AR_L2_PREFETCH_256B
#define AR_L2_PREFETCH_256B 0
#endif

namespace ar {

// ---------------------------------------------------------------------------
// Programmatic dependent launch (sm_90 and later).  Kernels here are launched
// with the programmatic-stream-serialization attribute, so one may start
// (get its blocks resident, set up shared memory) while the previous kernel
// in its stream is still running.  griddepcontrol.wait then blocks until
// every prerequisite grid has completed and its memory is visible, so each
// kernel calls pdl_enter() before it touches any global buffer, input or
// output.  It then lets the next kernel in the stream launch early too.
// Without the attribute both instructions do nothing.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// 16-byte packed vectors and single elements.
// ---------------------------------------------------------------------------

// Streaming 16-byte load: read-only path, not kept in L1 (each byte is read
// exactly once by exactly one thread).  The statement is volatile and clobbers
// memory so that the compiler keeps it after pdl_enter()'s griddepcontrol.wait
// and after any earlier store: several kernels read what the previous kernel
// in the stream wrote (two-shot phase 2 reads phase 1's residual_out, the norm
// reads a sum), and a load hoisted above the wait would see stale data.
__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 r;
#if AR_L2_PREFETCH_256B
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
#else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
#endif
    return r;
}

// Small read-mostly operands (weight, bias: one row reused by every row).
__device__ __forceinline__ uint4 ld_cached16(const void* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st16(void* p, uint4 v)
{
    *reinterpret_cast<uint4*>(p) = v;
}

template <typename T>
struct Lanes;

template <>
struct Lanes<float> {
    static constexpr int V = 4;
    __device__ static void unpack(const uint4& u, float* f)
    {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float* f)
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
};

template <>
struct Lanes<__half> {
    static constexpr int V = 8;
    __device__ static float2 two(uint32_t w)
    {
        __half2 h = *reinterpret_cast<const __half2*>(&w);
        return __half22float2(h);
    }
    __device__ static uint32_t word(float a, float b)
    {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static void unpack(const uint4& u, float* f)
    {
        float2 a = two(u.x), b = two(u.y), c = two(u.z), d = two(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ static uint4 pack(const float* f)
    {
        return make_uint4(word(f[0], f[1]), word(f[2], f[3]), word(f[4], f[5]), word(f[6], f[7]));
    }
    __device__ static float to_f(__half v) { return __half2float(v); }
    __device__ static __half from_f(float v) { return __float2half_rn(v); }
};

template <>
struct Lanes<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ static float2 two(uint32_t w)
    {
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w);
        return __bfloat1622float2(h);
    }
    __device__ static uint32_t word(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ static void unpack(const uint4& u, float* f)
    {
        float2 a = two(u.x), b = two(u.y), c = two(u.z), d = two(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ static uint4 pack(const float* f)
    {
        return make_uint4(word(f[0], f[1]), word(f[2], f[3]), word(f[4], f[5]), word(f[6], f[7]));
    }
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Unit<T, PACKED>: L fp32 lanes per unit; `raw` is what one load returns.
template <typename T, bool PACKED>
struct Unit;

template <typename T>
struct Unit<T, true> {
    static constexpr int L = Lanes<T>::V;
    using raw = uint4;
    __device__ static raw load(const void* base, uint64_t i)
    {
        return ld_stream16(static_cast<const uint4*>(base) + i);
    }
    __device__ static raw load_cached(const void* base, uint64_t i)
    {
        return ld_cached16(static_cast<const uint4*>(base) + i);
    }
    __device__ static void to_float(const raw& r, float* f) { Lanes<T>::unpack(r, f); }
    __device__ static void store(void* base, uint64_t i, const float* f)
    {
        st16(static_cast<uint4*>(base) + i, Lanes<T>::pack(f));
    }
};

template <typename T>
struct Unit<T, false> {
    static constexpr int L = 1;
    using raw = T;
    __device__ static raw load(const void* base, uint64_t i) { return static_cast<const T*>(base)[i]; }
    __device__ static raw load_cached(const void* base, uint64_t i) { return static_cast<const T*>(base)[i]; }
    __device__ static void to_float(const raw& r, float* f) { f[0] = Lanes<T>::to_f(r); }
    __device__ static void store(void* base, uint64_t i, const float* f)
    {
        static_cast<T*>(base)[i] = Lanes<T>::from_f(f[0]);
    }
};

template <int L>
__device__ __forceinline__ void add_lanes(float* acc, const float* v)
{
#pragma unroll
    for (int l = 0; l < L; ++l)
        acc[l] += v[l];
}

// x = partials[0][i] + ... + partials[R-1][i] in fp32, rank order.  The
// loads are issued before the adds so R loads are in flight at once.
template <typename T, bool PACKED, int R_CT>
__device__ __forceinline__ void sum_partials(const void* const* partials, int R, uint64_t i,
                                             float* x)
{
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;
    if constexpr (R_CT > 0) {
        typename U::raw v[R_CT];
#pragma unroll
        for (int r = 0; r < R_CT; ++r)
            v[r] = U::load(partials[r], i);
        U::to_float(v[0], x);
#pragma unroll
        for (int r = 1; r < R_CT; ++r) {
            float t[L];
            U::to_float(v[r], t);
            add_lanes<L>(x, t);
        }
    } else {
        U::to_float(U::load(partials[0], i), x);
        for (int r = 1; r < R; ++r) {
            float t[L];
            U::to_float(U::load(partials[r], i), t);
            add_lanes<L>(x, t);
        }
    }
}

// ---------------------------------------------------------------------------
// A2 / A3: the R-way sum (one-shot and two-shot work partitions).
//
// Grid (x, y): y indexes the slice (1 slice for one-shot, R rank slices for
// two-shot: the reduce-scatter of twoShotAllReduceKernel; its all-gather is
// void because the slices are written straight into `out`).  Each thread
// handles UNROLL units of its slice, so R * UNROLL 16-byte loads are in
// flight per thread.
// ---------------------------------------------------------------------------
template <typename T, bool PACKED, int R_CT, int UNROLL>
__global__ void __launch_bounds__(kFlatThreads)
k_sum(const SumArgs a)
{
    pdl_enter();
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;
    const uint64_t s_begin = static_cast<uint64_t>(blockIdx.y) * a.slice;
    const uint64_t s_end = min(s_begin + a.slice, a.nunits);
    const uint64_t first = s_begin + static_cast<uint64_t>(blockIdx.x) * (kFlatThreads * UNROLL) + threadIdx.x;

    if constexpr (R_CT > 0) {
        typename U::raw v[UNROLL][R_CT];
#pragma unroll
        for (int r = 0; r < R_CT; ++r) {
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const uint64_t i = first + static_cast<uint64_t>(u) * kFlatThreads;
                if (i < s_end)
                    v[u][r] = U::load(a.partials[r], i);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint64_t i = first + static_cast<uint64_t>(u) * kFlatThreads;
            if (i < s_end) {
                float acc[L];
                U::to_float(v[u][0], acc);
#pragma unroll
                for (int r = 1; r < R_CT; ++r) {
                    float t[L];
                    U::to_float(v[u][r], t);
                    add_lanes<L>(acc, t);
                }
                U::store(a.out, i, acc);
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint64_t i = first + static_cast<uint64_t>(u) * kFlatThreads;
            if (i < s_end) {
                float acc[L];
                sum_partials<T, PACKED, 0>(a.partials, a.R, i, acc);
                U::store(a.out, i, acc);
            }
        }
    }

    // Elements after the last full 16-byte vector (packed path only).
    if (PACKED && a.tail != 0 && blockIdx.x == 0 && blockIdx.y == gridDim.y - 1 && threadIdx.x == 0) {
        const uint64_t e0 = a.nunits * Lanes<T>::V;
        for (uint32_t t = 0; t < a.tail; ++t) {
            float acc;
            Unit<T, false>::to_float(static_cast<const T*>(a.partials[0])[e0 + t], &acc);
            for (int r = 1; r < a.R; ++r)
                acc += Lanes<T>::to_f(static_cast<const T*>(a.partials[r])[e0 + t]);
            static_cast<T*>(a.out)[e0 + t] = Lanes<T>::from_f(acc);
        }
    }
}

// ---------------------------------------------------------------------------
// Row reduction of the sum of squares over the `tpr` threads of one row.
// tpr is a power of two.  Up to a warp: an xor butterfly (every lane ends
// with the same, order-independent value because a+b == b+a exactly).
// Beyond a warp: butterfly per warp, then the warp totals of the row are
// added in warp order from shared memory.  Fixed tree => deterministic.
// Every thread of the block must call this (it may synchronise).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float row_sum(float v, int tpr, float* red)
{
    if (tpr <= 32) {
        for (int off = tpr >> 1; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, off);
        return v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        red[warp] = v;
    __syncthreads();
    const int wpr = tpr >> 5;
    const int first = (warp / wpr) * wpr;
    float s = red[first];
    for (int w = 1; w < wpr; ++w)
        s += red[first + w];
    return s;
}

// Same for a whole block of kFlatThreads threads (two-shot phase 1).
__device__ __forceinline__ float block_sum(float v, float* red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = red[0];
#pragma unroll
    for (int w = 1; w < kFlatThreads / 32; ++w)
        s += red[w];
    return s;
}

__device__ __forceinline__ float inv_rms(float sumsq, int hidden, float eps)
{
    return 1.0f / sqrtf(sumsq / static_cast<float>(hidden) + eps);
}

// ---------------------------------------------------------------------------
// A4: fused one-shot sum + bias + residual + RMSNorm
// (one_shot_all_reduce_norm_kernel -> rms_norm, "allreduce.d2").
//
// `tpr` threads (a power of two, = 32 * warps per token when >= 32) own one
// row; each handles VPT units of it and keeps their fp32 sums x on chip
// between the sum and the normalisation -- in registers (STAGE = false) or
// in shared memory (STAGE = true, which frees the registers for more rows in
// flight per SM).  Either way every input byte is read from HBM once and
// every output byte written once.  residual_out does not depend on the norm:
// with EARLY it is written as soon as x is known (spreading the row's writes
// over its reads), otherwise together with `out` after the row barrier.
// Which order keeps HBM busier depends on the shape (and it changes how the
// compiler schedules the loads), so both are compiled and the launch shape
// picks one.  Blocks hold blockDim.x / tpr rows.
// A thread reads back from shared memory only the values it wrote itself,
// so staging needs no barrier of its own.
// ---------------------------------------------------------------------------
template <typename T, bool PACKED, int R_CT, int VPT, bool STAGE, bool EARLY>
__global__ void __launch_bounds__(STAGE ? 1024 : oneshot_max_threads(VPT * Unit<T, PACKED>::L))
k_fused_oneshot(const FusedArgs a, const int tpr)
{
    pdl_enter();
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;
    __shared__ float red[32];
    extern __shared__ float xs_all[];  // STAGE: [rows per block][L][units_row] fp32

    const int lane_row = threadIdx.x & (tpr - 1);
    const int row_in_block = threadIdx.x / tpr;
    const int row = blockIdx.x * (blockDim.x / tpr) + row_in_block;
    const bool row_ok = row < a.tokens;
    const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
    float* xs = xs_all + static_cast<size_t>(row_in_block) * L * a.units_row;

    float x[STAGE ? 1 : VPT][L];
    typename U::raw wv[STAGE ? 1 : VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = lane_row + k * tpr;
        float* xk = x[STAGE ? 0 : k];
#pragma unroll
        for (int l = 0; l < L; ++l)
            xk[l] = 0.0f;
        if (row_ok && j < a.units_row) {
            sum_partials<T, PACKED, R_CT>(a.partials, a.R, row_off + j, xk);
            float t[L];
            if (a.bias != nullptr) {
                U::to_float(U::load_cached(a.bias, j), t);
                add_lanes<L>(xk, t);
            }
            U::to_float(U::load(a.residual, row_off + j), t);
            add_lanes<L>(xk, t);
            if constexpr (!STAGE)
                wv[k] = U::load_cached(a.weight, j);
            if constexpr (EARLY)
                U::store(a.residual_out, row_off + j, xk);
#pragma unroll
            for (int l = 0; l < L; ++l)
                ss = fmaf(xk[l], xk[l], ss);
            if constexpr (STAGE) {
#pragma unroll
                for (int l = 0; l < L; ++l)
                    xs[l * a.units_row + j] = xk[l];
            }
        }
    }

    ss = row_sum(ss, tpr, red);
    const float inv = inv_rms(ss, a.hidden, a.eps);

#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = lane_row + k * tpr;
        if (row_ok && j < a.units_row) {
            float xk[L], w[L], y[L];
            if constexpr (STAGE) {
#pragma unroll
                for (int l = 0; l < L; ++l)
                    xk[l] = xs[l * a.units_row + j];
                U::to_float(U::load_cached(a.weight, j), w);
            } else {
#pragma unroll
                for (int l = 0; l < L; ++l)
                    xk[l] = x[k][l];
                U::to_float(wv[k], w);
            }
            if constexpr (!EARLY)
                U::store(a.residual_out, row_off + j, xk);
#pragma unroll
            for (int l = 0; l < L; ++l)
                y[l] = xk[l] * inv * w[l];
            U::store(a.out, row_off + j, y);
        }
    }
}

// ---------------------------------------------------------------------------
// A4 for few rows: one row split across a thread-block cluster of C blocks.
// With one block per row, a single SM streams the whole row (R + 1 inputs of
// hidden elements), which bounds decode latency.  Here block c of the
// cluster of row t owns the contiguous slice [c*S, (c+1)*S) of the row's
// units (S = ceil(units_row / C)), keeps its x in registers, and reduces its
// slice's sum of squares; the C partial sums are exchanged through
// distributed shared memory between two cluster barriers and added in
// cluster-rank order (fixed, so deterministic).  The second barrier keeps
// every block's shared memory alive until all have read it.  Cluster
// barriers are hardware barriers over co-scheduled blocks: no spin loop.
// Packed path; grid = tokens * C blocks of `blockDim.x` threads, cluster (C).
// ---------------------------------------------------------------------------
template <typename T, int R_CT, int VPT>
__global__ void __launch_bounds__(oneshot_max_threads(VPT * Lanes<T>::V))
k_fused_oneshot_cluster(const FusedArgs a, const int csize)
{
    pdl_enter();
    namespace cg = cooperative_groups;
    using U = Unit<T, true>;
    constexpr int L = U::L;
    __shared__ float red[32];
    __shared__ float part;  // this block's partial sum of squares

    cg::cluster_group cluster = cg::this_cluster();
    const int crank = static_cast<int>(cluster.block_rank());
    const int row = static_cast<int>(blockIdx.x) / csize;
    const int slice = (a.units_row + csize - 1) / csize;
    const int j_begin = crank * slice;
    const int j_end = min(j_begin + slice, a.units_row);
    const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
    const int tpb = static_cast<int>(blockDim.x);

    float x[VPT][L];
    typename U::raw wv[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j_begin + static_cast<int>(threadIdx.x) + k * tpb;
#pragma unroll
        for (int l = 0; l < L; ++l)
            x[k][l] = 0.0f;
        if (j < j_end) {
            sum_partials<T, true, R_CT>(a.partials, a.R, row_off + j, x[k]);
            float t[L];
            if (a.bias != nullptr) {
                U::to_float(U::load_cached(a.bias, j), t);
                add_lanes<L>(x[k], t);
            }
            U::to_float(U::load(a.residual, row_off + j), t);
            add_lanes<L>(x[k], t);
            wv[k] = U::load_cached(a.weight, j);
            if (a.early_residual)
                U::store(a.residual_out, row_off + j, x[k]);
#pragma unroll
            for (int l = 0; l < L; ++l)
                ss = fmaf(x[k][l], x[k][l], ss);
        }
    }
    ss = row_sum(ss, tpb, red);
    if (threadIdx.x == 0)
        part = ss;
    cluster.sync();
    float tot = 0.0f;
    for (int c = 0; c < csize; ++c)
        tot += *cluster.map_shared_rank(&part, c);
    const float inv = inv_rms(tot, a.hidden, a.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j_begin + static_cast<int>(threadIdx.x) + k * tpb;
        if (j < j_end) {
            if (!a.early_residual)
                U::store(a.residual_out, row_off + j, x[k]);
            float w[L], y[L];
            U::to_float(wv[k], w);
#pragma unroll
            for (int l = 0; l < L; ++l)
                y[l] = x[k][l] * inv * w[l];
            U::store(a.out, row_off + j, y);
        }
    }
    cluster.sync();  // no block leaves while another may still read its `part`
}

// ---------------------------------------------------------------------------
// A4, persistent form for many rows: one row per block iteration, blocks
// stride over the rows.  The row's fp32 sums are staged in shared memory; the
// first units of the NEXT row (its partials and residual) are loaded before
// the row-reduction barrier, so loads stay in flight while the block waits
// at the barrier and writes the current row.  Packed path, R known at
// compile time, tpr == blockDim.x.
// ---------------------------------------------------------------------------
template <typename T, int R_CT, int VPT>
__global__ void __launch_bounds__(kMaxPersistThreads)
k_fused_oneshot_persist(const FusedArgs a)
{
    pdl_enter();
    using U = Unit<T, true>;
    constexpr int L = U::L;
    static_assert(R_CT > 0, "persistent one-shot needs R at compile time");
    __shared__ float red[2][32];
    extern __shared__ float xs[];  // [L][units_row] fp32

    const int tpr = blockDim.x;
    const int j0 = threadIdx.x;
    const bool j0_ok = j0 < a.units_row;
    uint4 pre[R_CT + 1];  // units j0 of the next row: R partials and the residual
    int row = blockIdx.x;
    if (row < a.tokens && j0_ok) {
        const uint64_t off = static_cast<uint64_t>(row) * a.units_row + j0;
#pragma unroll
        for (int r = 0; r < R_CT; ++r)
            pre[r] = U::load(a.partials[r], off);
        pre[R_CT] = U::load(a.residual, off);
    }
    int parity = 0;
    for (; row < a.tokens; row += gridDim.x, parity ^= 1) {
        const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * tpr;
            if (j < a.units_row) {
                float x[L], t[L];
                if (k == 0) {
                    U::to_float(pre[0], x);
#pragma unroll
                    for (int r = 1; r < R_CT; ++r) {
                        U::to_float(pre[r], t);
                        add_lanes<L>(x, t);
                    }
                } else {
                    sum_partials<T, true, R_CT>(a.partials, R_CT, row_off + j, x);
                }
                if (a.bias != nullptr) {
                    U::to_float(U::load_cached(a.bias, j), t);
                    add_lanes<L>(x, t);
                }
                U::to_float(k == 0 ? pre[R_CT] : U::load(a.residual, row_off + j), t);
                add_lanes<L>(x, t);
                if (a.early_residual)
                    U::store(a.residual_out, row_off + j, x);
#pragma unroll
                for (int l = 0; l < L; ++l) {
                    ss = fmaf(x[l], x[l], ss);
                    xs[l * a.units_row + j] = x[l];
                }
            }
        }
        const int next = row + gridDim.x;
        if (next < a.tokens && j0_ok) {
            const uint64_t off = static_cast<uint64_t>(next) * a.units_row + j0;
#pragma unroll
            for (int r = 0; r < R_CT; ++r)
                pre[r] = U::load(a.partials[r], off);
            pre[R_CT] = U::load(a.residual, off);
        }
        // Row reduction with a double-buffered scratch: a warp that runs ahead
        // into the next row writes the other buffer.
        ss = row_sum(ss, tpr, red[parity]);
        const float inv = inv_rms(ss, a.hidden, a.eps);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * tpr;
            if (j < a.units_row) {
                float x[L], w[L], y[L];
#pragma unroll
                for (int l = 0; l < L; ++l)
                    x[l] = xs[l * a.units_row + j];
                U::to_float(U::load_cached(a.weight, j), w);
                if (!a.early_residual)
                    U::store(a.residual_out, row_off + j, x);
#pragma unroll
                for (int l = 0; l < L; ++l)
                    y[l] = x[l] * inv * w[l];
                U::store(a.out, row_off + j, y);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// RMSNorm of x rows on its own (rms_norm_kernel_launcher -> rms_norm_kernel,
// "allreduce.d2": the norm that follows a plain all-reduce).  `tpr` threads
// own a row and each keeps VPT units of it in registers across the row
// reduction, so x is read from HBM once and out written once.  Unlike the
// fused kernels, the row here is the input itself: the registers hold the
// packed 16-byte vectors as loaded (half the registers of fp32 values for
// 16-bit types) and the second pass unpacks them again, exactly; the weight
// is loaded only in the second pass (it is small and cache-resident).  Fewer
// registers per row mean more rows, and more bytes, in flight per SM.
// x is a.partials[0]; out may alias x.
// ---------------------------------------------------------------------------
template <typename T, bool PACKED, int VPT>
__global__ void __launch_bounds__(norm_max_threads(PACKED, VPT), norm_min_blocks(PACKED, VPT))
k_rmsnorm(const FusedArgs a, const int tpr)
{
    pdl_enter();
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;
    __shared__ float red[32];

    const int lane_row = threadIdx.x & (tpr - 1);
    const int row = blockIdx.x * (blockDim.x / tpr) + static_cast<int>(threadIdx.x) / tpr;
    const bool row_ok = row < a.tokens;
    const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;

    typename U::raw xr[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = lane_row + k * tpr;
        if (row_ok && j < a.units_row)
            xr[k] = U::load(a.partials[0], row_off + j);
    }
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = lane_row + k * tpr;
        if (row_ok && j < a.units_row) {
            float x[L];
            U::to_float(xr[k], x);
#pragma unroll
            for (int l = 0; l < L; ++l)
                ss = fmaf(x[l], x[l], ss);
        }
    }
    ss = row_sum(ss, tpr, red);
    const float inv = inv_rms(ss, a.hidden, a.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = lane_row + k * tpr;
        if (row_ok && j < a.units_row) {
            float x[L], w[L], y[L];
            U::to_float(xr[k], x);
            U::to_float(U::load_cached(a.weight, j), w);
#pragma unroll
            for (int l = 0; l < L; ++l)
                y[l] = x[l] * inv * w[l];
            U::store(a.out, row_off + j, y);
        }
    }
}

// ---------------------------------------------------------------------------
// A6: two-shot fused phase 1 (twoShotAllReduceKernel in the fused route of
// AllReduceNormKernelLaunch, "allreduce.d2").  Block b owns chunk
// (b % nchunk) of row (b / nchunk): it writes the pre-norm sum to
// residual_out and the chunk's fp32 sum of squares (of the UNROUNDED x) to
// the workspace.
// ---------------------------------------------------------------------------
template <typename T, bool PACKED, int R_CT>
__global__ void __launch_bounds__(kFlatThreads)
k_twoshot_phase1(const FusedArgs a)
{
    pdl_enter();
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;
    __shared__ float red[kFlatThreads / 32];

    const uint64_t b = blockIdx.x;
    const int row = static_cast<int>(b / a.nchunk);
    const int chunk = static_cast<int>(b % a.nchunk);
    const int c_begin = chunk * a.chunk_units;
    const int c_end = min(c_begin + a.chunk_units, a.units_row);
    const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;

    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kChunkVPT; ++k) {
        const int j = c_begin + k * kFlatThreads + static_cast<int>(threadIdx.x);
        if (j < c_end) {
            float x[L], t[L];
            sum_partials<T, PACKED, R_CT>(a.partials, a.R, row_off + j, x);
            if (a.bias != nullptr) {
                U::to_float(U::load_cached(a.bias, j), t);
                add_lanes<L>(x, t);
            }
            U::to_float(U::load(a.residual, row_off + j), t);
            add_lanes<L>(x, t);
            U::store(a.residual_out, row_off + j, x);
#pragma unroll
            for (int l = 0; l < L; ++l)
                ss = fmaf(x[l], x[l], ss);
        }
    }
    ss = block_sum(ss, red);
    if (threadIdx.x == 0)
        a.sumsq[b] = ss;
}

// ---------------------------------------------------------------------------
// A7: two-shot fused phase 2 (rms_norm_kernel, "allreduce.d2").  Block b
// owns one (row, chunk) as in phase 1, but blocks walk the rows from the
// last to the first: the rows phase 1 wrote last are the likeliest to still
// sit in L2.  The row's chunk sums are added in chunk order.
// ---------------------------------------------------------------------------
template <typename T, bool PACKED>
__global__ void __launch_bounds__(kFlatThreads)
k_twoshot_phase2(const FusedArgs a)
{
    pdl_enter();
    using U = Unit<T, PACKED>;
    constexpr int L = U::L;

    const uint64_t b = static_cast<uint64_t>(gridDim.x) - 1 - blockIdx.x;
    const int row = static_cast<int>(b / a.nchunk);
    const int chunk = static_cast<int>(b % a.nchunk);
    const int c_begin = chunk * a.chunk_units;
    const int c_end = min(c_begin + a.chunk_units, a.units_row);
    const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;

    const float* ss_row = a.sumsq + static_cast<uint64_t>(row) * a.nchunk;
    float ss = ss_row[0];
    for (int c = 1; c < a.nchunk; ++c)
        ss += ss_row[c];
    const float inv = inv_rms(ss, a.hidden, a.eps);

#pragma unroll
    for (int k = 0; k < kChunkVPT; ++k) {
        const int j = c_begin + k * kFlatThreads + static_cast<int>(threadIdx.x);
        if (j < c_end) {
            float x[L], w[L], y[L];
            U::to_float(U::load(a.residual_out, row_off + j), x);
            U::to_float(U::load_cached(a.weight, j), w);
#pragma unroll
            for (int l = 0; l < L; ++l)
                y[l] = x[l] * inv * w[l];
            U::store(a.out, row_off + j, y);
        }
    }
}

}  // namespace ar
