// ar_tma.cuh -- the one-shot fused sum + bias + residual + RMSNorm fed by
// bulk asynchronous copies (the sm_90+ TMA bulk path) into a shared-memory
// ring, for sm_103a.
//
// Why: the register-fed one-shot kernel keeps every byte in flight in a
// register, so its bytes in flight per SM are capped by the register file
// and by occupancy, and a block that reaches its row barrier stops loading.
// Here one producer lane per block streams row chunks of all R partials and
// the residual into shared memory with cp.async.bulk (16-byte granular, no
// register cost) while the consumer warps sum, normalise and store.  The
// ring holds ~200 KB per SM in flight, and loads for later rows continue
// while the consumers wait at a row barrier.
//
// The residual input and the residual_out output are optional (both absent
// for the norm on its own: R = 1 partial holding x, no bias).
//
// Block = NC consumer threads (NC = vectors per chunk, a multiple of 32) plus
// one producer warp.  A row of units_row 16-byte vectors is split into
// ceil(units_row / NC) <= CPR chunks; consumer thread t owns vector
// c * NC + t of chunk c and keeps its fp32 sum in registers until the row's
// inverse RMS is known, so every input byte is read from HBM once and every
// output byte written once.  Blocks are persistent and stride over rows.
//
// Waits are bounded: an mbarrier wait gives up after kWaitLimitNs of
// %globaltimer time, counts the event in g_wait_timeouts (read by the host
// through take_wait_timeouts), and the block winds down -- a consumer warp
// that gave up releases no further slot, the consumers agree at the row
// barrier to stop, the producer's own wait for a release runs out, and it
// waits (again bounded) for the copies it issued before it exits.
#pragma once

#include "ar_kernels.cuh"

namespace ar {

// Bounded-wait limit: a legitimate wait here lasts microseconds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Bounded waits that gave up, in this translation unit's kernels.
static __device__ unsigned int g_wait_timeouts;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the asynchronous (copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test_parity(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase of `bar` with parity `parity` has completed; false
// if that did not happen within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_test_parity(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test_parity(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return true;
}

// Bulk copy global -> this block's shared memory; completion is counted in
// bytes on `bar`.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Barrier 1 over the `count` consumer threads; returns the OR of `pred`
// over them.
__device__ __forceinline__ bool consumers_sync_or(uint32_t count, bool pred)
{
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any)
        : "r"(static_cast<uint32_t>(pred)), "r"(count)
        : "memory");
    return any != 0;
}

template <typename T, int R_CT, int CPR>
__global__ void __launch_bounds__(tma_max_consumers(CPR) + 32)
k_fused_oneshot_tma(const FusedArgs a, const int stages)
{
    using U = Unit<T, true>;
    constexpr int L = U::L;
    const int R = R_CT > 0 ? R_CT : a.R;
    const bool has_res = a.residual != nullptr;
    const int inputs = R + (has_res ? 1 : 0);           // streamed tensors
    const int nc = static_cast<int>(blockDim.x) - 32;   // consumer threads = vectors per chunk
    const int nchunk = (a.units_row + nc - 1) / nc;     // <= CPR (checked by the host)
    const size_t slot_vecs = static_cast<size_t>(inputs) * nc;

    extern __shared__ __align__(128) unsigned char smem[];
    uint4* ring = reinterpret_cast<uint4*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(stages) * slot_vecs * 16);
    uint64_t* empty = full + stages;
    float* red = reinterpret_cast<float*>(empty + stages);

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], static_cast<uint32_t>(nc / 32));  // one arrival per consumer warp
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_enter();  // shared-memory set-up above overlaps the previous kernel

    if (tid >= nc) {
        // Producer warp: one lane issues every copy.
        if (tid != nc)
            return;
        uint32_t it = 0;  // copies-stages issued so far
        int s = 0;        // ring slot of stage `it`
        uint32_t ph = 0;  // parity of that slot's use: (it / stages) & 1
        bool ok = true;
        for (int row = blockIdx.x; row < a.tokens && ok; row += gridDim.x) {
            const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
            for (int c = 0; c < nchunk; ++c) {
                // Reusing a slot: wait until the consumers released its previous use.
                if (it >= static_cast<uint32_t>(stages) && !mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                    ok = false;
                    break;
                }
                const int j0 = c * nc;
                const uint32_t bytes = static_cast<uint32_t>(min(nc, a.units_row - j0)) * 16u;
                // a.stall_stage (tests only, 0 otherwise) leaves one stage unarmed,
                // so the waits on it run out and the abort path below is exercised.
                if (static_cast<uint32_t>(a.stall_stage) != it + 1u) {
                    mbar_arrive_expect_tx(&full[s], bytes * static_cast<uint32_t>(inputs));
                    uint4* dst = ring + static_cast<size_t>(s) * slot_vecs;
                    for (int r = 0; r < R; ++r)
                        bulk_copy_g2s(dst + static_cast<size_t>(r) * nc,
                                      static_cast<const uint4*>(a.partials[r]) + row_off + j0, bytes, &full[s]);
                    if (has_res)
                        bulk_copy_g2s(dst + static_cast<size_t>(R) * nc,
                                      static_cast<const uint4*>(a.residual) + row_off + j0, bytes, &full[s]);
                }
                ++it;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok)
            atomicAdd(&g_wait_timeouts, 1u);
        // The block must not exit with copies into its shared memory in
        // flight: wait for the last issued use of every slot to land.
        const uint32_t first = it > static_cast<uint32_t>(stages) ? it - stages : 0u;
        for (uint32_t k = first; k < it; ++k)
            if (!mbar_wait_bounded(&full[k % stages], (k / stages) & 1u))
                atomicAdd(&g_wait_timeouts, 1u);
        return;
    }

    // Consumers.  Weight and bias vectors of this thread's columns are the
    // same for every row: keep them in registers.
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nc >> 5;
    uint4 wv[CPR], bv[CPR];
#pragma unroll
    for (int c = 0; c < CPR; ++c) {
        const int j = c * nc + tid;
        wv[c] = make_uint4(0u, 0u, 0u, 0u);
        bv[c] = make_uint4(0u, 0u, 0u, 0u);
        if (c < nchunk && j < a.units_row) {
            wv[c] = U::load_cached(a.weight, j);
            if (a.bias != nullptr)
                bv[c] = U::load_cached(a.bias, j);
        }
    }

    int s = 0;        // ring slot of the next stage
    uint32_t ph = 0;  // parity of that slot's use
    bool gave_up = false;
    int parity = 0;   // row-reduction scratch buffer of this row
    for (int row = blockIdx.x; row < a.tokens; row += gridDim.x, parity ^= 1) {
        const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
        float x[CPR][L];
        float ss = 0.0f;
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
#pragma unroll
            for (int l = 0; l < L; ++l)
                x[c][l] = 0.0f;
            if (c < nchunk) {
                if (!gave_up && !mbar_wait_bounded(&full[s], ph))
                    gave_up = true;
                // The warp gives up as one, so lane 0's release below speaks for it.
                gave_up = __any_sync(0xffffffffu, gave_up);
                const int j = c * nc + tid;
                if (!gave_up && j < a.units_row) {
                    const uint4* src = ring + static_cast<size_t>(s) * slot_vecs + tid;
                    float t[L];
                    U::to_float(src[0], x[c]);
                    for (int r = 1; r < R; ++r) {
                        U::to_float(src[static_cast<size_t>(r) * nc], t);
                        add_lanes<L>(x[c], t);
                    }
                    if (a.bias != nullptr) {
                        U::to_float(bv[c], t);
                        add_lanes<L>(x[c], t);
                    }
                    if (has_res) {
                        U::to_float(src[static_cast<size_t>(R) * nc], t);
                        add_lanes<L>(x[c], t);
                    }
                    if (a.early_residual && a.residual_out != nullptr)
                        U::store(a.residual_out, row_off + j, x[c]);
#pragma unroll
                    for (int l = 0; l < L; ++l)
                        ss = fmaf(x[c][l], x[c][l], ss);
                }
                // The warp is done with the slot: its lanes' shared-memory reads
                // are ordered before lane 0's (releasing) arrival by __syncwarp.
                // A warp that gave up releases nothing more: the copies of a
                // stage it did not see complete may still be landing, and the
                // producer must not re-arm that slot; its own bounded wait for
                // the release ends its loop instead.
                __syncwarp();
                if (lane == 0 && !gave_up)
                    mbar_arrive(&empty[s]);
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // Row reduction: warp butterfly, then the warp totals in warp order.
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
        float* rp = red + parity * 32;
        if (lane == 0)
            rp[warp] = ss;
        if (consumers_sync_or(static_cast<uint32_t>(nc), gave_up)) {
            if (tid == 0)
                atomicAdd(&g_wait_timeouts, 1u);
            return;
        }
        float tot = rp[0];
        for (int w = 1; w < nwarps; ++w)
            tot += rp[w];
        const float inv = inv_rms(tot, a.hidden, a.eps);
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
            const int j = c * nc + tid;
            if (c < nchunk && j < a.units_row) {
                if (!a.early_residual && a.residual_out != nullptr)
                    U::store(a.residual_out, row_off + j, x[c]);
                float w[L], y[L];
                U::to_float(wv[c], w);
#pragma unroll
                for (int l = 0; l < L; ++l)
                    y[l] = x[c][l] * inv * w[l];
                U::store(a.out, row_off + j, y);
            }
        }
    }
}

}  // namespace ar
