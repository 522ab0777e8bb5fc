// ar_lamport.cuh -- the Lamport-style one-shot fused sum + bias + residual +
// RMSNorm (lamport_style_one_shot_all_reduce_norm_kernel_launcher ->
// lamport_style_one_shot_all_reduce_norm_kernel, "allreduce.d2"), for one
// GPU, sm_103a.
//
// The protocol.  Every rank writes its partial into a communication buffer
// that holds an "empty" marker wherever nothing has been written yet: the
// negative zero of the element type, a value the writers never store (a
// -0.0 lane of a partial is written as +0.0, the same number in every sum
// here; only the sign of an exact-zero result can change).  The reducer
// needs no barrier and no flag: it re-reads an element of the buffer until
// it is not the marker, which proves that this element has arrived, and once
// it has used the element it writes the marker back, so the buffer is empty
// again for the next call.  The data is its own ready flag.
//
// On one GPU the R ranks' writes are emulated inside the same launch.  The
// buffer holds one slot per rank (after the blocks' progress words); slot
// r = [slot_rows][units_row] 16-byte vectors at r * slot_rows * units_row,
// and row k of the call lives in ring
// row k mod ring_rows of every slot (ring_rows <= slot_rows: two steps of the
// grid's row groups, or all tokens when they are fewer).  Blocks push
// vectors of all R partials into their slots (the peers' NVLink writes of
// the multi-GPU protocol) and reduce rows as the register-resident one-shot
// kernel does -- tpr threads per row, VPT vectors per thread, fp32 sums in
// rank order, bias, residual, the row's sum of squares over a fixed tree --
// reading each partial from its slot instead of from the partial.  The rows
// a block reduces were pushed by another block, so blocks wait on one
// another: the launch is cooperative (all of its blocks resident at once, or
// the launch fails), so every push it waits for is made by a block that is
// already running.
//
// Ring reuse.  A ring row is used again, by row k + ring_rows, once row k
// has been reduced.  Each block publishes the last step it has finished
// reducing (a release store after a block barrier); before pushing into a
// ring row used earlier in the call, a block waits (acquire) until the block
// that reduces that ring row has finished the step that last used it, so it
// never overwrites an element not yet taken.  The reducer of row k +
// ring_rows is the very thread that reduced row k (the schedule below keeps
// slot position -> block fixed), so it cannot mistake row k's elements for
// row k + ring_rows's: its own write of the marker comes first in program
// order.  The ring is two steps deep, so a pusher waits only on a reduce two
// steps back, and the whole ring (tens of MB at prefill size) stays in L2
// instead of the buffer streaming through DRAM.
//
// Memory ordering.  Pushes are st.relaxed.gpu and polls ld.relaxed.gpu, both
// of 16 bytes: each 2- or 4-byte element is written once, from the marker to
// its value, and read until it is no longer the marker, so a vector read
// part-way through a push shows some elements still empty and is read
// again.  No fence is needed: nothing but the element itself is published.
// The marker is written back with a relaxed store by the one thread that read
// the element: a pusher that reuses the ring row observes it with a relaxed
// poll, and per-element coherence orders the marker (and the read before it)
// before the new push.  The next call's pushes follow the kernel boundary.
//
// Waits are bounded: a poll that has not seen its element after
// kWaitLimitNs gives up, counts the event in g_wait_timeouts (read by the
// host through take_wait_timeouts) and the thread polls no more in this
// launch; its outputs are then incomplete, and the buffer may hold elements
// pushed after the give-up, so it has to be emptied again (filled with the
// marker) before the next call.
#pragma once

#include "ar_tma.cuh"

namespace ar {

// The empty marker, as the 32-bit word of two 16-bit lanes or one fp32 lane.
template <typename T>
struct LamportMarker {
    static constexpr uint32_t word = 0x80008000u;  // -0.0 in both halves (fp16, bf16)
};
template <>
struct LamportMarker<float> {
    static constexpr uint32_t word = 0x80000000u;  // -0.0f
};

__device__ __forceinline__ uint4 ld_relaxed16(const void* p)
{
    uint4 r;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_relaxed16(void* p, uint4 v)
{
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Per 32-bit word: all-ones in each lane equal to the marker, zero elsewhere.
template <typename T>
__device__ __forceinline__ uint32_t marker_lanes(uint32_t w)
{
    if constexpr (sizeof(T) == 4)
        return w == LamportMarker<T>::word ? 0xffffffffu : 0u;
    else
        return __vcmpeq2(w, LamportMarker<T>::word);
}

// True if any lane of the vector still holds the marker (not yet pushed).
template <typename T>
__device__ __forceinline__ bool lamport_pending(const uint4& v)
{
    return (marker_lanes<T>(v.x) | marker_lanes<T>(v.y) | marker_lanes<T>(v.z) | marker_lanes<T>(v.w)) != 0u;
}

// The vector as a writer pushes it: every -0.0 lane becomes +0.0 (clearing
// the sign bit of a lane equal to the marker leaves all-zero bits).
template <typename T>
__device__ __forceinline__ uint4 lamport_clean(uint4 v)
{
    v.x &= ~marker_lanes<T>(v.x);
    v.y &= ~marker_lanes<T>(v.y);
    v.z &= ~marker_lanes<T>(v.z);
    v.w &= ~marker_lanes<T>(v.w);
    return v;
}

template <typename T>
__device__ __forceinline__ uint4 lamport_empty()
{
    constexpr uint32_t m = LamportMarker<T>::word;
    return make_uint4(m, m, m, m);
}

// Re-reads *p until no lane is the marker; `v` is a first read of it.
// Bounded: after kWaitLimitNs the thread gives up (and polls no more).
template <typename T>
__device__ __forceinline__ uint4 lamport_poll(const uint4* p, uint4 v, bool& gave_up)
{
    if (!lamport_pending<T>(v) || gave_up)
        return v;
    const unsigned long long t0 = global_ns();
    do {
        __nanosleep(32);
        v = ld_relaxed16(p);
        if (!lamport_pending<T>(v))
            return v;
    } while (global_ns() - t0 <= kWaitLimitNs);
    gave_up = true;
    atomicAdd(&g_wait_timeouts, 1u);
    return v;
}

// x = slot 0 + ... + slot R-1 of vector i in fp32, rank order, each read
// once it has arrived and then emptied again.  The first reads of RG ranks
// (all R by default) are issued before any is checked, so RG loads are in
// flight at once; fewer keep fewer registers.
template <typename T, int R_CT, int RG = R_CT>
__device__ __forceinline__ void lamport_take(uint4* lam, uint64_t slot_units, int R, uint64_t i, float* x,
                                             bool& gave_up)
{
    constexpr int L = Lanes<T>::V;
    if constexpr (R_CT > 0) {
        static_assert(RG > 0 && R_CT % RG == 0, "whole groups of ranks");
        if constexpr (RG == R_CT) {
            uint4 v[R_CT];
#pragma unroll
            for (int r = 0; r < R_CT; ++r)
                v[r] = ld_relaxed16(lam + r * slot_units + i);
#pragma unroll
            for (int r = 0; r < R_CT; ++r)
                v[r] = lamport_poll<T>(lam + r * slot_units + i, v[r], gave_up);
#pragma unroll
            for (int r = 0; r < R_CT; ++r)
                st_relaxed16(lam + r * slot_units + i, lamport_empty<T>());
            Lanes<T>::unpack(v[0], x);
#pragma unroll
            for (int r = 1; r < R_CT; ++r) {
                float t[L];
                Lanes<T>::unpack(v[r], t);
                add_lanes<L>(x, t);
            }
            return;
        }
#pragma unroll
        for (int r0 = 0; r0 < R_CT; r0 += RG) {
            uint4 v[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r)
                v[r] = ld_relaxed16(lam + (r0 + r) * slot_units + i);
#pragma unroll
            for (int r = 0; r < RG; ++r)
                v[r] = lamport_poll<T>(lam + (r0 + r) * slot_units + i, v[r], gave_up);
#pragma unroll
            for (int r = 0; r < RG; ++r)
                st_relaxed16(lam + (r0 + r) * slot_units + i, lamport_empty<T>());
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                if (r0 + r == 0) {
                    Lanes<T>::unpack(v[r], x);
                } else {
                    float t[L];
                    Lanes<T>::unpack(v[r], t);
                    add_lanes<L>(x, t);
                }
            }
        }
    } else {
        for (int r = 0; r < R; ++r) {
            uint4* p = lam + r * slot_units + i;
            const uint4 v = lamport_poll<T>(p, ld_relaxed16(p), gave_up);
            st_relaxed16(p, lamport_empty<T>());
            float t[L];
            Lanes<T>::unpack(v, t);
            if (r == 0) {
#pragma unroll
                for (int l = 0; l < L; ++l)
                    x[l] = t[l];
            } else {
                add_lanes<L>(x, t);
            }
        }
    }
}

__device__ __forceinline__ uint32_t ld_relaxed32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_relaxed32(uint32_t* p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The exchange area (kLamportRowWords words per row after the R slots) of a
// row split over csize blocks: word c holds block c's partial sum of squares
// and word kLamportMaxSplit counts the blocks that have read all of them;
// both start as the marker word.
//
// Block c's share of a split row's sum of squares in, the row's total out
// (added in block order, so every block of the row gets the same value).
// Called by the 32 lanes of one warp, all holding the same share; lane k
// waits for share k, so the csize waits overlap.  A share is never the
// marker: it is a sum of squares that starts at +0.0 (>= +0.0 or NaN),
// while the marker word is -0.0f (fp32) or a negative fp32 bit pattern
// (16-bit types).  The last of the csize blocks to count itself writes the
// marker back over the shares and the counter: its acquire-release add
// orders those stores after every other block's reads, which precede that
// block's own (release) add.
template <typename T>
__device__ __forceinline__ float lamport_exchange(uint32_t* xr, int c, int csize, float share, bool& gave_up)
{
    constexpr uint32_t m = LamportMarker<T>::word;
    const int lane = static_cast<int>(threadIdx.x & 31u);
    if (lane == c)
        st_relaxed32(xr + c, __float_as_uint(share));
    uint32_t v = m;
    if (lane < csize) {
        v = ld_relaxed32(xr + lane);
        if (v == m && !gave_up) {
            const unsigned long long t0 = global_ns();
            do {
                __nanosleep(32);
                v = ld_relaxed32(xr + lane);
            } while (v == m && global_ns() - t0 <= kWaitLimitNs);
            if (v == m) {
                gave_up = true;
                atomicAdd(&g_wait_timeouts, 1u);
            }
        }
    }
    float tot = 0.0f;
    for (int k = 0; k < csize; ++k) {
        const uint32_t vk = __shfl_sync(0xffffffffu, v, k);
        tot += vk == m ? 0.0f : __uint_as_float(vk);
    }
    __syncwarp();  // the lanes' reads are ordered before lane 0's add
    if (lane == 0) {
        uint32_t before;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(before)
                     : "l"(xr + kLamportMaxSplit)
                     : "memory");
        if (before == m + static_cast<uint32_t>(csize) - 1u) {
            for (int k = 0; k < csize; ++k)
                xr[k] = m;
            xr[kLamportMaxSplit] = m;
        }
    }
    return tot;
}

// Pushes vector i of every partial (at element index `src` of each partial)
// into its rank's slot at ring index `dst` (skip_rank >= 0: not that
// rank's).
template <typename T, int R_CT>
__device__ __forceinline__ void lamport_push(const FusedArgs& a, uint4* lam, uint64_t slot_units, int R, uint64_t src,
                                             uint64_t dst, int skip_rank)
{
    if constexpr (R_CT > 0) {
        uint4 v[R_CT];
#pragma unroll
        for (int r = 0; r < R_CT; ++r)
            v[r] = ld_stream16(static_cast<const uint4*>(a.partials[r]) + src);
#pragma unroll
        for (int r = 0; r < R_CT; ++r)
            if (r != skip_rank)
                st_relaxed16(lam + r * slot_units + dst, lamport_clean<T>(v[r]));
    } else {
        for (int r = 0; r < R; ++r) {
            const uint4 v = ld_stream16(static_cast<const uint4*>(a.partials[r]) + src);
            if (r != skip_rank)
                st_relaxed16(lam + r * slot_units + dst, lamport_clean<T>(v));
        }
    }
}

// Progress of the blocks through the steps of one call: word b holds (call
// epoch << 32) | (the last step block b has finished reducing).  The host
// gives every call its own epoch in [1, 2^31), so words left by earlier calls
// (or by the marker fill, whose high word has its top bit set) never match.
__device__ __forceinline__ void lamport_publish(unsigned long long* w, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(w), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long lamport_progress(const unsigned long long* w)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(w) : "memory");
    return v;
}

// Waits (bounded) until word *w shows this call's epoch and a step >= `step`.
__device__ __forceinline__ void lamport_wait_progress(const unsigned long long* w, uint32_t epoch, uint32_t step,
                                                      bool& gave_up)
{
    auto done = [&](unsigned long long v) {
        return static_cast<uint32_t>(v >> 32) == epoch && static_cast<uint32_t>(v) >= step;
    };
    if (gave_up || done(lamport_progress(w)))
        return;
    const unsigned long long t0 = global_ns();
    do {
        __nanosleep(64);
        if (done(lamport_progress(w)))
            return;
    } while (global_ns() - t0 <= kWaitLimitNs);
    gave_up = true;
    atomicAdd(&g_wait_timeouts, 1u);
}

// The fused kernel.  Packed path only (16-byte vectors).
//
// Work comes in groups.  csize == 1: a group is blockDim.x / tpr rows, tpr
// threads a row, VPT vectors a thread.  csize > 1: a group is one slice of a
// row split over csize blocks (consecutive groups), slice c = vectors
// [c*S, (c+1)*S) with S = ceil(units_row / csize), all blockDim.x == tpr
// threads on it; the slices' sums of squares meet in the exchange area
// through the same protocol as the data.
//
// Schedule.  The groups are dealt out in steps of G = gridDim.x: in a step,
// block b pushes the vectors of the group at position b (the very vectors
// its threads would reduce), then reduces the group at position (b + 1) mod
// G, which its neighbour pushes in the same step; a position the (short)
// last step does not reach is skipped.  So position p is always pushed by
// block p and reduced by block p - 1 (mod G), in every step -- which keeps
// each ring row's reducer the same thread (see "Ring reuse" above).  A
// reduce waits only for pushes (and split-row shares) of its own step and a
// push only for the reduce of its ring row two steps back, so the waits
// cannot form a cycle; G is a multiple of csize, so no split row straddles
// two steps.  A step's pushed vectors are polled while they are still in
// L2.  (Pushing one step ahead of the reduce measured slower: with two
// steps of pushes in flight beside the partials' stream, more of the ring's
// lines left L2 before they were polled.)
// `slot_rows` is the rows each rank's slot holds (the buffer layout, set by
// the host); `skip_rank` >= 0 leaves that rank's pushes out (tests of the
// bounded waits only; -1 = none).
template <typename T, int R_CT, int VPT>
__global__ void __launch_bounds__(lamport_max_threads(VPT * Lanes<T>::V))
k_fused_lamport(const FusedArgs a, uint4* lam_buffer, const int tpr, const int csize, const int skip_rank,
                const int slot_rows, const uint32_t epoch, const int ring_steps)
{
    pdl_enter();
    using U = Unit<T, true>;
    constexpr int L = U::L;
    __shared__ float red[2][32];
    __shared__ float tot_s[2];
    uint4* lam = lam_buffer;
    const int R = R_CT > 0 ? R_CT : a.R;
    const uint64_t slot_units = static_cast<uint64_t>(slot_rows) * a.units_row;
    const bool split = csize > 1;
    const int rows = split ? 1 : static_cast<int>(blockDim.x) / tpr;
    const int lane = split ? static_cast<int>(threadIdx.x) : static_cast<int>(threadIdx.x & (tpr - 1));
    const int row_in_block = split ? 0 : static_cast<int>(threadIdx.x) / tpr;
    const int slice = split ? (a.units_row + csize - 1) / csize : a.units_row;
    const int groups = split ? a.tokens * csize : (a.tokens + rows - 1) / rows;
    const int G = static_cast<int>(gridDim.x);
    // ring_steps steps of groups, in rows (never more than the slot holds).
    const long long ring_groups_rows =
        split ? static_cast<long long>(ring_steps) * G / csize : static_cast<long long>(ring_steps) * G * rows;
    const int ring_rows = static_cast<int>(min(static_cast<long long>(min(a.tokens, slot_rows)), ring_groups_rows));
    // Progress is published only when some ring row is used twice in this
    // call: otherwise no push ever waits for it, and the barrier and the
    // release store (which waits for the block's stores to complete) would
    // only lengthen a short call.
    const bool ring_reused = ring_rows < a.tokens;
    // The buffer: the blocks' progress words, then the R slots, then the
    // exchange area.
    unsigned long long* progress = reinterpret_cast<unsigned long long*>(lam);
    lam += kLamportProgressBytes / sizeof(uint4);
    uint32_t* xarea = reinterpret_cast<uint32_t*>(lam + static_cast<uint64_t>(R) * slot_units);
    const int b = static_cast<int>(blockIdx.x);
    const int q = (b + 1) % G;  // position this block reduces in every step
    const int reducer_of_mine = (b + G - 1) % G;  // the block that reduces the position this block pushes
    const uint32_t nsteps = static_cast<uint32_t>((groups + G - 1) / G);
    bool gave_up = false;

    // Push the group at this block's position of step s, if the step reaches
    // it (block-uniform).  A ring row used before in this call (by step
    // s - ring_steps) is pushed only once its reducer, the block before this
    // one, has published that step: it has taken the row and written the
    // marker back.
    auto push_step = [&](uint32_t s) {
        const int base = static_cast<int>(s) * G;
        if (b >= min(G, groups - base))
            return;
        const int gp = base + b;
        const int p_row = split ? gp / csize : gp * rows + row_in_block;
        const int p_begin = split ? (gp % csize) * slice : 0;
        const int p_end = min(p_begin + slice, a.units_row);
        const bool p_ok = p_row < a.tokens;
        const uint64_t p_off = static_cast<uint64_t>(p_row) * a.units_row;
        const uint64_t p_ring = static_cast<uint64_t>(p_row % ring_rows) * a.units_row;
        if ((split ? gp / csize : gp * rows) >= ring_rows) {
            if (threadIdx.x == 0)
                lamport_wait_progress(progress + reducer_of_mine, epoch, s - ring_steps, gave_up);
            __syncthreads();
        }
        // Vector by vector, all R ranks' loads in flight at once.
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = p_begin + lane + k * tpr;
            if (p_ok && j < p_end)
                lamport_push<T, R_CT>(a, lam, slot_units, R, p_off + j, p_ring + j, skip_rank);
        }
    };

    int parity = 0;
    for (uint32_t step = 0; step < nsteps; ++step, parity ^= 1) {
        const int base = static_cast<int>(step) * G;
        const int n = min(G, groups - base);
        const bool do_reduce = q < n;  // block-uniform
        const int gr = base + q;
        const int row = split ? gr / csize : gr * rows + row_in_block;
        const int c = split ? gr % csize : 0;
        const int j_begin = c * slice;
        const int j_end = min(j_begin + slice, a.units_row);
        const bool row_ok = do_reduce && row < a.tokens;
        const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
        const uint64_t row_ring = static_cast<uint64_t>(row % ring_rows) * a.units_row;

        // The residual of the reduced group does not depend on the buffer:
        // its loads go out first and complete behind the push.
        uint4 rv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j_begin + lane + k * tpr;
            if (row_ok && j < j_end)
                rv[k] = U::load(a.residual, row_off + j);
        }
        push_step(step);
        if (!do_reduce) {
            if (ring_reused) {
                __syncthreads();
                if (threadIdx.x == 0)
                    lamport_publish(progress + b, (static_cast<unsigned long long>(epoch) << 32) | step);
            }
            continue;
        }

        // Reduce: take every rank's vector from the buffer, then bias and
        // residual, in that order.
        float x[VPT][L];
        uint4 wv[VPT];
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j_begin + lane + k * tpr;
#pragma unroll
            for (int l = 0; l < L; ++l)
                x[k][l] = 0.0f;
            if (row_ok && j < j_end)
                lamport_take<T, R_CT>(lam, slot_units, R, row_ring + j, x[k], gave_up);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j_begin + lane + k * tpr;
            if (row_ok && j < j_end) {
                float t[L];
                if (a.bias != nullptr) {
                    U::to_float(U::load_cached(a.bias, j), t);
                    add_lanes<L>(x[k], t);
                }
                U::to_float(rv[k], t);
                add_lanes<L>(x[k], t);
                wv[k] = U::load_cached(a.weight, j);
                U::store(a.residual_out, row_off + j, x[k]);
#pragma unroll
                for (int l = 0; l < L; ++l)
                    ss = fmaf(x[k][l], x[k][l], ss);
            }
        }
        // Double-buffered scratch: a warp that runs ahead into the next
        // step writes the other half.
        ss = row_sum(ss, tpr, red[parity]);
        if (split) {
            if (threadIdx.x < 32) {
                const float tot = lamport_exchange<T>(xarea + static_cast<uint64_t>(row) * kLamportRowWords, c,
                                                      csize, ss, gave_up);
                if (threadIdx.x == 0)
                    tot_s[parity] = tot;
            }
            __syncthreads();
            ss = tot_s[parity];
        }
        const float inv = inv_rms(ss, a.hidden, a.eps);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j_begin + lane + k * tpr;
            if (row_ok && j < j_end) {
                float w[L], y[L];
                U::to_float(wv[k], w);
#pragma unroll
                for (int l = 0; l < L; ++l)
                    y[l] = x[k][l] * inv * w[l];
                U::store(a.out, row_off + j, y);
            }
        }
        // Every thread of the block has taken its vectors of this step and
        // written the marker back: publish the step (the release covers the
        // whole block's stores through the barrier before it).  Without it
        // the scratch stays safe: red and tot_s are double-buffered, and a
        // thread cannot reach the step after next before every thread has
        // passed the next step's barriers.
        if (ring_reused) {
            __syncthreads();
            if (threadIdx.x == 0)
                lamport_publish(progress + b, (static_cast<unsigned long long>(epoch) << 32) | step);
        }
    }
}

// Barrier over `count` threads (a multiple of 32) of this block, by id: the
// push and reduce warps of k_fused_lamport_ws synchronise apart.
__device__ __forceinline__ void named_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// row_sum over the `count` threads that reach named barrier `id` (threads
// 0 .. count-1 of `t`'s numbering; the warps of one row are consecutive).
__device__ __forceinline__ float row_sum_named(float v, int tpr, float* red, int id, int count, int t)
{
    if (tpr <= 32) {
        for (int off = tpr >> 1; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, off);
        return v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = t >> 5;
    if ((t & 31) == 0)
        red[warp] = v;
    named_sync(id, count);
    const int wpr = tpr >> 5;
    const int first = (warp / wpr) * wpr;
    float s = red[first];
    for (int w = 1; w < wpr; ++w)
        s += red[first + w];
    return s;
}

// The Lamport-style call with the push and the reduce in separate warps of
// each block (rows not split; the reduce side has blockDim.x / 2 threads,
// tpr a row, VPT vectors a thread, as k_fused_lamport).  Same buffer, ring,
// schedule positions and progress words as k_fused_lamport: block b pushes
// position b and reduces position (b + 1) mod G of every step.  But the push
// warps run through the steps on their own, limited only by the ring (a
// push into a reused ring row waits for its reducer's progress word), so a
// reduce finds its neighbour's data already pushed, and the partials' loads
// of later steps overlap the polls and the row reductions of earlier ones.
// Barriers: id 1 among the reduce warps, id 2 among the push warps; nothing
// after the split waits on the whole block.  MAXT is the largest block:
//   512 threads, VPT at most 4 (more would not fit 128 registers): the push
//     warps move two vectors of every rank per round (2R loads in flight a
//     thread), and a reduce thread takes all R ranks of a vector at once;
//   1024 threads, VPT at most 2 (64 registers): twice the warps; the push
//     warps move one vector of every rank per round, a reduce thread takes
//     the ranks of a vector four at a time (when R > 4) and loads its
//     weight after the row sum.
template <typename T, int R_CT, int VPT, int MAXT>
__global__ void __launch_bounds__(MAXT, 1)
k_fused_lamport_ws(const FusedArgs a, uint4* lam_buffer, const int tpr, const int skip_rank, const int slot_rows,
                   const uint32_t epoch, const int ring_steps)
{
    static_assert(MAXT == 512 || (MAXT == 1024 && VPT <= 2), "block and registers");
    constexpr int PV = MAXT > 512 ? 1 : 2;  // vectors of every rank a push thread moves per round
    pdl_enter();
    using U = Unit<T, true>;
    constexpr int L = U::L;
    __shared__ float red[2][32];
    uint4* lam = lam_buffer;
    const int R = R_CT > 0 ? R_CT : a.R;
    const int half = static_cast<int>(blockDim.x) / 2;
    const bool pusher = static_cast<int>(threadIdx.x) >= half;
    const int t = pusher ? static_cast<int>(threadIdx.x) - half : static_cast<int>(threadIdx.x);
    const int rows = half / tpr;
    const int lane = t & (tpr - 1);
    const int row_in_block = t / tpr;
    const int groups = (a.tokens + rows - 1) / rows;
    const int G = static_cast<int>(gridDim.x);
    const uint64_t slot_units = static_cast<uint64_t>(slot_rows) * a.units_row;
    const int ring_rows =
        static_cast<int>(min(static_cast<long long>(min(a.tokens, slot_rows)), static_cast<long long>(ring_steps) * G * rows));
    const bool ring_reused = ring_rows < a.tokens;  // publish progress only then (see k_fused_lamport)
    unsigned long long* progress = reinterpret_cast<unsigned long long*>(lam);
    lam += kLamportProgressBytes / sizeof(uint4);
    const int b = static_cast<int>(blockIdx.x);
    const uint32_t nsteps = static_cast<uint32_t>((groups + G - 1) / G);
    bool gave_up = false;

    if (pusher) {
        const int reducer_of_mine = (b + G - 1) % G;
        for (uint32_t step = 0; step < nsteps; ++step) {
            const int base = static_cast<int>(step) * G;
            if (b >= min(G, groups - base))
                break;  // later steps are shorter still (push-uniform)
            const int gp = base + b;
            const int p_row = gp * rows + row_in_block;
            const bool p_ok = p_row < a.tokens;
            const uint64_t p_off = static_cast<uint64_t>(p_row) * a.units_row;
            const uint64_t p_ring = static_cast<uint64_t>(p_row % ring_rows) * a.units_row;
            if (gp * rows >= ring_rows) {  // a ring row used before in this call
                if (t == 0)
                    lamport_wait_progress(progress + reducer_of_mine, epoch, step - ring_steps, gave_up);
                named_sync(2, half);
            }
            if constexpr (R_CT > 0) {
#pragma unroll
                for (int k = 0; k < VPT; k += PV) {
                    uint4 v[PV][R_CT];
                    bool ok[PV];
#pragma unroll
                    for (int h = 0; h < PV; ++h) {
                        const int j = lane + (k + h) * tpr;
                        ok[h] = k + h < VPT && p_ok && j < a.units_row;
                        if (ok[h]) {
#pragma unroll
                            for (int r = 0; r < R_CT; ++r)
                                v[h][r] = ld_stream16(static_cast<const uint4*>(a.partials[r]) + p_off + j);
                        }
                    }
#pragma unroll
                    for (int h = 0; h < PV; ++h) {
                        const int j = lane + (k + h) * tpr;
                        if (ok[h]) {
#pragma unroll
                            for (int r = 0; r < R_CT; ++r)
                                if (r != skip_rank)
                                    st_relaxed16(lam + r * slot_units + p_ring + j, lamport_clean<T>(v[h][r]));
                        }
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = lane + k * tpr;
                    if (p_ok && j < a.units_row)
                        lamport_push<T, R_CT>(a, lam, slot_units, R, p_off + j, p_ring + j, skip_rank);
                }
            }
        }
        return;
    }

    const int q = (b + 1) % G;  // the position this block reduces in every step
    int parity = 0;
    for (uint32_t step = 0; step < nsteps; ++step, parity ^= 1) {
        const int base = static_cast<int>(step) * G;
        const bool do_reduce = q < min(G, groups - base);  // reduce-uniform
        const int gr = base + q;
        const int row = gr * rows + row_in_block;
        const bool row_ok = do_reduce && row < a.tokens;
        const uint64_t row_off = static_cast<uint64_t>(row) * a.units_row;
        const uint64_t row_ring = static_cast<uint64_t>(row % ring_rows) * a.units_row;
        if (do_reduce) {
            uint4 rv[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = lane + k * tpr;
                if (row_ok && j < a.units_row)
                    rv[k] = U::load(a.residual, row_off + j);
            }
            float x[VPT][L];
            uint4 wv[VPT];
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = lane + k * tpr;
#pragma unroll
                for (int l = 0; l < L; ++l)
                    x[k][l] = 0.0f;
                if (row_ok && j < a.units_row)
                    lamport_take<T, R_CT, (MAXT > 512 && R_CT > 4) ? 4 : R_CT>(lam, slot_units, R, row_ring + j,
                                                                              x[k], gave_up);
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = lane + k * tpr;
                if (row_ok && j < a.units_row) {
                    float tv[L];
                    if (a.bias != nullptr) {
                        U::to_float(U::load_cached(a.bias, j), tv);
                        add_lanes<L>(x[k], tv);
                    }
                    U::to_float(rv[k], tv);
                    add_lanes<L>(x[k], tv);
                    if constexpr (MAXT <= 512)
                        wv[k] = U::load_cached(a.weight, j);
                    U::store(a.residual_out, row_off + j, x[k]);
#pragma unroll
                    for (int l = 0; l < L; ++l)
                        ss = fmaf(x[k][l], x[k][l], ss);
                }
            }
            ss = row_sum_named(ss, tpr, red[parity], 1, half, t);
            const float inv = inv_rms(ss, a.hidden, a.eps);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = lane + k * tpr;
                if (row_ok && j < a.units_row) {
                    float w[L], y[L];
                    if constexpr (MAXT > 512)  // loaded late: 64 registers a thread
                        wv[k] = U::load_cached(a.weight, j);
                    U::to_float(wv[k], w);
#pragma unroll
                    for (int l = 0; l < L; ++l)
                        y[l] = x[k][l] * inv * w[l];
                    U::store(a.out, row_off + j, y);
                }
            }
        }
        // Every reduce thread has taken its vectors of this step and written
        // the marker back: publish the step.
        if (ring_reused) {
            named_sync(1, half);
            if (t == 0)
                lamport_publish(progress + b, (static_cast<unsigned long long>(epoch) << 32) | step);
        }
    }
}

// Fills `nvec` 16-byte vectors, then `tail_halves` 2-byte halves, with the
// empty marker of T.
template <typename T>
__global__ void __launch_bounds__(kFlatThreads) k_lamport_fill(uint4* buf, uint64_t nvec, uint32_t tail_halves)
{
    pdl_enter();
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride)
        st16(buf + i, lamport_empty<T>());
    if (blockIdx.x == 0 && threadIdx.x < tail_halves) {
        // Little-endian halves of the marker word: (low, high).
        const uint32_t m = LamportMarker<T>::word;
        const unsigned short half = static_cast<unsigned short>((threadIdx.x & 1u) ? (m >> 16) : (m & 0xffffu));
        reinterpret_cast<unsigned short*>(buf + nvec)[threadIdx.x] = half;
    }
}

}  // namespace ar
