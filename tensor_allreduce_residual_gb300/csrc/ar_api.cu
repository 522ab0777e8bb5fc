// ar_api.cu -- the C ABI declared in include/ar.h: argument checks (the
// configurationSupported analogue), the AUTO choice and launch shape
// (selectImplementation / kernelLaunchConfig / heuristic_min_warp_number),
// and dispatch on element type (AllReduceDispatchType) -- all after the
// call graph of "allreduce.d2".  Host code only; it allocates nothing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "ar.h"
#include "ar_auto_table.h"
#include "ar_internal.h"

namespace {

using ar::FusedArgs;
using ar::OneShotShape;
using ar::SumArgs;

constexpr int kVersion = 10000;  // 1.0.0

int esize_of(int dtype)
{
    switch (dtype) {
    case AR_FP32: return 4;
    case AR_FP16: return 2;
    case AR_BF16: return 2;
    default: return 0;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int status_of(cudaError_t e) { return e == cudaSuccess ? AR_OK : AR_ERR_CUDA; }

// Calls f(T{}) with T the element type of `dtype`.
template <typename F>
cudaError_t by_dtype(int dtype, F&& f)
{
    switch (dtype) {
    case AR_FP32: return f(float{});
    case AR_FP16: return f(__half{});
    default: return f(__nv_bfloat16{});
    }
}

int strategy_status(int strategy)
{
    if (strategy == AR_ONESHOT || strategy == AR_TWOSHOT || strategy == AR_AUTO)
        return AR_OK;
    return AR_ERR_UNSUPPORTED;  // AR_NCCL (no NCCL, one GPU) or unknown
}

int next_pow2(int v)
{
    int p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

// ---------------------------------------------------------------- one-shot shape

// Bulk-copy-fed persistent shape (mode kTma): vpt = chunks per row, one
// consumer thread per vector of a chunk (a multiple of 32), and as many ring
// slots as the shared memory of `blocks_per_sm` blocks per SM allows.
// `inputs` = tensors streamed through the ring: R partials plus the residual.
bool tma_shape(int units_row, int vpt, int inputs, int blocks_per_sm, int max_stages, OneShotShape* sh)
{
    if (!(vpt == 1 || vpt == 2 || vpt == 4 || vpt == 8) || blocks_per_sm < 1 || blocks_per_sm > 4)
        return false;
    const int nc = ((units_row + vpt - 1) / vpt + 31) / 32 * 32;
    if (nc > ar::tma_max_consumers(vpt) || (units_row + nc - 1) / nc > vpt)
        return false;
    int budget = ar::kSmemPerSM / blocks_per_sm - ar::kSmemReservedPerBlock;
    if (budget > ar::kSmemPerBlockMax)
        budget = ar::kSmemPerBlockMax;
    int stages = max_stages >= ar::kTmaMinStages && max_stages < ar::kTmaMaxStages ? max_stages : ar::kTmaMaxStages;
    while (stages >= ar::kTmaMinStages && ar::tma_smem_bytes(inputs, nc, stages) > static_cast<size_t>(budget))
        --stages;
    if (stages < ar::kTmaMinStages)
        return false;
    sh->tpr = nc;
    sh->vpt = vpt;
    sh->rows = 1;
    sh->mode = ar::kTma;
    sh->smem_bytes = static_cast<int>(ar::tma_smem_bytes(inputs, nc, stages));
    sh->stages = stages;
    sh->blocks_per_sm = blocks_per_sm;
    return true;
}

// Row-split shape (mode kCluster): `cluster` blocks share a row, each owning
// ceil(units_row / cluster) units at `vpt` per thread; threads per block =
// that over vpt, rounded up to a power of two, at least a warp.
bool cluster_shape(int units_row, int vpt, int lanes, int cluster, OneShotShape* sh)
{
    if (!(vpt == 1 || vpt == 2 || vpt == 4 || vpt == 8) || !(cluster == 2 || cluster == 4 || cluster == 8))
        return false;
    const int slice = (units_row + cluster - 1) / cluster;
    int tpb = next_pow2((slice + vpt - 1) / vpt);
    if (tpb < 32)
        tpb = 32;
    if (tpb > ar::oneshot_max_threads(vpt * lanes))
        return false;
    sh->tpr = tpb;
    sh->vpt = vpt;
    sh->rows = 1;
    sh->mode = ar::kCluster;
    sh->smem_bytes = 0;
    sh->cluster = cluster;
    return true;
}

// One-shot fused shape.  Modes kRegisters / kStaged / kPersistent: threads per
// row = units_row / vpt rounded up to a power of two; blocks hold at least
// 128 threads; register-resident rows are limited by the registers a thread
// may use, staged rows by shared memory.  Mode kTma: tma_shape.  Returns
// false when the row does not fit (then only the two-shot path can take it).
bool oneshot_shape(int units_row, int vpt, int lanes, bool packed, int mode, int R, OneShotShape* sh,
                   int blocks_per_sm = 1, int max_stages = 0)
{
    if (mode == ar::kTma)
        return packed && tma_shape(units_row, vpt, R + 1, blocks_per_sm, max_stages, sh);
    if (mode == ar::kCluster)  // blocks_per_sm carries the cluster size for this mode
        return packed && cluster_shape(units_row, vpt, lanes, blocks_per_sm, sh);
    const int max_vpt = packed ? ar::kMaxVPTVec : ar::kMaxVPTScalar;
    const bool stage = mode != ar::kRegisters;
    if (vpt < 1 || vpt > max_vpt || (stage && (!packed || vpt > ar::kMaxVPTVec)))
        return false;
    const int tpr = next_pow2((units_row + vpt - 1) / vpt);
    const int max_threads = stage ? ar::kMaxTPR : ar::oneshot_max_threads(vpt * lanes);
    if (tpr > ar::kMaxTPR || tpr > max_threads)
        return false;
    // The persistent form needs whole-warp rows and R known at compile time.
    if (mode == ar::kPersistent &&
        (tpr < 128 || tpr > ar::kMaxPersistThreads || !(R == 1 || R == 2 || R == 4 || R == 8)))
        mode = ar::kStaged;
    sh->tpr = tpr;
    sh->vpt = vpt;
    sh->rows = tpr >= 128 ? 1 : 128 / tpr;
    sh->mode = mode;
    sh->smem_bytes = 0;
    if (stage) {
        const size_t bytes = static_cast<size_t>(sh->rows) * lanes * units_row * sizeof(float);
        if (bytes > static_cast<size_t>(ar::kMaxStageBytes))
            return false;
        sh->smem_bytes = static_cast<int>(bytes);
    }
    return true;
}

// Rule used when the measured table has no entry: aim for 512 threads per
// row up to 512 rows (every measured row shape was fastest near 512 threads
// per row there: fewer registers per thread, more loads in flight per row)
// and 256 beyond, with the smallest units-per-thread that reaches it.
int rule_vpt(int units_row, int tokens, int lanes, bool packed)
{
    const int max_vpt = packed ? ar::kMaxVPTVec : ar::kMaxVPTScalar;
    const int target = tokens <= 512 ? 512 : 256;
    int vpt = 1;
    while (vpt < max_vpt && (units_row + vpt - 1) / vpt > target)
        vpt <<= 1;
    while (vpt < max_vpt &&
           next_pow2((units_row + vpt - 1) / vpt) > ar::oneshot_max_threads(vpt * lanes))
        vpt <<= 1;
    return vpt;
}

// Rule for many rows when the measured table has no entry: the bulk-copy-fed
// persistent kernel with at most 512 consumer threads per row (the fewest
// chunks per row that allow it) and a ring of about kTmaRuleInflight bytes,
// the depth that measured fastest on the 8192 x 8192 prefill.  False when
// the row does not fit that kernel.
constexpr int kTmaRuleMinTokens = 2048;
constexpr int kTwoShotRuleMinTokens = 1024;
constexpr int kClusterRuleMaxTokens = 8;
constexpr size_t kTmaRuleInflight = 144 * 1024;

bool tma_rule_shape(int units_row, int R, OneShotShape* sh)
{
    int cpr = 1;
    while (cpr < 8 && (units_row + cpr - 1) / cpr > ar::tma_max_consumers(cpr))
        cpr <<= 1;
    // With many partials a stage of (R + 1) chunks can outgrow the ring: cut
    // the row into more, smaller chunks until two stages fit the budget.
    for (; cpr <= 8; cpr <<= 1) {
        const int nc = ((units_row + cpr - 1) / cpr + 31) / 32 * 32;
        const size_t stage = static_cast<size_t>(R + 1) * nc * 16;
        int stages = static_cast<int>((kTmaRuleInflight + stage / 2) / stage);
        if (stages < ar::kTmaMinStages)
            stages = ar::kTmaMinStages;
        if (tma_shape(units_row, cpr, R + 1, 1, stages, sh))
            return true;
    }
    return false;
}

const ar::AutoEntry* table_lookup(int esize, int R, int units_row, int tokens)
{
    for (const ar::AutoEntry& e : ar::kAutoTable) {
        if (e.esize == 0)
            break;
        if (e.esize == esize && e.R == R && e.units_row == units_row && tokens <= e.tokens_max)
            return &e;
    }
    return nullptr;
}

// AR_AUTO's partition for the reduce-only sum of n elements: the measured
// table (keyed on n in 16-byte vectors), else the rule -- R rank slices when
// the one-slice grid would have fewer blocks than the rank-slice grid (small
// n: more blocks in flight, less latency), one slice otherwise.  `units` is
// what the kernel walks: vectors on the packed path, elements otherwise.
// Both partitions give bit-identical values.
int sum_auto_strategy(int esize, int R, size_t n, bool packed)
{
    if (R == 1)
        return AR_ONESHOT;
    const uint64_t vectors = n / static_cast<size_t>(16 / esize);
    for (const ar::SumAutoEntry& e : ar::kSumAutoTable) {
        if (e.esize == 0)
            break;
        if (e.esize == esize && e.R == R && vectors <= static_cast<uint64_t>(e.units_max))
            return e.strategy;
    }
    const uint64_t units = packed ? vectors : n;
    const uint64_t per_block = static_cast<uint64_t>(ar::kFlatThreads) * ar::sum_unroll(R, packed);
    const uint64_t one = (units + per_block - 1) / per_block;
    const uint64_t slice = (units + R - 1) / R;
    const uint64_t two = static_cast<uint64_t>(R) * ((slice + per_block - 1) / per_block);
    return one < two ? AR_TWOSHOT : AR_ONESHOT;
}

// Measurement override of the one-shot shape.  Only the test build of the
// library (compiled with AR_TEST_HOOKS, libar_test.so) reads it, from
// AR_ONESHOT_SHAPE="vpt:mode", "vpt:mode:early", "vpt:mode:early:blocks_per_sm"
// or "vpt:mode:early:blocks_per_sm:max_stages" (e.g. "4:1", "2:0:1",
// "4:3:0:2", "4:3:1:1:3"; for mode 4 the fourth field is the cluster size,
// "1:4:1:8"), once per process; it then replaces the table and the rule for
// every packed call.  The sweeps that build the AUTO table and the tests of
// every launch shape use it.  The product library never reads the
// environment: its override is always empty.
struct ShapeOverride {
    int vpt = 0;
    int mode = 0;
    int early = 0;
    int blocks_per_sm = 1;
    int max_stages = 0;
};

#ifdef AR_TEST_HOOKS
const ShapeOverride& shape_override()
{
    static const ShapeOverride ov = [] {
        ShapeOverride o;
        if (const char* env = std::getenv("AR_ONESHOT_SHAPE")) {
            int v = 0, st = 0, early = 0, bps = 1, stages = 0;
            const int got = std::sscanf(env, "%d:%d:%d:%d:%d", &v, &st, &early, &bps, &stages);
            if (got >= 2 && v > 0 && st >= 0 && st <= ar::kCluster) {
                o.vpt = v;
                o.mode = st;
                o.early = got >= 3 && early != 0;
                o.blocks_per_sm = got >= 4 && bps > 0 ? bps : 1;
                o.max_stages = got == 5 && stages > 0 ? stages : 0;
            }
        }
        return o;
    }();
    return ov;
}

// Fault injection for the bulk-copy-fed kernel's bounded waits (test build
// only): AR_TEST_STALL_STAGE=k makes its producer leave stage k of every
// block unarmed, so the waits on it run out (about a second) and the kernel
// takes its abort path; ar_device_status then reports AR_ERR_TIMEOUT.  Read
// once per process; unset means no stall.
int test_stall_stage()
{
    static const int v = [] {
        const char* e = std::getenv("AR_TEST_STALL_STAGE");
        const int k = e != nullptr ? std::atoi(e) : -1;
        return k >= 0 ? k + 1 : 0;
    }();
    return v;
}

// Fault injection for the Lamport call's bounded waits (test build only):
// AR_TEST_LAMPORT_SKIP_RANK=r leaves rank r's pushes out, so the polls of
// its slot run out (about a second); ar_device_status then reports
// AR_ERR_TIMEOUT.  Read once per process; unset means -1 (none).
int test_lamport_skip_rank()
{
    static const int v = [] {
        const char* e = std::getenv("AR_TEST_LAMPORT_SKIP_RANK");
        const int r = e != nullptr ? std::atoi(e) : -1;
        return r >= 0 && r < AR_MAX_RANKS ? r : -1;
    }();
    return v;
}
#else
const ShapeOverride& shape_override()
{
    static const ShapeOverride none;
    return none;
}
int test_stall_stage() { return 0; }
int test_lamport_skip_rank() { return -1; }
#endif

struct FusedPlan {
    int strategy;      // AR_ONESHOT or AR_TWOSHOT
    bool oneshot_ok;   // the row fits the one-shot kernel
    OneShotShape shape;
};

// Resolves AUTO and the one-shot shape for a fused call.
FusedPlan plan_fused(int esize, int R, int hidden, int tokens, bool packed, int strategy)
{
    const int lanes = packed ? 16 / esize : 1;
    const int units_row = hidden / lanes;
    FusedPlan p{};
    int vpt = rule_vpt(units_row, tokens, lanes, packed);
    int mode = ar::kRegisters;
    int early = 1;
    int bps = 1;
    int max_stages = 0;
    int auto_strategy = AR_ONESHOT;
    if (packed) {
        if (const ar::AutoEntry* e = table_lookup(esize, R, units_row, tokens)) {
            auto_strategy = e->strategy;
            if (e->vpt > 0) {
                vpt = e->vpt;
                mode = e->mode;
                early = e->early;
                bps = e->blocks_per_sm > 0 ? e->blocks_per_sm : 1;
                max_stages = e->max_stages;
            }
        }
        const ShapeOverride& ov = shape_override();
        if (ov.vpt > 0) {
            vpt = ov.vpt;
            mode = ov.mode;
            early = ov.early;
            bps = ov.blocks_per_sm;
            max_stages = ov.max_stages;
        }
    }
    const bool measured = packed && (table_lookup(esize, R, units_row, tokens) != nullptr || shape_override().vpt > 0);
    if (!measured && packed && tokens >= kTmaRuleMinTokens && tma_rule_shape(units_row, R, &p.shape)) {
        p.shape.early_residual = 1;
        p.oneshot_ok = true;
        p.strategy = strategy == AR_AUTO ? AR_ONESHOT : strategy;
        return p;
    }
    // A few long rows: split each across a cluster of 8 blocks (measured at
    // one token: 3.1 us against 4.0 us for R=8 bf16 H=8192, 3.2 against 4.5
    // for R=2 bf16 H=16384).
    if (!measured && packed && tokens <= kClusterRuleMaxTokens && units_row >= 1024 &&
        cluster_shape(units_row, units_row >= 2048 ? 2 : 1, lanes, 8, &p.shape)) {
        p.shape.early_residual = 0;
        p.oneshot_ok = true;
        p.strategy = strategy == AR_AUTO ? AR_ONESHOT : strategy;
        return p;
    }
    // Rows too long for the bulk-copy-fed kernel, many of them: the two-shot
    // path (measured on 16384-wide bf16 rows: 29.7 us against 36.0 us for
    // the register-resident one-shot kernel at 1024 rows).
    if (!measured && tokens >= kTwoShotRuleMinTokens && units_row > ar::tma_max_consumers(8) * 8)
        auto_strategy = AR_TWOSHOT;
    p.oneshot_ok = oneshot_shape(units_row, vpt, lanes, packed, mode, R, &p.shape, bps, max_stages);
    if (!p.oneshot_ok)  // the chosen shape does not fit this row: the rule's shape
        p.oneshot_ok = oneshot_shape(units_row, rule_vpt(units_row, tokens, lanes, packed), lanes,
                                     packed, ar::kRegisters, R, &p.shape);
    p.shape.early_residual = early;
    if (!p.oneshot_ok)
        auto_strategy = AR_TWOSHOT;
    p.strategy = strategy == AR_AUTO ? auto_strategy : strategy;
    return p;
}

// Two-shot chunking: chunks of kFlatThreads * kChunkVPT units per row.
int twoshot_nchunk(int units_row)
{
    const int chunk = ar::kFlatThreads * ar::kChunkVPT;
    return (units_row + chunk - 1) / chunk;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Register-resident norm shape: 4 packed vectors per thread for rows of 512
// to 1024 vectors (8 for longer rows, whose blocks would pass 256 threads),
// 8 below 512 (16 elements on the element-wise path), and fewer when a row
// would get less than a warp; blocks of at least 128 threads.  Measured on
// 8192-row tensors: 42.2 us (8192 bf16) and 20.6 us (4096 fp16), both at 4
// per thread, 0.94 and 0.96 of the copy peak.
// `vpt` forces the units per thread (measurement only).  False when the row
// does not fit one block.
bool norm_shape(int units_row, bool packed, OneShotShape* sh, int vpt = 0)
{
    const int max_vpt = packed ? ar::kMaxVPTVec : ar::kMaxVPTScalar;
    if (vpt <= 0) {
        vpt = packed && units_row >= 512 ? 4 : max_vpt;
        while (vpt > 1 && (units_row + vpt - 1) / vpt < 32)
            vpt >>= 1;
        // A row too long for 4 vectors a thread in one block takes 8.
        if (packed && vpt == 4 && next_pow2((units_row + 3) / 4) > ar::norm_max_threads(true, 4))
            vpt = 8;
    }
    if (vpt > max_vpt)
        return false;
    const int tpr = next_pow2((units_row + vpt - 1) / vpt);
    if (tpr > ar::norm_max_threads(packed, vpt))
        return false;
    sh->tpr = tpr;
    sh->vpt = vpt;
    sh->rows = tpr >= 128 ? 1 : 128 / tpr;
    sh->mode = ar::kRegisters;
    sh->smem_bytes = 0;
    return true;
}

// Lamport-style call.  Up to 8 rows whose R partials hold at least 8192
// 16-byte vectors: each row split over 4 blocks, with the smallest units per
// thread that fit lamport_max_threads (R=8 bf16 rows of 8192: 6.5 us at one
// token against 7.4 us unsplit; splitting over 8 blocks, or splitting
// shorter rows, measured slower: the exchange of the partial sums of squares
// costs about as much as it saves).  Otherwise the register-resident
// one-shot shape (heuristic_min_warp_number: threads per row from the
// one-shot rule), its blocks capped at lamport_max_threads.  The shape
// override forces either: mode kRegisters with its units per thread, or
// mode kCluster with its units per thread and split (measurement only).
int lamport_split_rule(int tokens, int R, int units_row)
{
    return tokens <= 8 && static_cast<long long>(R) * units_row >= 8192 ? 4 : 1;
}

// Rows not split, at least this many: separate push and reduce warps
// (k_fused_lamport_ws), when the reduce side has at most 256 threads of at
// most 4 vectors each, or at most 512 threads of at most 2; two vectors a
// thread first where that makes the reduce side more than 256 threads
// (blocks of up to 1024 threads at 64 registers: twice the warps, half the
// dependent take rounds a step).
// Measured at R=8 bf16 H=8192, one role / split roles with 4 vectors (512
// threads) / split roles with 2 vectors (1024 threads): 569-571 / 507-532 /
// 467-469 us at 8192 rows, 147-148 / 134-137 / 124.4-124.6 us at 2048,
// 80 / 74-77 / 69.2-69.4 us at 1024; at 256 rows one role is fastest
// (18.7 against 25.1 and 22.3 us).
constexpr int kLamportRolesMinTokens = 1024;

// Ring depth of the Lamport buffer, in grid steps.  Deeper rings measured
// slower (3: 565-594 us, 4: 631 us against 532-570 us at 8192 rows of R=8
// bf16 H=8192): more of the ring leaves L2 before it is polled.
constexpr int kLamportRingSteps = 2;

bool lamport_shape(int units_row, int tokens, int lanes, int R, OneShotShape* sh)
{
    const ShapeOverride& ov = shape_override();
    auto fits = [&](int vpt) {
        if (!(oneshot_shape(units_row, vpt, lanes, true, ar::kRegisters, R, sh) &&
              sh->tpr * sh->rows <= ar::lamport_max_threads(vpt * lanes)))
            return false;
        const bool roles_fit = (sh->tpr * sh->rows <= 256 && vpt <= 4) || (sh->tpr * sh->rows <= 512 && vpt <= 2);
        sh->roles = roles_fit && (ov.vpt > 0 ? ov.early : tokens >= kLamportRolesMinTokens) ? 1 : 0;
        sh->stages = ov.vpt > 0 && ov.max_stages >= 2 && ov.max_stages <= ar::kLamportMaxRingSteps
                         ? ov.max_stages
                         : kLamportRingSteps;
        return true;
    };
    auto fits_split = [&](int vpt, int c) {
        sh->roles = 0;
        sh->stages = kLamportRingSteps;
        return static_cast<long long>(tokens) * c <= INT32_MAX && cluster_shape(units_row, vpt, lanes, c, sh) &&
               sh->tpr <= ar::lamport_max_threads(vpt * lanes);
    };
    if (ov.vpt > 0 && ov.mode == ar::kRegisters && fits(ov.vpt))
        return true;
    if (ov.vpt > 0 && ov.mode == ar::kCluster && fits_split(ov.vpt, ov.blocks_per_sm))
        return true;
    int c = lamport_split_rule(tokens, R, units_row);
    while (c > 1 && (units_row + c - 1) / c < 32)  // no slice shorter than a warp
        c >>= 1;
    if (c > 1)
        for (int vpt = 1; vpt <= ar::kMaxVPTVec; vpt <<= 1)
            if (fits_split(vpt, c))
                return true;
    if (tokens >= kLamportRolesMinTokens && fits(2) && sh->roles && sh->tpr * sh->rows > 256)
        return true;
    for (int vpt = rule_vpt(units_row, tokens, lanes, true); vpt <= ar::kMaxVPTVec; vpt <<= 1)
        if (fits(vpt))
            return true;
    return false;
}

// Bytes of the Lamport buffer for the launch shape `sh`: the blocks'
// progress words, the R slots (a ring of at most kLamportRingGroups row
// groups each), then the exchange area (per token).
size_t lamport_buffer_bytes(int R, int hidden, int tokens, int esize, const OneShotShape& sh)
{
    const int csize = sh.mode == ar::kCluster ? sh.cluster : 1;
    const int slot_rows = ar::lamport_slot_rows(tokens, sh.rows, csize);
    return static_cast<size_t>(ar::kLamportProgressBytes) + static_cast<size_t>(R) * slot_rows * hidden * esize +
           static_cast<size_t>(tokens) * ar::kLamportRowWords * sizeof(uint32_t);
}

// A value of its own for every Lamport call, in [1, 2^31): the progress
// words its blocks publish carry it, so words that earlier calls (or the
// marker fill) left in the buffer never pass for this call's.
uint32_t next_lamport_epoch()
{
    static std::atomic<uint32_t> counter{0};
    return counter.fetch_add(1, std::memory_order_relaxed) % 0x7fffffffu + 1u;
}

}  // namespace

namespace ar {

// Programmatic dependent launch is always on in the product library; the
// test build switches it off with AR_PDL=0 (read once), to measure its effect.
bool pdl_enabled()
{
#ifdef AR_TEST_HOOKS
    static const bool on = [] {
        const char* e = std::getenv("AR_PDL");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
#else
    return true;
#endif
}

}  // namespace ar

extern "C" {

int ar_version(void) { return kVersion; }

const char* ar_strerror(int code)
{
    switch (code) {
    case AR_OK: return "success";
    case AR_ERR_INVALID_ARG: return "invalid argument";
    case AR_ERR_UNSUPPORTED: return "unsupported configuration";
    case AR_ERR_WORKSPACE: return "workspace missing or too small";
    case AR_ERR_CUDA: return "CUDA launch error";
    case AR_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown status code";
    }
}

size_t ar_workspace_size(int R, size_t n, int dtype)
{
    if (R < 1 || R > AR_MAX_RANKS || n == 0 || esize_of(dtype) == 0)
        return 0;
    // At most one (row, chunk) entry per element: reached by hidden == 1.
    return round256(n * sizeof(float));
}

size_t ar_workspace_size_rows(int R, int hidden, int tokens, int dtype)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0 || esize_of(dtype) == 0)
        return 0;
    // The element-wise path (hidden not a multiple of the lane count, or a
    // misaligned pointer) has the most chunks; size for it.
    return round256(static_cast<size_t>(tokens) * twoshot_nchunk(hidden) * sizeof(float));
}

int ar_sum(const void* const* partials, int R, void* out, size_t n, int dtype, int strategy,
           ar_stream_t stream)
{
    if (R < 1 || R > AR_MAX_RANKS)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (int st = strategy_status(strategy))
        return st;
    if (n == 0)
        return AR_OK;
    if (partials == nullptr || out == nullptr)
        return AR_ERR_INVALID_ARG;
    bool packed = aligned16(out);
    for (int r = 0; r < R; ++r) {
        if (partials[r] == nullptr)
            return AR_ERR_INVALID_ARG;
        packed = packed && aligned16(partials[r]);
    }
    if (R == 1 && partials[0] == out)
        return AR_OK;  // tpSize == 1 passthrough, in place: nothing to do

    SumArgs a{};
    for (int r = 0; r < R; ++r)
        a.partials[r] = partials[r];
    a.out = out;
    a.R = R;
    const int lanes = 16 / esize;
    a.nunits = packed ? n / lanes : n;
    a.tail = packed ? static_cast<uint32_t>(n % lanes) : 0u;

    // Both strategies give bit-identical values (the two-shot slices only
    // change which block reads what); AUTO takes the partition measured
    // faster for this size.
    if (strategy == AR_AUTO)
        strategy = sum_auto_strategy(esize, R, n, packed);
    int nslices = 1;
    if (strategy == AR_TWOSHOT && R > 1) {
        a.slice = (a.nunits + R - 1) / R;
        nslices = a.slice == 0 ? 1 : R;
    }
    if (nslices == 1)
        a.slice = a.nunits;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return status_of(by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        return ar::launch_sum<T>(a, packed, nslices, s);
    }));
}

int ar_residual_rmsnorm(const void* const* partials, int R, const void* bias, const void* residual,
                        const void* weight, float eps, int hidden, int tokens, void* out,
                        void* residual_out, void* intermediate, size_t intermediate_bytes, int dtype,
                        int strategy, ar_stream_t stream)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (int st = strategy_status(strategy))
        return st;
    if (!std::isfinite(eps) || eps < 0.0f)
        return AR_ERR_INVALID_ARG;
    if (tokens == 0)
        return AR_OK;
    if (partials == nullptr || residual == nullptr || weight == nullptr || out == nullptr ||
        residual_out == nullptr || out == residual_out)
        return AR_ERR_INVALID_ARG;
    const int lanes = 16 / esize;
    bool packed = hidden % lanes == 0 && aligned16(residual) && aligned16(weight) &&
                  aligned16(out) && aligned16(residual_out) && (bias == nullptr || aligned16(bias));
    for (int r = 0; r < R; ++r) {
        if (partials[r] == nullptr)
            return AR_ERR_INVALID_ARG;
        packed = packed && aligned16(partials[r]);
    }

    FusedPlan plan = plan_fused(esize, R, hidden, tokens, packed, strategy);
    const int units_row = packed ? hidden / lanes : hidden;
    const int nchunk = twoshot_nchunk(units_row);
    const size_t ws_need = static_cast<size_t>(tokens) * nchunk * sizeof(float);
    const bool ws_ok = intermediate != nullptr && intermediate_bytes >= ws_need &&
                       (reinterpret_cast<uintptr_t>(intermediate) & 3u) == 0;
    if (plan.strategy == AR_TWOSHOT && !ws_ok) {
        if (strategy == AR_AUTO && plan.oneshot_ok)
            plan.strategy = AR_ONESHOT;  // AUTO without workspace: stay one-shot
        else
            return AR_ERR_WORKSPACE;
    }
    if (plan.strategy == AR_ONESHOT && !plan.oneshot_ok)
        return AR_ERR_UNSUPPORTED;

    FusedArgs a{};
    for (int r = 0; r < R; ++r)
        a.partials[r] = partials[r];
    a.bias = bias;
    a.residual = residual;
    a.weight = weight;
    a.out = out;
    a.residual_out = residual_out;
    a.sumsq = static_cast<float*>(intermediate);
    a.R = R;
    a.hidden = hidden;
    a.tokens = tokens;
    a.units_row = units_row;
    a.nchunk = nchunk;
    a.chunk_units = ar::kFlatThreads * ar::kChunkVPT;
    a.eps = eps;
    a.early_residual = plan.shape.early_residual;
    a.stall_stage = test_stall_stage();

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return status_of(by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        if (plan.strategy == AR_ONESHOT)
            return ar::launch_fused_oneshot<T>(a, packed, plan.shape, s);
        return ar::launch_fused_twoshot<T>(a, packed, s);
    }));
}

int ar_rmsnorm(const void* x, const void* weight, float eps, int hidden, int tokens, void* out, int dtype,
               ar_stream_t stream)
{
    if (hidden < 1 || tokens < 0)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (!std::isfinite(eps) || eps < 0.0f)
        return AR_ERR_INVALID_ARG;
    if (tokens == 0)
        return AR_OK;
    if (x == nullptr || weight == nullptr || out == nullptr)
        return AR_ERR_INVALID_ARG;
    const int lanes = 16 / esize;
    const bool packed = hidden % lanes == 0 && aligned16(x) && aligned16(weight) && aligned16(out);
    const int units_row = packed ? hidden / lanes : hidden;
    OneShotShape sh{};
    // The register-resident row kernel.  The shape override (measurement
    // only) can force its units per thread, or the bulk-copy-fed persistent
    // kernel with x as its only streamed input (slower here: 80 us at
    // 8192 x 8192 bf16, 27 us at 8192 x 4096 fp16).
    const ShapeOverride& ov = shape_override();
    bool tma = false;
    bool ok = false;
    if (packed && ov.vpt > 0) {
        tma = ov.mode == ar::kTma;
        ok = tma ? tma_shape(units_row, ov.vpt, 1, ov.blocks_per_sm, ov.max_stages, &sh)
                 : norm_shape(units_row, packed, &sh, ov.vpt);
    }
    if (!ok) {
        tma = false;
        if (!norm_shape(units_row, packed, &sh))
            return AR_ERR_UNSUPPORTED;
    }
    FusedArgs a{};
    a.partials[0] = x;
    a.weight = weight;
    a.out = out;
    a.R = 1;
    a.hidden = hidden;
    a.tokens = tokens;
    a.units_row = units_row;
    a.eps = eps;
    a.early_residual = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return status_of(by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        return tma ? ar::launch_rmsnorm_tma<T>(a, sh, s) : ar::launch_rmsnorm<T>(a, packed, sh, s);
    }));
}

int ar_allreduce(const ar_params* p, int fusion_op, int strategy, ar_stream_t stream)
{
    if (p == nullptr)
        return AR_ERR_INVALID_ARG;
    if (fusion_op == AR_FUSION_NONE)
        return ar_sum(p->partials, p->R, p->out, p->n, p->dtype, strategy, stream);
    if (fusion_op != AR_FUSION_RESIDUAL_RMS_NORM)
        return AR_ERR_UNSUPPORTED;
    if (p->hidden < 1 || p->n % static_cast<size_t>(p->hidden) != 0 ||
        p->n / static_cast<size_t>(p->hidden) > static_cast<size_t>(INT32_MAX))
        return AR_ERR_INVALID_ARG;
    const int tokens = static_cast<int>(p->n / static_cast<size_t>(p->hidden));
    return ar_residual_rmsnorm(p->partials, p->R, p->bias, p->residual, p->weight, p->eps,
                               p->hidden, tokens, p->out, p->residual_out, p->workspace,
                               p->workspace_bytes, p->dtype, strategy, stream);
}

int ar_query_launch(int R, int hidden, int tokens, int dtype, int strategy, ar_launch_plan* plan)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0 || plan == nullptr)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (int st = strategy_status(strategy))
        return st;
    const int lanes = 16 / esize;
    const bool packed = hidden % lanes == 0;
    const FusedPlan fp = plan_fused(esize, R, hidden, tokens, packed, strategy);
    if (fp.strategy == AR_ONESHOT && !fp.oneshot_ok)
        return AR_ERR_UNSUPPORTED;
    ar_launch_plan p{};
    p.strategy = fp.strategy;
    if (fp.strategy == AR_TWOSHOT) {
        p.kernel = AR_KERNEL_TWOSHOT;
        p.threads_per_row = ar::kFlatThreads * twoshot_nchunk(packed ? hidden / lanes : hidden);
        p.units_per_thread = ar::kChunkVPT;
        p.rows_per_block = 1;
        p.threads_per_block = ar::kFlatThreads;
    } else {
        const OneShotShape& sh = fp.shape;
        p.threads_per_row = sh.tpr;
        p.units_per_thread = sh.vpt;
        p.rows_per_block = sh.rows;
        p.early_residual = sh.early_residual;
        p.smem_bytes = sh.mode == ar::kRegisters ? 0 : sh.smem_bytes;
        switch (sh.mode) {
        case ar::kRegisters:
            p.kernel = AR_KERNEL_ONESHOT_REGISTERS;
            p.threads_per_block = sh.tpr * sh.rows;
            break;
        case ar::kStaged:
            p.kernel = AR_KERNEL_ONESHOT_SHARED;
            p.threads_per_block = sh.tpr * sh.rows;
            break;
        case ar::kPersistent:
            p.kernel = AR_KERNEL_ONESHOT_PERSISTENT;
            p.threads_per_block = sh.tpr;
            break;
        case ar::kCluster:
            p.kernel = AR_KERNEL_ONESHOT_CLUSTER;
            p.threads_per_row = sh.tpr * sh.cluster;
            p.threads_per_block = sh.tpr;
            p.blocks_per_sm = 0;
            p.stages = 0;
            p.cluster = sh.cluster;
            break;
        default:
            p.kernel = AR_KERNEL_ONESHOT_BULK;
            p.threads_per_block = sh.tpr + 32;
            p.blocks_per_sm = sh.blocks_per_sm;
            p.stages = sh.stages;
            break;
        }
    }
    *plan = p;
    return AR_OK;
}

int ar_device_status(void)
{
    unsigned int total = 0;
    cudaError_t e = cudaSuccess;
    const int dtypes[] = {AR_FP32, AR_FP16, AR_BF16};
    for (int dt : dtypes) {
        unsigned int n = 0;
        const cudaError_t ed = by_dtype(dt, [&](auto tag) {
            using T = decltype(tag);
            return ar::take_wait_timeouts<T>(&n);
        });
        if (ed != cudaSuccess)
            e = ed;
        total += n;
    }
    unsigned int np = 0;
    const cudaError_t ep = ar::take_peer_wait_timeouts(&np);
    if (ep != cudaSuccess)
        e = ep;
    total += np;
    if (e != cudaSuccess)
        return AR_ERR_CUDA;
    return total != 0 ? AR_ERR_TIMEOUT : AR_OK;
}

size_t ar_config_workspace_size(int R, size_t n, int hidden, int dtype)
{
    const int esize = esize_of(dtype);
    if (R < 1 || R > AR_MAX_RANKS || n == 0 || esize == 0 || hidden < 0)
        return 0;
    size_t fused = 0;
    if (hidden > 0) {
        if (n % static_cast<size_t>(hidden) != 0 || n / static_cast<size_t>(hidden) > static_cast<size_t>(INT32_MAX))
            return 0;
        fused = ar_workspace_size_rows(R, hidden, static_cast<int>(n / static_cast<size_t>(hidden)), dtype);
    }
    return static_cast<size_t>(R) * round256(n * esize) + fused;
}

int ar_allreduce_config(const ar_params* p, int fusion_op, int strategy, int config, ar_stream_t stream)
{
    if (p == nullptr)
        return AR_ERR_INVALID_ARG;
    if ((config & ~(AR_CONFIG_USE_MEMCPY | AR_CONFIG_RESIDUAL_RMS_NORM)) != 0)
        return AR_ERR_UNSUPPORTED;
    const int op = (config & AR_CONFIG_RESIDUAL_RMS_NORM) ? AR_FUSION_RESIDUAL_RMS_NORM : fusion_op;
    if (!(config & AR_CONFIG_USE_MEMCPY))
        return ar_allreduce(p, op, strategy, stream);
    if (op != AR_FUSION_NONE && op != AR_FUSION_RESIDUAL_RMS_NORM)
        return AR_ERR_UNSUPPORTED;
    if (p->R < 1 || p->R > AR_MAX_RANKS)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(p->dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (p->n == 0)
        return ar_allreduce(p, op, strategy, stream);
    for (int r = 0; r < p->R; ++r)
        if (p->partials[r] == nullptr)
            return AR_ERR_INVALID_ARG;
    const int hidden = op == AR_FUSION_RESIDUAL_RMS_NORM ? p->hidden : 0;
    if (op == AR_FUSION_RESIDUAL_RMS_NORM && (p->hidden < 1 || p->n % static_cast<size_t>(p->hidden) != 0))
        return AR_ERR_INVALID_ARG;
    const size_t need = ar_config_workspace_size(p->R, p->n, hidden, p->dtype);
    if (need == 0)
        return AR_ERR_INVALID_ARG;
    if (p->workspace == nullptr || p->workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
        return AR_ERR_WORKSPACE;
    // Stage every partial into its slot of the registered buffer, then reduce
    // from the slots (the USE_MEMCPY route of AllReduceDispatchMemcpy).
    const size_t slot = round256(p->n * esize);
    char* ws = static_cast<char*>(p->workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ar_params q = *p;
    for (int r = 0; r < p->R; ++r) {
        if (cudaMemcpyAsync(ws + r * slot, p->partials[r], p->n * esize, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return AR_ERR_CUDA;
        q.partials[r] = ws + r * slot;
    }
    q.workspace = ws + static_cast<size_t>(p->R) * slot;
    q.workspace_bytes = p->workspace_bytes - static_cast<size_t>(p->R) * slot;
    return ar_allreduce(&q, op, strategy, stream);
}

int ar_query_strategy(int R, size_t n, int hidden, int dtype, int fusion_op, int* chosen,
                      int* warps_per_token)
{
    if (R < 1 || R > AR_MAX_RANKS || chosen == nullptr)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (fusion_op == AR_FUSION_NONE) {
        // The partition of the packed path (16-byte aligned pointers).
        *chosen = sum_auto_strategy(esize, R, n, true);
        if (warps_per_token)
            *warps_per_token = 0;
        return AR_OK;
    }
    if (fusion_op != AR_FUSION_RESIDUAL_RMS_NORM)
        return AR_ERR_UNSUPPORTED;
    if (hidden < 1 || n % static_cast<size_t>(hidden) != 0 ||
        n / static_cast<size_t>(hidden) > static_cast<size_t>(INT32_MAX))
        return AR_ERR_INVALID_ARG;
    const int tokens = static_cast<int>(n / static_cast<size_t>(hidden));
    const bool packed = hidden % (16 / esize) == 0;
    FusedPlan plan = plan_fused(esize, R, hidden, tokens, packed, AR_AUTO);
    *chosen = plan.strategy;
    const int row_threads = plan.shape.tpr * (plan.shape.mode == ar::kCluster ? plan.shape.cluster : 1);
    if (warps_per_token)
        *warps_per_token = plan.strategy == AR_ONESHOT ? (row_threads + 31) / 32 : 0;
    return AR_OK;
}

size_t ar_lamport_buffer_size(int R, int hidden, int tokens, int dtype)
{
    const int esize = esize_of(dtype);
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0 || esize == 0)
        return 0;
    const int lanes = 16 / esize;
    OneShotShape sh{};
    if (hidden % lanes != 0 || !lamport_shape(hidden / lanes, tokens, lanes, R, &sh))
        return 0;
    return round256(lamport_buffer_bytes(R, hidden, tokens, esize, sh));
}

int ar_lamport_init(void* buffer, size_t bytes, int dtype, ar_stream_t stream)
{
    if (esize_of(dtype) == 0)
        return AR_ERR_UNSUPPORTED;
    if (buffer == nullptr || !aligned16(buffer) || bytes % 2 != 0)
        return AR_ERR_INVALID_ARG;
    if (bytes == 0)
        return AR_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return status_of(by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        return ar::launch_lamport_fill<T>(buffer, bytes, s);
    }));
}

int ar_lamport_supported(int R, int hidden, int tokens, int dtype, int* warps_per_token)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    const int lanes = 16 / esize;
    OneShotShape sh{};
    if (hidden % lanes != 0 || !lamport_shape(hidden / lanes, tokens, lanes, R, &sh))
        return AR_ERR_UNSUPPORTED;
    if (warps_per_token)
        *warps_per_token = (sh.tpr * (sh.mode == ar::kCluster ? sh.cluster : 1) + 31) / 32;
    return AR_OK;
}

int ar_residual_rmsnorm_lamport(const void* const* partials, int R, const void* bias, const void* residual,
                                const void* weight, float eps, int hidden, int tokens, void* out,
                                void* residual_out, void* lamport_buffer, size_t lamport_bytes, int dtype,
                                ar_stream_t stream)
{
    if (R < 1 || R > AR_MAX_RANKS || hidden < 1 || tokens < 0)
        return AR_ERR_INVALID_ARG;
    const int esize = esize_of(dtype);
    if (esize == 0)
        return AR_ERR_UNSUPPORTED;
    if (!std::isfinite(eps) || eps < 0.0f)
        return AR_ERR_INVALID_ARG;
    if (tokens == 0)
        return AR_OK;
    if (partials == nullptr || residual == nullptr || weight == nullptr || out == nullptr ||
        residual_out == nullptr || out == residual_out)
        return AR_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        if (partials[r] == nullptr)
            return AR_ERR_INVALID_ARG;
    const int lanes = 16 / esize;
    bool packed = hidden % lanes == 0 && aligned16(residual) && aligned16(weight) && aligned16(out) &&
                  aligned16(residual_out) && (bias == nullptr || aligned16(bias));
    for (int r = 0; r < R; ++r)
        packed = packed && aligned16(partials[r]);
    if (!packed)
        return AR_ERR_UNSUPPORTED;
    const int units_row = hidden / lanes;
    OneShotShape sh{};
    if (!lamport_shape(units_row, tokens, lanes, R, &sh))
        return AR_ERR_UNSUPPORTED;
    const size_t need = lamport_buffer_bytes(R, hidden, tokens, esize, sh);
    if (lamport_buffer == nullptr || !aligned16(lamport_buffer) || lamport_bytes < need)
        return AR_ERR_WORKSPACE;

    FusedArgs a{};
    for (int r = 0; r < R; ++r)
        a.partials[r] = partials[r];
    a.bias = bias;
    a.residual = residual;
    a.weight = weight;
    a.out = out;
    a.residual_out = residual_out;
    a.R = R;
    a.hidden = hidden;
    a.tokens = tokens;
    a.units_row = units_row;
    a.eps = eps;
    a.early_residual = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int skip = test_lamport_skip_rank();
    const cudaError_t e = by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        return ar::launch_fused_lamport<T>(a, lamport_buffer, sh, skip < R ? skip : -1, next_lamport_epoch(), s);
    });
    if (e == cudaErrorInvalidConfiguration || e == cudaErrorCooperativeLaunchTooLarge ||
        e == cudaErrorNotSupported)
        return AR_ERR_UNSUPPORTED;
    return status_of(e);
}

}  // extern "C"
