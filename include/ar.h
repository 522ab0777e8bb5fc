/*
 * ar.h -- C ABI of the single-GPU R-way all-reduce (sum) and the fused
 * sum + bias + residual + RMSNorm that follows a row-parallel linear layer.
 *
 * The R "rank" partials are R device buffers in the memory of ONE GPU; they
 * stand in for the peer buffers that the TensorRT-LLM all-reduce reads
 * through AllReduceParams::peer_comm_buffer_ptrs[MAX_RANKS_PER_NODE]
 * ("type.d2", AllReduceParams).  There is no second GPU, no NCCL and no
 * cross-device barrier: the partials are complete when the call is issued
 * on a stream ordered after their producers.
 *
 * Conventions shared by every entry point
 *   - Return value: an int status (AR_OK or a negative AR_ERR_* code),
 *     after the plugin's int32 enqueue(..., workspace, stream) noexcept
 *     ("All Reduce Plugin", IPluginV3OneRuntime::enqueue).  No C++
 *     exception crosses the ABI.
 *   - Asynchrony: calls enqueue kernels on `stream` and return at once.
 *     A launch failure reported by the CUDA runtime maps to AR_ERR_CUDA.
 *     Argument errors are detected on the host before anything is launched.
 *   - Memory: every buffer is owned by the caller and lives in device
 *     memory of the current device.  The `partials` array itself is a HOST
 *     array of R device pointers; it is read during the call only.  The
 *     library allocates nothing.  Its only device state is the scratch
 *     array of ar_residual_rmsnorm_noalloc and a count of bounded waits
 *     that gave up (ar_device_status); every other call is thread-safe.
 *   - Layout: tensors are dense and row-major.  The fused call sees
 *     [tokens, hidden] rows; bias and weight are [hidden]; every tensor of
 *     one call has the same element type (ar_dtype); eps is a float.
 *   - Alignment: 16-byte aligned pointers (and, for the fused call, hidden a
 *     multiple of 16/sizeof(element)) take the 16-byte packed path; anything
 *     else takes a slower element-wise path.  Misalignment is not an error,
 *     except for ar_residual_rmsnorm_lamport, which has the packed path only
 *     and returns AR_ERR_UNSUPPORTED.
 *   - Aliasing: out may be one of partials[r] and residual_out may be
 *     residual (each element is read before it is written).  out and
 *     residual_out must differ.  Any other overlap is undefined.
 *   - Empty input (n == 0 or tokens == 0) returns AR_OK and launches nothing.
 *   - Determinism: the sum of every element is accumulated in fp32 in the
 *     fixed order partials[0], ..., partials[R-1], bias, residual, and every
 *     row reduction uses a fixed tree, so results are bit-identical from run
 *     to run.  residual_out is also bit-identical across strategies, and
 *     equal in value through the Lamport-style call (which may flip the sign
 *     of an exact zero).
 */
#ifndef TENSOR_ALLREDUCE_RESIDUAL_AR_H
#define TENSOR_ALLREDUCE_RESIDUAL_AR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* ar_stream_t;

/* Element types.  "type.d2" (PackedOn16Bytes<T>) packs float (4 lanes) and
 * half (8 lanes) into 16 bytes; bfloat16 (8 lanes) is added beside them. */
typedef enum { AR_FP32 = 0, AR_FP16 = 1, AR_BF16 = 2 } ar_dtype;

/* Strategy codes: the values of AllReduceStrategyType ("type.d2").
 * NCCL is recognised but rejected (one GPU, no NCCL). */
typedef enum { AR_NCCL = 0, AR_ONESHOT = 1, AR_TWOSHOT = 2, AR_AUTO = 3 } ar_strategy;

/* Fusion codes: the values of AllReduceFusionOp ("type.d2"). */
typedef enum { AR_FUSION_NONE = 0, AR_FUSION_RESIDUAL_RMS_NORM = 1 } ar_fusion_op;

enum {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = -1,  /* bad R, NULL required pointer, bad size, eps < 0 ... */
    AR_ERR_UNSUPPORTED = -2,  /* NCCL strategy, unknown dtype/strategy/fusion, row too long for ONESHOT */
    AR_ERR_WORKSPACE = -3,    /* TWOSHOT fused without a large enough workspace */
    AR_ERR_CUDA = -4,         /* the CUDA runtime reported an error at launch */
    AR_ERR_TIMEOUT = -5       /* a kernel gave up a bounded wait (see ar_device_status) */
};

/* MAX_RANKS_PER_NODE ("type.d2", AllReduceParams::peer_comm_buffer_ptrs):
 * the pages name the bound but not its value. */
#define AR_MAX_RANKS 16

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int ar_version(void);

/* Text for a status code.  Never NULL; the string is static. */
const char* ar_strerror(int code);

/*
 * ar_workspace_size -- analogue of getMaxRequiredWorkspaceSize
 * ("allreduce.d2", common/customAllReduceUtils.h, reached from
 * selectImplementation and from CustomAllReduceHelper.max_workspace_size_auto).
 *
 * Bytes of device workspace that cover ANY fused call of R partials whose
 * tokens * hidden <= n, with either strategy, rounded up to 256.  The
 * workspace holds one fp32 partial sum of squares per (row, chunk) of the
 * two-shot path; the bound is reached by hidden == 1.  Returns 0 when
 * R < 1, R > AR_MAX_RANKS, n == 0 or dtype is unknown.
 */
size_t ar_workspace_size(int R, size_t n, int dtype);

/* Exact workspace bytes for a fused call of this shape (rounded up to 256);
 * 0 if the shape is invalid. */
size_t ar_workspace_size_rows(int R, int hidden, int tokens, int dtype);

/*
 * ar_sum -- out[i] = sum over r of partials[r][i], i < n.
 * The all-reduce (sum) of the tensor-parallel ranks' partial activations
 * ("All Reduce Plugin", AllReducePlugin description), computed by the
 * oneShotAllReduceKernel / twoShotAllReduceKernel routes of
 * AllReduceDispatch ("allreduce.d2").
 *
 *   partials  host array of R device pointers, each to n elements
 *   R         1 .. AR_MAX_RANKS.  R == 1 is the tpSize == 1 passthrough
 *             ("All Reduce Plugin": passthrough without tensor parallelism):
 *             a device copy, or nothing at all when out == partials[0].
 *   out       device pointer to n elements (may equal one of partials[r])
 *   n         element count
 *   dtype     ar_dtype
 *   strategy  AR_ONESHOT: every block reduces a slice of the whole tensor.
 *             AR_TWOSHOT: the tensor is cut into R rank slices and block
 *             group r reduces slice r (the reduce-scatter; the all-gather
 *             is void on one GPU because the slices land in out directly).
 *             AR_AUTO: chosen by ar_query_strategy.  Values are
 *             bit-identical across strategies.
 * Errors: AR_ERR_INVALID_ARG (R out of range, NULL pointer with n > 0),
 *         AR_ERR_UNSUPPORTED (AR_NCCL, unknown dtype or strategy),
 *         AR_ERR_CUDA.
 */
int ar_sum(const void* const* partials, int R, void* out, size_t n,
           int dtype, int strategy, ar_stream_t stream);

/*
 * ar_residual_rmsnorm -- the RESIDUAL_RMS_NORM fusion (AllReduceFusionOp and
 * AllReduceFusionParams in "type.d2"; the one-shot
 * one_shot_all_reduce_norm_kernel -> rms_norm route and the two-shot
 * twoShotAllReduceKernel -> rms_norm_kernel route of AllReduceNormKernelLaunch
 * in "allreduce.d2").  For every row t < tokens and column j < hidden:
 *
 *     x[t,j]            = sum_r partials[r][t,j] + bias[j] + residual[t,j]
 *     residual_out[t,j] = x[t,j]                               (pre-norm sum)
 *     out[t,j]          = x[t,j] / sqrt(mean_j(x[t,:]^2) + eps) * weight[j]
 *
 * The pages name the fields but print no formula; this is the textbook
 * RMSNorm (eps inside the square root, no mean subtraction, no offset).
 * x is accumulated in fp32 in the order partials[0..R-1], bias, residual.
 *
 *   partials      host array of R device pointers, each [tokens, hidden]
 *   bias          device [hidden], or NULL for no bias (the GEMM bias,
 *                 added once after the sum, not once per rank)
 *   residual      device [tokens, hidden]
 *   weight        device [hidden]
 *   eps           float, >= 0 (AllReduceFusionParams::eps is a float)
 *   out           device [tokens, hidden]: the normalised rows
 *   residual_out  device [tokens, hidden]: the pre-norm sum x, which the
 *                 pages call intermediate_buffer; may equal residual
 *   intermediate  device workspace for AR_TWOSHOT (fp32 per-chunk sums of
 *                 squares); may be NULL for AR_ONESHOT
 *   intermediate_bytes  its size; at least ar_workspace_size_rows(...)
 *   strategy      AR_ONESHOT: one kernel, each row held on chip between the
 *                 sum and the norm (one pass over HBM).
 *                 AR_TWOSHOT: phase 1 writes residual_out and the per-chunk
 *                 sums of squares, phase 2 normalises residual_out.
 *                 AR_AUTO: chosen by ar_query_strategy; falls back to
 *                 ONESHOT when the workspace is missing or too small.
 * Errors: AR_ERR_INVALID_ARG (R out of range, hidden < 1, tokens < 0, NULL
 *         required pointer, eps < 0 or not finite, out == residual_out),
 *         AR_ERR_UNSUPPORTED (AR_NCCL, unknown dtype or strategy, a row too
 *         long for AR_ONESHOT), AR_ERR_WORKSPACE (AR_TWOSHOT without a large
 *         enough workspace), AR_ERR_CUDA.
 */
int ar_residual_rmsnorm(const void* const* partials, int R, const void* bias,
                        const void* residual, const void* weight, float eps,
                        int hidden, int tokens, void* out, void* residual_out,
                        void* intermediate, size_t intermediate_bytes,
                        int dtype, int strategy, ar_stream_t stream);

/*
 * ar_rmsnorm -- out[t,j] = x[t,j] / sqrt(mean_j(x[t,:]^2) + eps) * weight[j],
 * the row normalisation on its own: rms_norm_kernel_launcher ->
 * rms_norm_kernel of "allreduce.d2", which the pages run after a plain
 * all-reduce and as the second phase of the two-shot fused route.  With
 * ar_sum before it this is the unfused route of the fused call.
 *
 *   x       device [tokens, hidden]; out may equal x (in place)
 *   weight  device [hidden]
 *   eps     float, >= 0
 *   out     device [tokens, hidden]
 * Each row is held in registers between its sum of squares and its output,
 * so hidden <= 16384.  Same accumulation (fp32, fixed reduction tree) and
 * alignment rules as ar_residual_rmsnorm.  tokens == 0 launches nothing.
 * Errors: AR_ERR_INVALID_ARG (hidden < 1, tokens < 0, NULL pointer, eps < 0
 *         or not finite), AR_ERR_UNSUPPORTED (unknown dtype, hidden > 16384),
 *         AR_ERR_CUDA.
 */
int ar_rmsnorm(const void* x, const void* weight, float eps, int hidden, int tokens, void* out,
               int dtype, ar_stream_t stream);

/*
 * ar_host_staging_size -- bytes of device staging that
 * ar_residual_rmsnorm_host needs for chunks of `chunk_tokens` rows: two
 * buffers of (R + 3) [chunk_tokens, hidden] tensors plus a two-shot
 * workspace each, then weight and bias (all 256-byte aligned).  0 for an
 * invalid shape.
 */
size_t ar_host_staging_size(int R, int hidden, int chunk_tokens, int dtype);

/*
 * ar_residual_rmsnorm_host -- ar_residual_rmsnorm on tensors in HOST memory
 * (partials, bias, residual, weight, out, residual_out: same shapes and
 * meaning), for data that is not resident on the device.  The call copies
 * the rows in chunks of chunk_tokens rows (the last chunk_tokens rows in
 * shrinking pieces, halves until at most 128 rows are left, so that little
 * is left to do after the last copy in) into `staging` (device memory of at least
 * ar_host_staging_size(R, hidden, chunk_tokens, dtype) bytes, 256-byte
 * aligned, owned by the caller), runs the fused kernels on each chunk on
 * `stream`, and copies the outputs back, with the copies of chunk i+1 and
 * i-1 overlapping the kernels of chunk i (two staging buffers, two copy
 * streams).  No pages' counterpart: the plugin of "All Reduce Plugin"
 * works on device tensors only.
 *
 * Asynchronous like every call here: it returns once everything is queued.
 * Work queued on `stream` before the call happens before the first copy,
 * and work queued on `stream` after it sees the outputs in host memory (so
 * cudaStreamSynchronize(stream) waits for them).  Host buffers must stay
 * valid and unchanged until then; they should be pinned (cudaHostAlloc /
 * cudaHostRegister), otherwise the copies do not overlap.  The first call
 * on a device creates two streams and a few events there and keeps them
 * for the life of the process.  Calls that may run at the same time need
 * separate staging buffers.
 * Errors: as ar_residual_rmsnorm, plus AR_ERR_INVALID_ARG (chunk_tokens < 1,
 *         NULL staging) and AR_ERR_WORKSPACE (staging too small or not
 *         256-byte aligned).
 */
int ar_residual_rmsnorm_host(const void* const* partials, int R, const void* bias,
                             const void* residual, const void* weight, float eps,
                             int hidden, int tokens, void* out, void* residual_out,
                             void* staging, size_t staging_bytes, int chunk_tokens,
                             int dtype, int strategy, ar_stream_t stream);

/*
 * ar_params -- one structure holding every argument, after AllReduceParams
 * (elts_total, peer_comm_buffer_ptrs, local_output_buffer_ptr) and its
 * AllReduceFusionParams member (bias_buffer, residual_buffer, hidden_size,
 * weight_buffer, eps, intermediate_buffer) in "type.d2".  local_rank and
 * deserialize() have no counterpart: there are no peer processes.
 */
typedef struct {
    const void* partials[AR_MAX_RANKS]; /* peer_comm_buffer_ptrs, first R used */
    int R;
    int dtype;                          /* ar_dtype */
    size_t n;                           /* elts_total (tokens * hidden when fused) */
    void* out;                          /* local_output_buffer_ptr */
    const void* bias;                   /* bias_buffer, nullable */
    const void* residual;               /* residual_buffer */
    const void* weight;                 /* weight_buffer */
    float eps;                          /* eps */
    int hidden;                         /* hidden_size */
    void* residual_out;                 /* intermediate_buffer: the pre-norm sum */
    void* workspace;                    /* two-shot sums of squares */
    size_t workspace_bytes;
} ar_params;

/* Dispatch on the fusion op, after customAllReduce -> AllReduceDispatchMemcpy
 * ("allreduce.d2"): AR_FUSION_NONE calls ar_sum (bias, residual, weight,
 * residual_out and workspace ignored); AR_FUSION_RESIDUAL_RMS_NORM calls
 * ar_residual_rmsnorm with tokens = n / hidden (n must be a multiple of
 * hidden).  Same errors as those two; AR_ERR_INVALID_ARG for a NULL p. */
int ar_allreduce(const ar_params* p, int fusion_op, int strategy, ar_stream_t stream);

/* AllReduceStrategyConfig bit flags ("type.d2"). */
enum { AR_CONFIG_USE_MEMCPY = 1, AR_CONFIG_RESIDUAL_RMS_NORM = 2 };

/*
 * ar_config_workspace_size -- workspace bytes ar_allreduce_config needs with
 * AR_CONFIG_USE_MEMCPY for R partials of n elements (hidden > 0 for the
 * fused op, whose two-shot sums of squares follow the copies; 0 for the
 * sum): R slots of n elements, each rounded up to 256 bytes, plus the
 * fused workspace.  0 for an invalid shape.
 */
size_t ar_config_workspace_size(int R, size_t n, int hidden, int dtype);

/*
 * ar_allreduce_config -- ar_allreduce with the AllReduceStrategyConfig flags
 * of "type.d2" (the `config` of AllReduceDispatchMemcpy in "allreduce.d2").
 *   AR_CONFIG_RESIDUAL_RMS_NORM  run the fused op whatever fusion_op says.
 *   AR_CONFIG_USE_MEMCPY         first copy every partials[r] (device to
 *       device, on `stream`) into slot r of p->workspace, the caller's
 *       registered buffer, and reduce from the copies; the fused op's
 *       two-shot workspace follows the R slots.  p->workspace must be
 *       256-byte aligned and hold ar_config_workspace_size(...) bytes.
 *       On one GPU this only adds the copies' traffic: it measures what
 *       staging the inputs costs against reading them in place.
 * Results are bit-identical to ar_allreduce's.
 * Errors: those of ar_allreduce, AR_ERR_UNSUPPORTED for unknown config
 *         bits, AR_ERR_WORKSPACE for a missing, misaligned or small
 *         workspace with AR_CONFIG_USE_MEMCPY, AR_ERR_CUDA if a copy cannot
 *         be queued.  Argument errors of the reduction itself are found
 *         after the copies are queued.
 */
int ar_allreduce_config(const ar_params* p, int fusion_op, int strategy, int config, ar_stream_t stream);

/*
 * ar_query_strategy -- what AR_AUTO resolves to (the selectImplementation /
 * kernelLaunchConfig / heuristic_min_warp_number analogue, "allreduce.d2").
 * For the fused op n = tokens * hidden.  *chosen receives AR_ONESHOT or
 * AR_TWOSHOT; *warps_per_token (nullable) receives the warps that cooperate
 * on one row in the one-shot fused kernel (0 for the reduce-only op, and
 * for the two-shot fused op, whose blocks each cover a chunk of a row).
 * The choice assumes a workspace is available.
 * Errors: AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED.
 */
int ar_query_strategy(int R, size_t n, int hidden, int dtype, int fusion_op,
                      int* chosen, int* warps_per_token);

/* Kernels a fused call can run (ar_launch_plan::kernel). */
typedef enum {
    AR_KERNEL_ONESHOT_REGISTERS = 1,  /* k_fused_oneshot, row sums in registers */
    AR_KERNEL_ONESHOT_SHARED = 2,     /* k_fused_oneshot, row sums in shared memory */
    AR_KERNEL_ONESHOT_PERSISTENT = 3, /* k_fused_oneshot_persist */
    AR_KERNEL_ONESHOT_BULK = 4,       /* k_fused_oneshot_tma: persistent, fed by bulk copies */
    AR_KERNEL_TWOSHOT = 5,            /* k_twoshot_phase1 then k_twoshot_phase2 */
    AR_KERNEL_ONESHOT_CLUSTER = 6     /* k_fused_oneshot_cluster: a row split across a block cluster */
} ar_kernel;

/* Launch plan of a fused call (see ar_query_launch). */
typedef struct {
    int strategy;          /* AR_ONESHOT or AR_TWOSHOT */
    int kernel;            /* ar_kernel */
    int threads_per_row;   /* threads that cooperate on one row */
    int units_per_thread;  /* one-shot: 16-byte vectors (or elements) per thread per row;
                              bulk-copy kernel: chunks per row */
    int rows_per_block;    /* rows a block holds at once */
    int threads_per_block;
    int blocks_per_sm;     /* persistent kernels: blocks per SM the grid is sized for; else 0 */
    int stages;            /* bulk-copy kernel: ring slots per block; else 0 */
    int smem_bytes;        /* dynamic shared memory per block */
    int early_residual;    /* one-shot: residual_out written before the row's norm is known */
    int cluster;           /* row-split kernel: blocks (one cluster) per row; else 0 */
} ar_launch_plan;

/*
 * ar_query_launch -- the kernel and launch shape that ar_residual_rmsnorm
 * would use for this shape and strategy, assuming 16-byte aligned pointers
 * and a large enough workspace (the kernelLaunchConfig /
 * heuristic_min_warp_number analogue, "allreduce.d2").  Launches nothing.
 * Errors: AR_ERR_INVALID_ARG (bad R, hidden, tokens or NULL plan),
 *         AR_ERR_UNSUPPORTED (unknown dtype or strategy, AR_NCCL, or
 *         AR_ONESHOT for a row too long for the one-shot kernels).
 */
int ar_query_launch(int R, int hidden, int tokens, int dtype, int strategy, ar_launch_plan* plan);

/*
 * ar_device_status -- whether any kernel of this library on the current
 * device gave up a bounded wait since the last call.  The one-shot fused
 * kernel that streams rows through a shared-memory ring waits on barriers
 * that its own copies complete; each such wait is limited to one second,
 * after which the kernel stops early (its outputs are then incomplete),
 * records the event and returns instead of hanging.  No pages' counterpart:
 * the pages' kernels wait on peer GPUs through block_barrier /
 * multi_gpu_barrier ("allreduce.d2"), which have no equivalent here.
 * Returns AR_OK (nothing recorded), AR_ERR_TIMEOUT (something was recorded;
 * the record is cleared), or AR_ERR_CUDA.  Synchronous: it reads device
 * memory, so it waits for work queued on the legacy default stream.
 */
int ar_device_status(void);

/* Size of the scratch array that ar_residual_rmsnorm_noalloc uses (1 MiB). */
#define AR_NOALLOC_SCRATCH_BYTES ((size_t)1 << 20)

/*
 * ar_residual_rmsnorm_noalloc -- ar_residual_rmsnorm with strategy
 * AR_TWOSHOT, except that the two-shot scratch (the per-chunk sums of
 * squares) is not a caller buffer: it is an array of AR_NOALLOC_SCRATCH_BYTES
 * that the library keeps in device memory.  The pages have no counterpart of
 * this call.  It is for callers that cannot obtain device memory at the
 * point of the call: code running under an allocator that owns all of the
 * device's memory (a framework's caching pool, an inference engine that
 * hands out memory only when it is built), or code that must not call
 * cudaMalloc / cudaFree because they can wait on work already running on the
 * device.  Inputs and outputs are still the caller's buffers, with the same
 * meaning, layout, aliasing rules and results as in ar_residual_rmsnorm.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 * Limit: a call is accepted when ar_workspace_size_rows(R, hidden, tokens,
 *   dtype) <= AR_NOALLOC_SCRATCH_BYTES (for example up to 16384 tokens of
 *   hidden 8192, whatever the pointers' alignment).  Larger calls return
 *   AR_ERR_WORKSPACE before anything is launched.
 * Memory: every device that loads the library holds its own copy of the
 *   array until the process exits.
 * Set-up: the first call on a device, with that device current, looks up
 *   the array's device address (cudaGetSymbolAddress) and keeps it for
 *   later calls; make that first call before any stream capture begins.
 *   The address is kept together with the id of the CUDA context it
 *   belongs to: after cudaDeviceReset (which destroys the array with its
 *   context), or from another context the caller has made current, the
 *   next call looks the address up again, and that call too belongs before
 *   any stream capture.  A failed look-up returns AR_ERR_CUDA.
 * Sharing: all calls on a device use the same array and it keeps what the
 *   last call wrote.  Each call writes every entry it reads before reading
 *   it, so nothing is cleared between calls.  Calls whose work overlaps on
 *   the GPU (different streams not ordered by events, or several host
 *   threads) race on the array and may return wrong results: order them.
 * Errors: those of ar_residual_rmsnorm with AR_TWOSHOT, plus AR_ERR_WORKSPACE
 *   for a call beyond the limit and AR_ERR_UNSUPPORTED for a device index
 *   of 64 or more.
 */
int ar_residual_rmsnorm_noalloc(const void* const* partials, int R, const void* bias,
                                const void* residual, const void* weight, float eps,
                                int hidden, int tokens, void* out, void* residual_out,
                                int dtype, ar_stream_t stream);

/*
 * Lamport-style fused call (lamport_style_one_shot_all_reduce_norm_kernel
 * and its launcher, is_lamport_supported and heuristic_min_warp_number,
 * "allreduce.d2").  The pages name these steps but do not spell them out;
 * this is the protocol those names stand for, on one GPU:
 *   - a communication buffer holds one slot per rank, filled beforehand with
 *     an "empty" marker, the negative zero of the element type;
 *   - each rank writes its partial into its slot, storing any -0.0 element
 *     as +0.0 so that no data element equals the marker;
 *   - the reducer reads each element of every slot until it is no longer
 *     the marker (the data is its own ready flag: no barrier, no flag
 *     word), computes the fused op, and writes the marker back, leaving the
 *     buffer empty for the next call.
 * Here the R ranks' writes are made by the same kernel launch that reduces
 * (one cooperative launch: its blocks push first, then reduce rows pushed
 * by other blocks), so the call reads the R partials like the other fused
 * calls and returns the same out and residual_out, except that an element
 * of residual_out or out that is an exact zero may have the other sign.
 * On one GPU it moves more bytes through L2 than the one-shot call (the
 * buffer is written, read and emptied: 3 * R * tokens * hidden elements
 * more), and it is provided for the protocol, not for speed.
 *
 * Buffer layout: 4096 bytes of progress words (one per block of the
 *   launch: they tell a block when a ring row has been emptied), then slot
 *   r = [slot_rows][hidden] elements at offset 4096 + r * slot_rows * hidden
 *   * element size, then 64 bytes per token of exchange area for rows split
 *   over several blocks.  The slots are a ring:
 *   row k of a call uses ring row k mod ring_rows, where ring_rows (at most
 *   slot_rows) covers two steps of the launch's row groups, so a slot holds
 *   at most 1024 row groups (one to several rows each, by the launch shape)
 *   however many tokens the call has; a row beyond the ring waits for its
 *   ring row to be emptied by the reduce of the row before it.
 *   ar_lamport_buffer_size gives the bytes.  The buffer is caller-owned
 *   device memory, 16-byte aligned, and must hold the marker everywhere
 *   before its first call: fill it once with ar_lamport_init; every call
 *   that completes leaves its slots and exchange area that way (the progress
 *   words it leaves are never mistaken for a later call's).  A buffer filled for one element type
 *   serves calls of that type only (the fp32 and 16-bit markers differ).
 *   Calls that share a buffer must be ordered (one stream, or events).
 */

/* Bytes of the Lamport buffer for R partials of [tokens, hidden] elements
 * (the R ring slots and the exchange area, rounded up to 256); 0 for bad
 * arguments or a shape the call cannot take (ar_lamport_supported). */
size_t ar_lamport_buffer_size(int R, int hidden, int tokens, int dtype);

/*
 * ar_lamport_init -- fills `bytes` of `buffer` with the empty marker of
 * `dtype`, asynchronously on `stream`.  buffer: device memory, 16-byte
 * aligned; bytes: even (0 does nothing).
 * Errors: AR_ERR_INVALID_ARG (NULL or misaligned buffer, odd bytes),
 *         AR_ERR_UNSUPPORTED (unknown dtype), AR_ERR_CUDA.
 */
int ar_lamport_init(void* buffer, size_t bytes, int dtype, ar_stream_t stream);

/*
 * ar_lamport_supported -- the is_lamport_supported analogue: AR_OK if the
 * Lamport call can take this shape, with *warps_per_token (nullable) set to
 * the warps that reduce one row (the heuristic_min_warp_number analogue).
 * The shape must have hidden a multiple of 16 / element size and a row that
 * fits: at most 512 threads (256 when a thread holds more than 16 values)
 * reduce a row, up to 8 16-byte vectors a thread, except that up to 8
 * tokens whose R partials hold at least 8192 vectors a row are split over 4
 * such blocks.  So rows of up to 2048 vectors (16384 fp16 / bf16, 8192 fp32
 * elements) are always taken, and up to 4 times longer ones in that split
 * case.  From 1024 tokens, where a row's reducing threads number at most
 * 256 with at most 4 vectors each, or at most 512 with at most 2, the same
 * block also holds as many threads again that push the partials (blocks of
 * up to 1024 threads).
 * Host-side only: launches nothing.  Pointer alignment is checked by the
 * call itself.
 * Errors: AR_ERR_INVALID_ARG (bad R, hidden or tokens),
 *         AR_ERR_UNSUPPORTED (unknown dtype, or a shape the call cannot take).
 */
int ar_lamport_supported(int R, int hidden, int tokens, int dtype, int* warps_per_token);

/*
 * ar_residual_rmsnorm_lamport -- the fused op of ar_residual_rmsnorm (same
 * arguments with the same meaning and layout; no strategy, and the
 * Lamport buffer in place of the two-shot workspace) through the Lamport
 * protocol.
 *   lamport_buffer  device buffer of at least ar_lamport_buffer_size(R,
 *                   hidden, tokens, dtype) bytes, 16-byte aligned, filled
 *                   with the marker (ar_lamport_init) and left so on return.
 * Aliasing: residual_out may be residual and out may be a partial (each
 *   partial element is pushed before anything that depends on it is
 *   written); the buffer may not overlap any other argument.
 * Requirements: every tensor pointer 16-byte aligned and hidden a multiple
 *   of 16 / element size (the 16-byte packed path); otherwise
 *   AR_ERR_UNSUPPORTED.
 * Waits: each poll of an element gives up after one second; the kernel then
 *   finishes without hanging, its outputs are incomplete, the event is
 *   recorded for ar_device_status (AR_ERR_TIMEOUT), and the buffer must be
 *   filled again with ar_lamport_init before it is used again.
 * Errors: those of ar_residual_rmsnorm, plus AR_ERR_WORKSPACE for a NULL,
 *   misaligned or too small buffer; AR_ERR_UNSUPPORTED as above, or if the
 *   device cannot make the launch cooperative.
 */
int ar_residual_rmsnorm_lamport(const void* const* partials, int R, const void* bias,
                                const void* residual, const void* weight, float eps,
                                int hidden, int tokens, void* out, void* residual_out,
                                void* lamport_buffer, size_t lamport_bytes, int dtype,
                                ar_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * The all-reduce across the GPUs of one node: one process (rank) per GPU,
 * every rank's partial in its own GPU's memory, each rank reading its peers'
 * registered buffers directly (AllReduceParams::peer_comm_buffer_ptrs
 * [MAX_RANKS_PER_NODE], "type.d2"; oneShotAllReduceKernel and
 * twoShotAllReduceKernel with their block barriers, "allreduce.d2").  Every
 * rank gets out = sum over ranks of each rank's input, accumulated in fp32 in
 * rank order (the same values on every rank, and the same values as ar_sum
 * over the R inputs).
 *
 * Set-up, on every rank: allocate (cudaMalloc, or a caching allocator's
 * device memory) ar_comm_buffer_size(world, max_bytes) bytes, export its IPC
 * handle with ar_comm_export, exchange the handles among the ranks (any
 * host-side channel: the Python binding uses torch.distributed), call
 * ar_comm_create with all of them in rank order, then pass a host-side
 * barrier among the ranks before the first ar_allreduce_peer: create zeroes
 * this rank's flag words, and no peer may signal into them before that.
 * Every rank must then make the same sequence of calls (same n, dtype and
 * strategy).  With world == 1 no handle is needed (handles may be NULL).
 *
 * Waits: every block barrier gives up after one second (a rank that never
 * arrives); the kernel then finishes without the missing data, the event is
 * recorded for ar_device_status (AR_ERR_TIMEOUT) and out is incomplete.
 * Plain peer loads and stores over NVLink; no multicast.  Not measured on more
 * than one GPU: every box this library was built and tested on has one
 * (world == 1 runs the same kernels, barrier included).
 * ---------------------------------------------------------------------------
 */
#define AR_IPC_HANDLE_BYTES 64
typedef struct ar_comm ar_comm;

/* Bytes each rank registers: 16 KiB of flag words plus two data areas of
 * max_bytes (rounded up to 256); 0 for bad arguments. */
size_t ar_comm_buffer_size(int world, size_t max_bytes);

/* Writes the AR_IPC_HANDLE_BYTES-byte CUDA IPC handle of `buffer` (device
 * memory of the current device, the start of an allocation) to `handle`
 * (host memory).  Errors: AR_ERR_INVALID_ARG, AR_ERR_CUDA. */
int ar_comm_export(const void* buffer, void* handle);

/* Creates this rank's communicator: rank in [0, world), world in
 * [1, AR_MAX_RANKS], buffer = this rank's registered buffer (16-byte
 * aligned) of buffer_bytes >= ar_comm_buffer_size(world, max_bytes),
 * handles = world * AR_IPC_HANDLE_BYTES bytes (host), rank q's at q (this
 * rank's own is not read).  Maps every peer's buffer (cudaIpcOpenMemHandle)
 * and zeroes this rank's flag words (synchronously).  On success *comm is
 * the handle to pass to ar_allreduce_peer and ar_comm_destroy.
 * Errors: AR_ERR_INVALID_ARG, AR_ERR_WORKSPACE (buffer too small),
 *         AR_ERR_CUDA (a mapping or the zeroing failed; nothing is kept). */
int ar_comm_create(int rank, int world, void* buffer, size_t buffer_bytes, size_t max_bytes, const void* handles,
                   ar_comm** comm);

/* Unmaps the peers' buffers and frees the communicator (the caller frees
 * its own buffer).  Errors: AR_ERR_INVALID_ARG, AR_ERR_CUDA. */
int ar_comm_destroy(ar_comm* comm);

/*
 * ar_allreduce_peer -- out = sum over the ranks of `input`, n elements of
 * dtype, on every rank.  input and out: this rank's device memory, 16-byte
 * aligned; out may equal input.  n * element size <= max_bytes.  The
 * current device must be the one the communicator was created on.
 *   strategy  AR_ONESHOT: every rank reads all n elements of every peer.
 *             AR_TWOSHOT: rank r reduces slice r of every peer (the
 *             reduce-scatter) and gathers the other slices from their
 *             ranks (the all-gather).  AR_AUTO: one-shot for up to 2 ranks
 *             or under 1 MiB, two-shot beyond (a size rule, not measured).
 *             Values are bit-identical across strategies.
 * Asynchronous on `stream`; stream-ordered with the calls before it.
 * After a wait gave up (AR_ERR_TIMEOUT from ar_device_status), the ranks'
 * barrier words no longer agree on the calls made: destroy the
 * communicator on every rank and create it again before the next call.
 * Errors: AR_ERR_INVALID_ARG (also: another current device),
 * AR_ERR_UNSUPPORTED (dtype, strategy, or a misaligned pointer),
 * AR_ERR_WORKSPACE (n beyond max_bytes), AR_ERR_CUDA.
 */
int ar_allreduce_peer(ar_comm* comm, const void* input, void* out, size_t n, int dtype, int strategy,
                      ar_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TENSOR_ALLREDUCE_RESIDUAL_AR_H */
