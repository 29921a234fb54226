/*
 * dt.h -- C ABI of libdt: DTensor-style tensor-parallel linears and layout
 * transforms on one GB300 (sm_103a).
 *
 * Every mesh rank is a LOGICAL shard: all P ranks' local tensors ("slots")
 * live in the HBM of one GPU, and what a multi-GPU framework does with
 * collectives is done here by one kernel over all slots.
 *
 * Sources (page title and section):
 *  - Hyper-Parallel DTensor API (MindSpore hyper-parallel pull request 121):
 *    DeviceMesh / placements / layout, distribute_tensor, redistribute,
 *    reduce_partial, full_tensor, shape, local_shape.
 *  - DTorch user guide, "Module parallel", section 3 (Linear implementation
 *    walkthrough): tp_dim, tp_shard_type, weight/bias placements and the
 *    input placement checks; section 2: EmbeddingWithReplicateOutput.
 *  - Model parallelism (wineandchord), "Tensor Parallel": Y_i = X W_i
 *    (column), Y = sum_i X_i W_i (row), weights stored [in, out].
 *  - nanotron tutorial ch. 5, sections 5.1 and 5.5: ALL_REDUCE and
 *    REDUCE_SCATTER modes of the row-parallel linear.
 *
 * Conventions for every entry point
 *  - Pointers named "device" are CUDA device pointers on the current GPU;
 *    everything else (descriptors, slot arrays, stride arrays, output
 *    scalars) is host memory that is read during the call only.
 *  - The caller owns all device memory: inputs, outputs and workspaces.  The
 *    library allocates no device memory, on any call.  A linear's workspace
 *    (its size from the *_workspace_size query of that call) holds the
 *    split tail's scratch: where the tensor-core GEMM's last wave would
 *    leave CTA pairs idle, the remaining tiles' K range is divided over all
 *    pairs and the pieces' fp32 partials meet in the workspace.  A call given
 *    no workspace, or one too small, runs every tile whole: same results up
 *    to fp32 summation order, slower where the split pays.  The workspace's
 *    contents between calls are the caller's (the library zeroes what it
 *    needs zeroed on the call's stream); calls whose kernels may overlap on
 *    the GPU need separate workspaces.
 *  - The library keeps host-side caches (TMA descriptors; launch plans keyed
 *    by the operands' layouts, slot pointers, strides, workspace and stream,
 *    so a repeated call skips planning) and, made once and kept, per device
 *    one auxiliary stream with two events (a redistribute call with both
 *    copies and Partial reductions runs the reductions there, forked from
 *    and joined back to the caller's stream).  dt_clear_cache() drops the
 *    caches.
 *  - Environment switches, read once per process:
 *      DT_GEMM_SPLIT=0     turns the split tail off; =2 splits every last
 *                          wave the finishing can take, whether or not the
 *                          cost model expects a gain (to compare schedules);
 *      DT_GEMM_BANDS=m,n   fixes the GEMM tile order's band height and block
 *                          width (in 256 x 256 tiles) instead of the host's
 *                          choice, to compare orders.
 *    Two test hooks exercise the bounded-wait exit without a fault:
 *      DT_GEMM_WAIT_LIMIT_MS=n  bounds every GEMM barrier wait at n ms
 *                               (1..10000; default 2000);
 *      DT_GEMM_STARVE=1         makes the GEMM producers issue no copies,
 *                               so every wait runs out and the launch
 *                               reports DT_DEV_ERR_TIMEOUT.
 *      DT_RD_WAIT_LIMIT_MS=n,   the same two hooks for the bulk (TMA) copy
 *      DT_RD_STARVE=1           kernel of dt_redistribute.
 *  - Compute calls are asynchronous on the given stream (a cudaStream_t;
 *    NULL = the legacy default stream).  Their return value covers the checks
 *    done on the host before any launch; on any error nothing is launched.
 *  - Errors found on the GPU are OR-ed, as DT_DEV_* bits, into the int32 at
 *    device address d_status (read it after synchronising).  Kernels never
 *    trap.  d_status may be NULL: the bits then go to a status word inside
 *    the library, read and cleared by dt_read_device_status().
 *  - Inputs and outputs must not overlap.
 *  - Empty tensors are valid operands.  A slot with no elements may have a
 *    NULL pointer and any strides.  A call with nothing to write (no tokens,
 *    no output columns) returns DT_OK without launching or calling CUDA.  A
 *    linear whose inner dim K is 0 writes its bias, or zeros.
 *  - dt_last_error() returns a human-readable reason for the last non-OK
 *    status returned on the calling thread.
 */
#ifndef DT_H_
#define DT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols keep default visibility even when the library is built
 * with -fvisibility=hidden. */
#if defined(__GNUC__)
#define DT_API __attribute__((visibility("default")))
#else
#define DT_API
#endif

#define DT_MAX_MESH_DIMS 4
#define DT_MAX_TENSOR_DIMS 4
#define DT_MAX_SLOTS 64

/* CUDA stream handle; the same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* dt_stream_t;

typedef enum dt_status {
  DT_OK = 0,
  DT_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, bad count */
  DT_ERR_SHAPE = 2,        /* shapes of the operands do not agree */
  DT_ERR_PLACEMENT = 3,    /* placement breaks the layer's rule (the DTorch
                              guide's `assert input.check_placement(...)`) */
  DT_ERR_UNSUPPORTED = 4,  /* legal in principle, not provided (e.g. Shard -> Partial) */
  DT_ERR_ALIGNMENT = 5,    /* pointer or stride alignment the kernel needs */
  DT_ERR_CUDA = 6,         /* a CUDA runtime or driver call failed */
  DT_ERR_CAPACITY = 7      /* more slots, tasks or groups than one call plans, or a
                              linear dimension at or above 2^31 - 512 (the GEMM
                              kernels' coordinates are 32-bit) */
} dt_status;

/* Bits OR-ed into *d_status by kernels. */
#define DT_DEV_ERR_INDEX 0x1   /* an embedding id was outside [0, vocab): its row was zero-filled */
#define DT_DEV_ERR_TIMEOUT 0x2 /* a bounded wait (GEMM or bulk copy kernel) gave up; its outputs are not valid */

typedef enum dt_dtype { DT_BF16 = 0, DT_FP32 = 1, DT_INT32 = 2 } dt_dtype;

/* Placement kinds (Hyper-Parallel DTensor API, placement-type table). */
typedef enum dt_pkind { DT_REPLICATE = 0, DT_SHARD = 1, DT_PARTIAL = 2 } dt_pkind;
/* Partial reductions.  SUM adds the partial values in rank order in fp32;
 * AVG divides that sum once (fp32, correctly rounded) by the number of
 * partial values; MAX keeps the largest in rank order.  bf16 results are
 * rounded once at the end.  All Partial dims of one layout use one op. */
typedef enum dt_reduce_op { DT_SUM = 0, DT_AVG = 1, DT_MAX = 2 } dt_reduce_op;

/* Row-parallel output modes (nanotron 5.1; DTorch RowParallelLinear keeps Partial). */
typedef enum dt_tp_mode {
  DT_TP_PARTIAL = 0,        /* output Partial() on tp: P materialised partial products */
  DT_TP_ALL_REDUCE = 1,     /* output Replicate() on tp: the summed product */
  DT_TP_REDUCE_SCATTER = 2  /* output Shard(0) on tp: each slot keeps a block of rows */
} dt_tp_mode;

typedef struct dt_placement {
  int32_t kind; /* dt_pkind */
  int32_t dim;  /* tensor dim for DT_SHARD; negative counts from the end */
  int32_t op;   /* dt_reduce_op for DT_PARTIAL */
} dt_placement;

/*
 * A global tensor's distribution over a logical mesh.
 *  - Ranks are numbered row-major over mesh_shape (last mesh dim fastest), as
 *    in the printed distribute_tensor example (ranks 0,1 hold rows 0-1).
 *  - A Shard splits a dim torch.chunk-style: width ceil(n/p), trailing parts
 *    may be short or empty.  Two mesh dims sharding one tensor dim nest in
 *    mesh-dim order.
 *  - Slots: with materialize_replicas == 0, ranks that differ only in their
 *    Replicate coordinates share ONE slot.  Slots are numbered row-major
 *    over the non-Replicate mesh dims.  With materialize_replicas != 0,
 *    slot == rank.
 */
typedef struct dt_layout {
  int32_t mesh_ndim;
  int32_t mesh_shape[DT_MAX_MESH_DIMS];
  dt_placement placements[DT_MAX_MESH_DIMS];
  int32_t ndim;
  int64_t gshape[DT_MAX_TENSOR_DIMS];
  int32_t dtype; /* dt_dtype */
  int32_t materialize_replicas;
} dt_layout;

/*
 * A distributed tensor: a layout plus one device pointer per slot.
 * slots[s] points at slot s's local tensor (local shape from
 * dt_layout_slot_box); it may be NULL only when that slot is empty.
 * strides: NULL for contiguous row-major slots, else a host array of
 * nslots * layout.ndim element strides (slot-major).
 */
typedef struct dt_dtensor {
  dt_layout layout;
  int32_t nslots;
  void* const* slots;
  const int64_t* strides;
} dt_dtensor;

/* ---- host-only layout queries (Hyper-Parallel DTensor API: Layout, shape, local_shape) ---- */

/* Number of slots of a layout.  Errors: DT_ERR_INVALID_ARG on a malformed layout. */
DT_API dt_status dt_layout_nslots(const dt_layout* layout, int32_t* nslots);

/* Slot holding rank `rank`'s local tensor. */
DT_API dt_status dt_layout_slot_of_rank(const dt_layout* layout, int32_t rank, int32_t* slot);

/* Local shape and global offset (layout.ndim entries each) of slot `slot`. */
DT_API dt_status dt_layout_slot_box(const dt_layout* layout, int32_t slot, int64_t* local_shape,
                             int64_t* global_offset);

/* ---- data movement ---- */

/*
 * redistribute(): move `src` to `dst` placements on the same mesh and global
 * shape (Hyper-Parallel DTensor API: redistribute, reduce_partial,
 * full_tensor, distribute_tensor).  The transitions are
 *   Shard(a) -> Shard(b)  (all-to-all),  Shard -> Replicate (all-gather),
 *   Replicate -> Shard (slicing),  Partial -> Replicate (all-reduce),
 *   Partial -> Shard (reduce-scatter),  Replicate -> Partial (coordinate 0
 *   keeps the value, the others get zeros), Partial -> Partial (kept).
 * Partial sums add the partial values of an element in rank order in fp32
 * and round a bf16 result once, to nearest even: results are bit-exact and
 * independent of the launch shape.  Shard -> Partial returns
 * DT_ERR_UNSUPPORTED; dtypes must match; int32 supports no Partial.
 * Copies whose rows are all 16-byte aligned on both sides run on the bulk
 * (TMA) copy engine, the others on a warp copy kernel; only the bulk kernel
 * waits (bounded), and a wait that gives up sets DT_DEV_ERR_TIMEOUT in
 * *d_status (NULL: the library's status word).
 */
DT_API dt_status dt_redistribute(const dt_dtensor* src, const dt_dtensor* dst, int32_t* d_status,
                          dt_stream_t stream);

/*
 * n independent redistributes, src[i] -> dst[i], each with the rules and
 * results of dt_redistribute.  The pages move one tensor per call; this
 * batched form (no counterpart there) packs the copies of all n pairs into
 * one kernel launch and their Partial reductions into one more, as far as a
 * launch's parameter block holds (128 source and 128 destination slots, 192
 * boxes, 256 partial references), and starts further launches beyond that.
 * Pairs may differ in mesh, shape, dtype and reduce op; a launch holds one
 * dtype (and, for reductions, one op), so each further dtype or op adds a
 * launch.  All tensors of a call live on one device (that of the first
 * non-empty destination slot, where the kernels run).  No dst[i] may
 * overlap any src[j] or another dst[j] of the same call: the pairs run
 * concurrently.  Every pair is checked before anything launches; an error
 * names the pair and nothing runs.  n == 0 is a no-op.
 */
DT_API dt_status dt_redistribute_batch(int32_t n, const dt_dtensor* src, const dt_dtensor* dst,
                                int32_t* d_status, dt_stream_t stream);

/*
 * EmbeddingWithReplicateOutput (DTorch guide, section 2): table Shard(1) on
 * tp (slot i holds [vocab, d_i] bf16 or fp32, d_i from the torch.chunk split
 * of the embedding dim), ids int32 Replicate on tp, out Replicate on tp with
 * shape ids.shape + [dim].  out[t, o_i:o_i+d_i] = table_i[ids[t], :]; an id
 * outside [0, vocab) zero-fills that row and sets DT_DEV_ERR_INDEX.
 * Other mesh dims must be Replicate for all three.  With no tokens (or an
 * empty embedding dim) the call returns DT_OK without launching; a table of
 * no rows with tokens to gather is refused with DT_ERR_SHAPE.
 */
DT_API dt_status dt_tp_embedding(const dt_dtensor* ids, const dt_dtensor* table, const dt_dtensor* out,
                          int32_t tp_mesh_dim, int32_t* d_status, dt_stream_t stream);

/* ---- linears (weights stored [in, out] as in the wineandchord reference) ----
 *
 * Every linear takes `workspace` / `workspace_bytes`: NULL (size ignored) or
 * caller-owned device memory, 256-byte aligned, of any size.  With at least
 * the bytes its *_workspace_size query reports, the call splits the tensor-
 * core GEMM's last wave where that pays (see the ownership convention
 * above); with less it runs every tile whole.  The queries take the call's
 * operands (host descriptors only, nothing is read from the device), check
 * them as the call would, and answer for the CURRENT device, whose number
 * of co-resident CTA pairs decides the split; without a CUDA device they
 * return DT_ERR_CUDA.
 * bf16 operands whose row pitch is not a multiple of 16 bytes, or whose base
 * is not 16-byte aligned (the shards of a dim that torch.chunk splits
 * unevenly, e.g. 8190 columns over 4), cannot be read by TMA.  With enough
 * workspace (the query counts it) the call copies each such operand into
 * the workspace with a padded pitch and runs on the tensor cores; with less
 * it runs on a CUDA-core kernel, an order of magnitude slower, and
 * dt_cuda_core_gemm_count() counts the launch.  fp32 linears always run on
 * the CUDA-core kernel and need no workspace (0 bytes).
 */

/*
 * ColumnParallelLinear: Y_i = X W_i (+ b_i) for every tp shard i, all shards
 * in one launch (wineandchord "Column parallel"; DTorch tp_shard_type "col").
 *   x    [..., K] Replicate on tp            (bf16 or fp32)
 *   w    [K, N]   Shard(1) on tp             (same dtype as x)
 *   bias [N]      Shard(0) on tp, or NULL    (bf16 or fp32)
 *   y    [..., N] Shard(-1) on tp            (bf16 or fp32; fp32 accumulate)
 * On other mesh dims w and bias must be Replicate and x, y must agree.
 * tp_mesh_dim < 0 means no TP (ReplicateParallelLinear).  Leading dims of x
 * and y are flattened and must be collapsible with unit inner stride.
 * bf16 operands run on the tcgen05 tensor-core GEMM (operands whose pitch
 * TMA cannot describe through a padded copy in the workspace, see above);
 * fp32 runs on a CUDA-core kernel.
 */
DT_API dt_status dt_column_parallel_linear(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias,
                                    const dt_dtensor* y, int32_t tp_mesh_dim, void* workspace,
                                    size_t workspace_bytes, int32_t* d_status, dt_stream_t stream);

/*
 * Several column-parallel linears that share one input (e.g. fused q/k/v),
 * in ONE launch: y[j] = column_parallel(x, w[j], bias[j]) for j < n.
 * w, y: arrays of n descriptors; bias: NULL or an array of n descriptors
 * whose entries may have nslots == 0 for "no bias".
 */
DT_API dt_status dt_column_parallel_linear_multi(const dt_dtensor* x, int32_t n, const dt_dtensor* w,
                                          const dt_dtensor* bias, const dt_dtensor* y,
                                          int32_t tp_mesh_dim, void* workspace, size_t workspace_bytes,
                                          int32_t* d_status, dt_stream_t stream);

/* Workspace bytes of dt_column_parallel_linear(_multi) on these operands
 * (n = 1 for the single form; the bias does not change it). */
DT_API dt_status dt_column_parallel_linear_workspace_size(const dt_dtensor* x, int32_t n, const dt_dtensor* w,
                                                          const dt_dtensor* y, int32_t tp_mesh_dim,
                                                          size_t* bytes);

/*
 * RowParallelLinear: Y = sum_i X_i W_i (+ b) (wineandchord "Row parallel";
 * DTorch tp_shard_type "row"; nanotron TensorParallelRowLinear).
 *   x    [..., K] Shard(-1) on tp
 *   w    [K, N]   Shard(0) on tp
 *   bias [N]      Replicate, or NULL; added ONCE (DTorch keeps the row bias
 *                 Partial so the shards' biases sum to one bias)
 *   y    mode DT_TP_ALL_REDUCE:     [..., N] Replicate on tp
 *        mode DT_TP_REDUCE_SCATTER: [..., N] Shard(0) on tp
 *        mode DT_TP_PARTIAL:        [..., N] Partial on tp (bias on part 0)
 * For ALL_REDUCE and REDUCE_SCATTER the sum over shards is fused into the
 * fp32 tensor-core accumulator: no partial product is written to memory.
 */
DT_API dt_status dt_row_parallel_linear(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias,
                                 const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim, void* workspace,
                                 size_t workspace_bytes, int32_t* d_status, dt_stream_t stream);

/* Workspace bytes of dt_row_parallel_linear on these operands. */
DT_API dt_status dt_row_parallel_linear_workspace_size(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* y,
                                                       int32_t mode, int32_t tp_mesh_dim, size_t* bytes);

/*
 * Llama-style TP MLP (nanotron 5.1: the MLP follows the attention's
 * column/row pattern):
 *   H_i = bf16( SiLU(X Wg_i) * (X Wu_i) )     gate/up column-parallel, one launch,
 *                                            two accumulators per tile, SiLU in fp32
 *   Y   = row_parallel(H, Wd, mode)           down projection
 * x [M, K] Replicate, w_gate/w_up [K, F] Shard(1), w_down [F, N] Shard(0),
 * y per `mode` as in dt_row_parallel_linear.  All bf16 (y bf16 or fp32).
 * workspace: caller-owned device memory, 256-byte aligned.  It receives H
 * at its start, as one [M, F] bf16 row-major tensor per distinct x slot
 * (shard i = the columns of chunk i; blocks 256-byte aligned), which the
 * call needs (DT_ERR_INVALID_ARG when the workspace is smaller); the bytes
 * after H are the two GEMMs' split-tail scratch, as for the linears.
 * dt_tp_mlp_workspace_size reports H plus that scratch for the current
 * device (DT_ERR_CUDA without one).
 */
DT_API dt_status dt_tp_mlp_workspace_size(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up,
                                          const dt_dtensor* w_down, const dt_dtensor* y, int32_t mode,
                                          int32_t tp_mesh_dim, size_t* bytes);
DT_API dt_status dt_tp_mlp(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up,
                    const dt_dtensor* w_down, const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim,
                    void* workspace, size_t workspace_bytes, int32_t* d_status, dt_stream_t stream);

/*
 * The TP MLP for callers that cannot allocate device memory at call time
 * (for example a serving loop that must not allocate once running, or host
 * code that does not own the device allocator).  Same operands, results and
 * errors as dt_tp_mlp, but H lives in a buffer built into the library: a
 * device array of DT_TP_MLP_STATIC_WORKSPACE_BYTES that every GPU which
 * loads the library holds until the process exits.  This entry point has no
 * counterpart in the pages; it exists for such callers only.
 *  - It allocates nothing (no cudaMalloc, no allocator of any library), and
 *    it runs every GEMM tile whole (it has no split-tail scratch).
 *  - Problems whose H (the [M, F] bf16 blocks described for dt_tp_mlp)
 *    exceeds the array are rejected with DT_ERR_CAPACITY.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress).  CUDA loads the library's device code
 *    lazily, so that first call is also when the device reserves the
 *    array, and it fails with DT_ERR_CUDA if the device has no room left.
 *    Make the first call on each device at start-up, before memory is
 *    committed elsewhere and before any stream capture.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    (different streams, or different host threads) race on H.  H is fully
 *    rewritten by every call, so nothing needs clearing in between.
 */
#define DT_TP_MLP_STATIC_WORKSPACE_BYTES (32 * 1024 * 1024)
DT_API dt_status dt_tp_mlp_static_workspace(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up,
                                            const dt_dtensor* w_down, const dt_dtensor* y, int32_t mode,
                                            int32_t tp_mesh_dim, int32_t* d_status, dt_stream_t stream);

/* ---- utilities ---- */

/* Static description of a status code. */
DT_API const char* dt_status_string(dt_status status);

/* Reason for the last non-OK status on this thread ("" if none). */
DT_API const char* dt_last_error(void);

/* Copy the library's own device status word (used when d_status == NULL)
 * to *bits and, if clear != 0, reset it.  Synchronous on the current device. */
DT_API dt_status dt_read_device_status(int32_t* bits, int32_t clear);

/* Drop the host-side caches (TMA descriptors, launch plans).  Not to be
 * called while another thread launches. */
DT_API dt_status dt_clear_cache(void);

/* Number of kernels this library has launched in this process so far
 * (every successful launch on any stream counts once). */
DT_API uint64_t dt_launch_count(void);

/* Of those, the launches of the CUDA-core GEMM: linears whose operands are
 * fp32 or whose bf16 pitches or bases TMA cannot describe (row pitch not a
 * multiple of 16 bytes, base not 16-byte aligned) run there, an order of
 * magnitude slower than the tensor cores. */
DT_API uint64_t dt_cuda_core_gemm_count(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
DT_API int32_t dt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DT_H_ */
