/*
 * cm.h -- C ABI of the decomposed collective matmul on one GB300 (sm_103a).
 *
 * Two operations, each over N logical ranks whose buffers all live in one
 * GPU's HBM:
 *
 *  AllGather -> GEMM (cm_ag_gemm).  Rank r holds the row shard X_r [m, K] of
 *  an activation that is gathered along rows, and its weight shard W_r
 *  [K, n]; it needs Y_r = concat_j(X_j) @ W_r [N*m, n].  The decomposition
 *  ("Overlap Communication with Dependent Computation via Decomposition in
 *  Large Deep Learning Models", section "The idea", AllGather -> Einsum;
 *  "Hiding Tensor-Parallel Collectives: AG/RS Overlap in Megatron",
 *  section 3) runs N steps: at step i rank r multiplies the shard it holds
 *  and writes the product into that shard's rows of Y_r (a
 *  DynamicUpdateSlice), while forwarding the shard to its ring neighbour.
 *
 *  GEMM -> ReduceScatter (cm_gemm_rs).  Rank r holds X_r [M, k] and W_r
 *  [k, n]; bucket o (rows o*M/N .. (o+1)*M/N - 1) of sum_r X_r @ W_r belongs
 *  to rank o.  The decomposition (same page, Einsum -> ReduceScatter; "Hiding
 *  Tensor-Parallel Collectives", section 5) circulates fp32 accumulating
 *  buckets: a rank adds its partial product to the bucket it received and
 *  forwards it; after N hops the bucket is home and is written out.
 *
 * Ring schedules (cm_plan):
 *  - CM_RING_UNI: one ring, rank r sends to r+1 (mod N), receives from r-1.
 *  - CM_RING_BIDI: the N-1 foreign shards / contributions are split between
 *    a clockwise stream of a = ceil((N-1)/2) hops and a counter-clockwise
 *    stream of b = floor((N-1)/2) hops (same page, bidirectional rings; the
 *    owner's "realigning addition" of section "What it costs" adds the two
 *    partial buckets and its own product).
 *  - CM_RING_NONE: the undecomposed operation ("Hiding Tensor-Parallel
 *    Collectives", sections 2 and 4): every shard is read in place and each
 *    output is one GEMM (for ReduceScatter, all ranks' products summed in
 *    one fp32 accumulator).  The monolithic comparator.
 *  - chunks: each shard (AG) or bucket (RS) moves and is signalled as
 *    `chunks` contiguous row blocks ("Hiding Tensor-Parallel Collectives",
 *    section 3, the chunk-size trade-off).  Results do not depend on it.
 *
 * Conventions shared by every call:
 *  - Ownership: the caller owns every device buffer (inputs, outputs,
 *    workspace).  The library owns only the host-side plan.  No call
 *    allocates device memory.
 *  - Asynchrony: compute calls enqueue work on `stream` and return; argument
 *    errors are returned synchronously; device-side errors (a bounded wait
 *    that timed out) are reported by cm_check_status.
 *  - Pointers are device pointers unless stated, 16-byte aligned.
 *  - bf16 inputs, fp32 accumulation (tensor memory), output bf16 (RNE) or fp32.
 *  - No C++ exception crosses this boundary.
 */
#ifndef CM_H_
#define CM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cm_status {
    CM_OK = 0,
    CM_ERR_INVALID_ARG = 1,   /* null / out-of-range argument */
    CM_ERR_SHAPE = 2,         /* shape not divisible as required */
    CM_ERR_ALIGNMENT = 3,     /* pointer or inner extent misaligned for TMA */
    CM_ERR_UNSUPPORTED = 4,   /* legal request this build does not run */
    CM_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    CM_ERR_TIMEOUT = 6,       /* a device-side bounded wait expired */
    CM_ERR_WORKSPACE = 7,     /* workspace null or smaller than required */
    CM_ERR_BOUNDS = 8         /* debug build: a computed index fell outside its buffer (access not made) */
} cm_status;

typedef enum cm_direction {
    CM_RING_UNI = 0,
    CM_RING_BIDI = 1,
    CM_RING_NONE = 2
} cm_direction;

typedef enum cm_dtype { CM_BF16 = 0, CM_F32 = 1 } cm_dtype;

/* Weight layout per rank: CM_W_KN = W_r stored [K][n] row-major;
 * CM_W_NK = W_r stored [n][K] (nn.Linear order, K contiguous). */
typedef enum cm_wlayout { CM_W_KN = 0, CM_W_NK = 1 } cm_wlayout;

typedef enum cm_op { CM_OP_AG_GEMM = 0, CM_OP_GEMM_RS = 1 } cm_op;

typedef struct cm_plan_s *cm_plan_t;
typedef struct CUstream_st *cm_stream_t;   /* identical to cudaStream_t */

/* Largest N a plan accepts, and largest chunk count. */
#define CM_MAX_RANKS 16
#define CM_MAX_CHUNKS 8

/*
 * cm_plan -- build the ring schedule for N logical ranks.  Host only; no
 * device work.  n_ranks in [1, CM_MAX_RANKS], chunks in [1, CM_MAX_CHUNKS].
 * On success *out owns a plan to be released with cm_plan_destroy.
 * Errors: CM_ERR_INVALID_ARG.
 */
cm_status cm_plan(int n_ranks, int chunks, cm_direction dir, cm_plan_t *out);

/* Release a plan (NULL is accepted). */
cm_status cm_plan_destroy(cm_plan_t plan);

/* Number of ring steps of `op` under this plan (N for the unidirectional
 * ring, ceil((N-1)/2)+1 for the bidirectional one, 1 for CM_RING_NONE). */
int cm_plan_steps(cm_plan_t plan, cm_op op);

/*
 * cm_plan_step -- the schedule entry of `rank` at `step` on ring stream
 * `stream` (0 = clockwise, r -> r+1; 1 = counter-clockwise, r -> r-1).
 *  *obj: shard (AG) or bucket (RS) id the rank multiplies for, -1 if idle.
 *  *src: rank the shard / partial bucket came from (AG: the rank itself at
 *        step 0; RS: -1 when the rank starts the bucket).
 *  *dst: rank it is forwarded to after this step, -1 if it goes no further
 *        (RS: -1 means the bucket is home and written to the output).
 * At step 0 of a bidirectional AG plan the own shard is listed on both
 * streams (it is sent both ways) and multiplied once.  In a bidirectional RS
 * plan the owner's entry at the last step lists the clockwise source; the
 * owner also adds the partial bucket that came counter-clockwise.  A
 * CM_RING_NONE plan has no ring: its single step lists obj = src = dst = -1.
 * Host only.
 * Errors: CM_ERR_INVALID_ARG for an out-of-range rank/step/stream.
 */
cm_status cm_plan_step(cm_plan_t plan, cm_op op, int rank, int step, int stream,
                       int *obj, int *src, int *dst);

/*
 * One entry of the task table the persistent kernel executes, in execution
 * order.  A task is one partial GEMM of one rank at one step; flag ids name
 * per-chunk device counters (word = id * chunks + chunk).  Order: for a
 * one-way ring, rank-blocked -- rank 0's step 0, rank 1's steps 0..1, ...,
 * rank N-1's steps 0..N-1, then rank 0's steps 1..N-1, rank 1's steps
 * 2..N-1, ... -- so each rank's weight shard is streamed in two runs; for a
 * bidirectional ring, stream-blocked (each stream's tasks in that order, the
 * counter-clockwise one over mirrored ranks; see CM_OPT_TASK_ORDER); for
 * CM_RING_NONE and the step-serial mode, step-major and by rank inside a
 * step (CM_OPT_TASK_ORDER runs a ring step-major too).  Every flag a task
 * waits on is raised by an earlier
 * task.  Exposed so tests can check the table's dependency structure on the
 * host.
 */
typedef struct cm_task {
    int16_t rank;          /* r: selects W_r (and Y_r for AG) */
    int16_t a_slab;        /* AG: shard slab in x / slot slab in workspace; RS: r*N + bucket */
    int16_t a_src;         /* 0 = one slab of x read in place, 1 = a workspace slot,
                              2 = every rank's slab summed in one accumulator (RS, no ring) */
    int16_t out_idx;       /* AG: shard id s (rows s*m of Y_r); RS: bucket id o */
    int16_t out_buf;       /* RS: accumulator buffer written, -1 = final output y[o] */
    int16_t in_buf[2];     /* RS: accumulator buffers read (-1 none) */
    int16_t fwd_slot[2];   /* AG: workspace slots the shard is forwarded into (-1 none) */
    int16_t wait_in[2];    /* flags that must reach their target before reading inputs */
    int16_t wait_free[2];  /* flags that must reach their target before overwriting a slot/buffer */
    int16_t sig_fwd[2];    /* AG: flags bumped once per forwarded row tile */
    int16_t sig_done;      /* AG: bumped per tile once its slot reads landed; RS: per finished tile */
    int16_t step;          /* ring step of this task */
    int16_t stream;        /* 0 clockwise (or own / owner), 1 counter-clockwise */
    int16_t tile_group;    /* (size << 8) | position: the tiles of a group of
                              consecutive same-rank tasks are interleaved
                              (column tile outermost) so they share W_r in L2 */
} cm_task;

/* Copy the task table of `op` into out[0..capacity); returns the number of
 * tasks (which may exceed capacity), or -1 for a bad plan/op.  Host only.
 * For CM_OP_GEMM_RS it lists the per-step-buffer table when
 * CM_OPT_RS_IN_PLACE is 0 and the in-place one otherwise (a call chooses
 * between the two by its shape when the option is 2). */
int cm_plan_tasks(cm_plan_t plan, cm_op op, cm_task *out, int capacity);

/*
 * Workspace bytes for one call; 0 for a bad plan or a non-positive size.
 * Holds a 256-byte status block (status word, tile counters), the per-chunk
 * flags and, for a ring with N > 1: for AG, one receive slot per (rank, ring
 * stream, step), each [m][K] bf16, written once per call, so no task waits
 * for one to be freed; for RS, one fp32 accumulator [M/N][n] per (bucket,
 * ring stream) when the buckets are kept in place, or per (rank, ring
 * stream, step) otherwise (CM_OPT_RS_IN_PLACE).  The caller allocates it (256-byte
 * aligned) and owns it; its contents need no initialisation (each call clears
 * the status block and flags with one memset on its stream).  Calls that
 * share a workspace must be ordered on the GPU (one stream).
 */
size_t cm_ag_gemm_workspace_size(cm_plan_t plan, int64_t m, int64_t K);
size_t cm_gemm_rs_workspace_size(cm_plan_t plan, int64_t M, int64_t n);

/*
 * cm_ag_gemm -- decomposed AllGather -> GEMM.
 *  x  [N][m][K] bf16: shard X_j at x + j*m*K (the gathered X is x itself).
 *  w  N weight shards, bf16: W_r at w + r*K*n, laid out per `wlayout`.
 *  y  [N][N*m][n] (y_dtype): Y_r at y + r*N*m*n; rows j*m..j*m+m-1 hold X_j @ W_r.
 *  ws, ws_bytes: workspace of at least cm_ag_gemm_workspace_size(plan, m, K)
 *  bytes.  Outputs must not alias inputs or the workspace; inputs are not
 *  modified.  Enqueued on `stream`; returns before the GPU work runs.
 *  Errors (synchronous, nothing enqueued): CM_ERR_INVALID_ARG for a null
 *  plan/pointer or a bad enum; CM_ERR_SHAPE if m, K or n is not positive,
 *  exceeds 2^30, or m % chunks != 0; CM_ERR_ALIGNMENT if K or n is not a
 *  multiple of 8 or a pointer is not 16-byte aligned; CM_ERR_WORKSPACE if
 *  ws_bytes is too small; CM_ERR_UNSUPPORTED if the device cannot run the
 *  kernel; CM_ERR_CUDA if a launch or tensor-map encoding fails.  Device-side
 *  failures (a bounded wait that timed out) come from cm_check_status.
 */
cm_status cm_ag_gemm(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout,
                     void *y, cm_dtype y_dtype, int64_t m, int64_t K, int64_t n,
                     void *ws, size_t ws_bytes, cm_stream_t stream);

/*
 * cm_gemm_rs -- decomposed GEMM -> ReduceScatter.
 *  x  [N][M][k] bf16: X_r at x + r*M*k.
 *  w  N weight shards, bf16: W_r at w + r*k*n, laid out per `wlayout`.
 *  y  [N][M/N][n] (y_dtype): bucket o = rows o*M/N.. of sum_r X_r @ W_r.
 *  ws, ws_bytes: workspace of at least cm_gemm_rs_workspace_size(plan, M, n)
 *  bytes.  Accumulation across ranks is fp32, in ring order; the home rank
 *  rounds once to y_dtype.  On one GPU a bucket is not copied from rank to
 *  rank: it stays in one workspace buffer per ring stream, and passing it
 *  on is releasing its readiness flag to the next contributor, which adds
 *  its product into it there -- or, with per-step buffers, the next
 *  contributor reads it and writes the sum to a buffer of its own
 *  (CM_OPT_RS_IN_PLACE chooses).  Outputs
 *  must not alias inputs or the workspace.
 *  Errors: as cm_ag_gemm, with CM_ERR_SHAPE also for M % N != 0 or
 *  (M/N) % chunks != 0, and k in the role of K.
 */
cm_status cm_gemm_rs(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout,
                     void *y, cm_dtype y_dtype, int64_t M, int64_t k, int64_t n,
                     void *ws, size_t ws_bytes, cm_stream_t stream);

/*
 * cm_gemm_rs_pipelined -- GEMM -> ReduceScatter with pipeline chunks instead
 * of a moving bucket ("Hiding Tensor-Parallel Collectives: AG/RS Overlap in
 * Megatron", section 6): every rank computes its full fp32 partial product
 * X_r @ W_r, chunk by chunk, and the reduction of chunk j (owner o's rows of
 * that chunk = the sum over ranks r = 0..N-1 of their partials, rounded once
 * to y_dtype) runs on a second, library-owned stream while the GEMM computes
 * chunk j + 1.  A chunk is a contiguous row block of every bucket, M/N/chunks
 * rows (the plan's chunk count; its direction is not used).
 *  Arguments, layouts and result: those of cm_gemm_rs (same output).
 *  Workspace: cm_gemm_rs_pipelined_workspace_size(plan, M, n) bytes (the
 *  partial products, N * M * n fp32, plus a status block), 256-byte aligned.
 *  Stream: asynchronous on `stream`; the library's second stream waits on an
 *  event after each chunk's GEMM and `stream` waits for the last reduction,
 *  so work queued on `stream` afterwards sees the output.  Calls on one
 *  device are serialised on the host (the second stream is shared).
 *  Errors: as cm_gemm_rs.
 */
size_t cm_gemm_rs_pipelined_workspace_size(cm_plan_t plan, int64_t M, int64_t n);
cm_status cm_gemm_rs_pipelined(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout,
                               void *y, cm_dtype y_dtype, int64_t M, int64_t k, int64_t n,
                               void *ws, size_t ws_bytes, cm_stream_t stream);

/*
 * cm_backward_pair -- the backward pass of the column-parallel layer whose
 * forward is cm_ag_gemm (Y_r = concat_j(X_j) @ W_r^T, W_r stored [n][K]):
 *   data gradient   dX_o = rows [o*m, (o+1)*m) of sum_r dY_r @ W_r
 *                   -- a GEMM -> ReduceScatter, run as the decomposed ring
 *                   of cm_gemm_rs with W_r read as [k = n][K];
 *   weight gradient dW_r = dY_r^T @ concat_j(X_j)
 *                   -- it needs every rank's gathered input, an AllGather the
 *                   data gradient does not need, so it runs on a second,
 *                   library-owned stream under the GEMM-RS ("bulk overlap").
 * ("Tensor Parallelism > Communication Patterns": the backward pass is the
 * forward's dual; "Hiding Tensor-Parallel Collectives: AG/RS Overlap in
 * Megatron", section 7.)
 *  x   [N][m][K] bf16: the forward input shards (read by the AllGather)
 *  w   [N][n][K] bf16: the forward weights
 *  dy  [N][N*m][n] bf16: each rank's output gradient
 *  dx  [N][m][K]: the sequence-sharded input gradient (dx_dtype)
 *  dw  [N][n][K]: the weight gradients (dw_dtype)
 *  Buffers: the caller must not write x or dy until `stream` has passed
 *  this call (the second stream reads x; `stream` waits for it before the
 *  weight-gradient GEMM).  The gathered inputs live in the workspace,
 *  cm_backward_pair_workspace_size(plan, m, K, n) bytes, 256-byte aligned.
 *  Shapes: n, K and N*m at least 64; K and n multiples of 8; m divisible
 *  by the plan's chunks.  Errors as cm_gemm_rs.
 */
size_t cm_backward_pair_workspace_size(cm_plan_t plan, int64_t m, int64_t K, int64_t n);
cm_status cm_backward_pair(cm_plan_t plan, const void *x, const void *w, const void *dy,
                           void *dx, cm_dtype dx_dtype, void *dw, cm_dtype dw_dtype,
                           int64_t m, int64_t K, int64_t n, void *ws, size_t ws_bytes,
                           cm_stream_t stream);

/*
 * cm_cannon_gemm -- Cannon-style 2-D rotation on a q x q grid of logical
 * ranks (q * q = the plan's rank count: 1, 4, 9 or 16), the contracting-
 * dimension-sharded special case of the decomposition ("Overlap
 * Communication with Dependent Computation via Decomposition in Large Deep
 * Learning Models", section "What people did before": shard rotation
 * interleaved with partial products).  C = A @ B with every operand in
 * q x q blocks:
 *   a  [q*q][bm][bk] bf16, block A_{i,k} at index i*q + k
 *   b  [q*q] blocks of B, B_{k,j} at index k*q + j, each [bn][bk]
 *      (CM_W_NK) or [bk][bn] (CM_W_KN)
 *   c  [q*q][bm][bn] (c_dtype), block C_{i,j} at index i*q + j
 * Rank (i, j) starts from A_{i,(i+j) mod q} and B_{(i+j) mod q, j} (the
 * skew, read in place), then for q steps multiplies what it holds into an
 * fp32 accumulator while the next blocks rotate in -- A from the right
 * neighbour (i, j+1), B from below (i+1, j) -- by copies on a second,
 * library-owned stream under the step's GEMM.  One kernel launch per step.
 *  Workspace: cm_cannon_workspace_size(plan, bm, bk, bn) bytes, 256-byte
 *  aligned (accumulators and two sets of rotated blocks).
 *  Errors: CM_ERR_SHAPE if the rank count is not a square; otherwise as
 *  cm_gemm_rs (bk and bn multiples of 8).
 */
size_t cm_cannon_workspace_size(cm_plan_t plan, int64_t bm, int64_t bk, int64_t bn);
cm_status cm_cannon_gemm(cm_plan_t plan, const void *a, const void *b, cm_wlayout b_layout,
                         void *c, cm_dtype c_dtype, int64_t bm, int64_t bk, int64_t bn,
                         void *ws, size_t ws_bytes, cm_stream_t stream);

/*
 * cm_check_status -- synchronise `stream` and read the device status word of
 * the last call that used `ws`.  Returns CM_OK, CM_ERR_TIMEOUT (a bounded
 * wait expired; the outputs of that call are undefined), CM_ERR_BOUNDS (a
 * library built with bounds checks -- CM_DEBUG_BOUNDS -- found a computed
 * flag, slot, row or buffer index outside its buffer and skipped that
 * access; the outputs are undefined) or CM_ERR_CUDA.  If info is non-NULL it
 * receives {code, task, chunk, site} of the first failure.
 */
cm_status cm_check_status(const void *ws, cm_stream_t stream, int32_t info[4]);

/* Static English text for a status code. */
const char *cm_status_string(cm_status status);

/*
 * Plan options (host only):
 *  CM_OPT_TIMEOUT_NS     bound of every device-side wait, in ns (default 1e9).
 *  CM_OPT_SERIAL_STEPS   1: launch one kernel per ring step (step barriers
 *                        instead of flags between steps); a debugging mode.
 *  CM_OPT_GRID           persistent grid size, 0 = one CTA per SM.
 *  CM_OPT_SKIP_SIGNAL    fault injection: value = (op << 16) | (rank << 8) | step;
 *                        that task never signals its forward/done flags, so
 *                        its consumers time out.  -1 clears it.
 *  CM_OPT_KERNEL         tile kernel.  0 (default) and 2: 256 x 256 tiles on
 *                        CTA pairs (tcgen05 cta_group::2), one pair per
 *                        cluster; 1: 128 x 256 tiles on single CTAs.  Other
 *                        values: CM_ERR_INVALID_ARG.
 *  CM_OPT_STATIC_TILES   CTA-pair kernel: 0 (default) hands tiles out in
 *                        order from a global counter as clusters free up;
 *                        1 gives cluster c the tiles c, c + clusters, ...
 *  CM_OPT_TILE_GROUP     largest number of consecutive same-rank tasks whose
 *                        tiles are interleaved (1..8, default 4).
 *  CM_OPT_L2_HINTS       CTA-pair kernel, L2 eviction priority of operand
 *                        loads: bits 0-3 for A, 4-7 for B; 0 normal,
 *                        1 evict_last, 2 evict_first (default 0).
 *  CM_OPT_L2_PROMOTION   TMA L2 promotion of operand loads: 0 none, 1 64 B,
 *                        2 128 B, 3 256 B (default 3).
 *  CM_OPT_ROW_BAND       tile order: row tiles per band (1..4096), or 0 (the
 *                        default) for as many row tiles as hold about 32 MB
 *                        of the A operand.  Each band of a task group's row
 *                        tiles runs through every column tile before the
 *                        next band starts; 4096 puts a whole group in one
 *                        band.
 *  CM_OPT_BULK_OVERLAP   cm_backward_pair: 1 (default) runs the weight
 *                        gradient's AllGather on a second stream under the
 *                        data-gradient GEMM-RS; 0 runs it first on `stream`.
 *  CM_OPT_RS_PRELOAD     cm_gemm_rs on the CTA-pair kernel (one pair per
 *                        cluster): 1 brings a tile's received partial bucket
 *                        in through the operand ring and copies it into the
 *                        tile's tensor-memory accumulator before the partial
 *                        GEMM adds onto it, so the epilogue only stores;
 *                        0 adds the received bucket in the epilogue; 3
 *                        preloads half of it (the first two of each
 *                        epilogue warp's four 32-column slices) and adds the
 *                        rest in the epilogue; 2 (the default) preloads all
 *                        of it when a tile has at most 8 K slices of 64
 *                        (k <= 512), where the epilogue sets the pace, and
 *                        none beyond (the epilogue then hides under the
 *                        partial GEMM).  The same sum, in a different fp32
 *                        order.  With buckets kept in place (below) only
 *                        the owner's tiles read a bucket, so only they are
 *                        preloaded.
 *  CM_OPT_RS_IN_PLACE    cm_gemm_rs (and the backward pair's data gradient)
 *                        on a ring: 1 keeps each bucket in one fp32 buffer
 *                        per ring stream that the first contributor writes
 *                        and every later one adds its partial product into
 *                        where it lies (a reduce-add at L2), in ring order,
 *                        each after its predecessor's flag; 0 gives every
 *                        (rank, stream, step) its own buffer, written once by
 *                        the previous rank and read by the next; 2 (default)
 *                        chooses per call: in place when one stream's buckets
 *                        (M*n*4 bytes) take at most 128 MB and stay in L2,
 *                        per-step buffers otherwise.  The same fp32 sums in
 *                        the same order.  The workspace size follows the
 *                        choice (N buffers per stream in place, N per stream
 *                        and step otherwise), so size the workspace after
 *                        setting it, for the call's M and n.
 *  CM_OPT_TASK_ORDER     order of a one-way ring's tasks: 1 rank-blocked
 *                        (see cm_task: each weight shard streamed in two
 *                        runs), 2 step-major (every rank's step 0, then every
 *                        rank's step 1, ...: a task is as far as possible from
 *                        the ones it waits for), 0 (default) step-major when
 *                        the weight shards of all ranks together take at most
 *                        48 MB -- they stay in L2 either way -- and
 *                        rank-blocked otherwise.  cm_plan_tasks lists the
 *                        step-major table under 2 and the ring's own order
 *                        under 0 and 1.  A bidirectional ring's own order
 *                        is stream-blocked: the clockwise stream's tasks
 *                        rank-blocked, then the counter-clockwise stream's
 *                        rank-blocked over the mirrored ranks, each owner
 *                        after the tasks it waits for.  The same results.
 *  CM_OPT_RS_EPILOGUE    how the CTA-pair kernel moves GEMM -> ReduceScatter
 *                        tiles out of tensor memory: 1 every epilogue warp
 *                        on every tile, the bucket slices copied by TMA
 *                        through shared memory (reduce-add, store or load);
 *                        2 two groups of epilogue warps, one per tensor-memory
 *                        accumulator, so that two tiles drain at once, with
 *                        coalesced vector adds (red.global.add.v4.f32),
 *                        stores and loads; 3 every epilogue warp on every
 *                        tile (as 1) with the vector accesses of 2, so that a
 *                        tile drains in half the time of a group's and the
 *                        TMA unit carries only operand loads; 0 (default) two groups for rings
 *                        of 8 ranks (one-way) or 16 (either) whose tiles
 *                        have at least 28 K slices of 64 and read nothing
 *                        back (buckets in place, pipelined partials), the
 *                        TMA path otherwise -- per-step buffers and Cannon's
 *                        chained accumulator included (the faster of the two
 *                        in measurement).
 *                        The same fp32 additions in the same order: the same
 *                        bits.
 *  CM_OPT_RS_COL_SLABS   cm_gemm_rs: the tile order in `value` passes over
 *                        the tasks, each over one slab of the column tiles
 *                        (the largest count not above `value` that divides
 *                        them), so that a pass touches 1/value of every
 *                        bucket; 1: one pass; 0 (default): two for a one-way
 *                        ring whose buckets take at most 128 MB and whose
 *                        tiles have at least 16 K slices, else one.  Values
 *                        0..64.
 *                        The same fp32 additions in the same order: the same
 *                        bits.
 *  CM_OPT_RS_BUCKET_HINT cm_gemm_rs on the CTA-pair kernel with the TMA
 *                        epilogue: L2 eviction priority of the bucket writes
 *                        and adds -- 1
 *                        evict_first, 2 evict_last, 3 none; 0 (default)
 *                        evict_last when one ring stream's buckets (M*n*4
 *                        bytes) take at most 128 MB and can stay in L2,
 *                        none otherwise.  Only cache behaviour changes: the
 *                        same bits.
 *  CM_OPT_DEBUG_FLAG_OFFSET  only in a library built with bounds checks
 *                        (CM_DEBUG_BOUNDS; other builds return
 *                        CM_ERR_INVALID_ARG): adds `value` (>= 0) to the flag
 *                        id of every GEMM -> ReduceScatter task's done signal,
 *                        a planted mistake that puts those signals beyond the
 *                        flag words, so that tests can see the checks turn it
 *                        into CM_ERR_BOUNDS.  0 clears it.
 */
typedef enum cm_option {
    CM_OPT_TIMEOUT_NS = 0,
    CM_OPT_SERIAL_STEPS = 1,
    CM_OPT_GRID = 2,
    CM_OPT_SKIP_SIGNAL = 3,
    CM_OPT_KERNEL = 4,
    CM_OPT_STATIC_TILES = 5,
    CM_OPT_TILE_GROUP = 6,
    CM_OPT_L2_HINTS = 7,
    CM_OPT_L2_PROMOTION = 8,
    CM_OPT_ROW_BAND = 9,
    CM_OPT_BULK_OVERLAP = 10,
    CM_OPT_RS_PRELOAD = 11,
    CM_OPT_RS_IN_PLACE = 12,
    CM_OPT_TASK_ORDER = 13,
    CM_OPT_RS_EPILOGUE = 14,
    CM_OPT_DEBUG_FLAG_OFFSET = 15,
    CM_OPT_RS_COL_SLABS = 16,
    CM_OPT_RS_BUCKET_HINT = 17
} cm_option;

cm_status cm_plan_set_option(cm_plan_t plan, cm_option option, int64_t value);

/*
 * Cost model ("Overlap Communication with Dependent Computation via
 * Decomposition in Large Deep Learning Models", section "The idea", knowing
 * when to decline, and section "What it costs").  A peak-rate estimate of
 * one rank's time for the decomposed ring and for the native collective
 * followed by the undecomposed GEMM, from rates the caller measured.  Host
 * only; no device work.
 *
 * cm_rates (all per rank, all > 0 except hop_us >= 0):
 *   gemm_tflops  dense bf16 GEMM rate of one rank (TFLOP/s)
 *   ring_gbs     one ring link in one direction (GB/s)
 *   coll_gbs     algorithm bandwidth of the native AllGather / ReduceScatter
 *                (GB/s); the ring drives fewer links, so usually ring_gbs
 *                is below it
 *   hop_us       fixed cost of one message (one chunk over one hop: the flag
 *                round trip), in us; it holds the link
 *   mem_gbs      local memory bandwidth, for the bidirectional ring's
 *                realigning addition (GB/s)
 *
 * cm_cost_estimate -- predicted time in us of one candidate: n_ranks,
 *   chunks (1..CM_MAX_CHUNKS) and direction (CM_RING_NONE = native
 *   collective, then GEMM).  Shapes as the compute calls: AG rows = m (one
 *   shard), K, n; RS rows = M (divisible by n_ranks), K = k, n.
 *   Errors: CM_ERR_INVALID_ARG for a bad argument or rate, CM_ERR_SHAPE if
 *   M is not divisible by n_ranks (RS).
 * cm_plan_choose -- the fastest of: native, and one-way and bidirectional
 *   rings with 1, 2, 4 ... max_chunks chunks that split the shard (AG) or
 *   bucket (RS) evenly.  *dir = CM_RING_NONE means "decline: keep the
 *   native collective".  Ties keep the simpler choice.  *us (optional)
 *   receives the predicted time.
 */
typedef struct cm_rates {
    double gemm_tflops;
    double ring_gbs;
    double coll_gbs;
    double hop_us;
    double mem_gbs;
} cm_rates;

cm_status cm_cost_estimate(int n_ranks, int chunks, cm_direction dir, cm_op op, int64_t rows, int64_t K,
                           int64_t n, const cm_rates *rates, double *us);
cm_status cm_plan_choose(int n_ranks, cm_op op, int64_t rows, int64_t K, int64_t n, const cm_rates *rates,
                         int max_chunks, int *chunks, cm_direction *dir, double *us);

/*
 * One Einsum that offers both collectives (same page, section "The idea":
 * where an Einsum has both a gathered input and a scattered output, the
 * cost model also decides which of the two to overlap).  Per rank: the A
 * operand is the AllGather of N row
 * shards [m, K]; the rank multiplies the gathered [N*m, K] by its [K, n]
 * weight; the [N*m, n] fp32 result is summed over the ranks and scattered
 * (bucket o = rows o*m .. o*m + m - 1).  Only one collective can become the
 * ring; the other stays native.
 *
 * cm_einsum_cost -- predicted time in us of one candidate:
 *   decompose = CM_OP_AG_GEMM: the AllGather ring (chunks, dir), then the
 *     native ReduceScatter;
 *   decompose = CM_OP_GEMM_RS: the native AllGather, then the ReduceScatter
 *     ring;
 *   decompose = -1 (or dir CM_RING_NONE, or n_ranks 1): both native around
 *     the GEMM.
 *   Errors: CM_ERR_INVALID_ARG for a bad argument or rate.
 * cm_plan_choose_einsum -- the fastest of: both native, and each collective
 *   decomposed with one-way and bidirectional rings of 1, 2, 4 ...
 *   max_chunks chunks that split m evenly.  *decompose receives
 *   CM_OP_AG_GEMM, CM_OP_GEMM_RS or -1 (decline: both native); *chunks and
 *   *dir the ring; *us (optional) the predicted time.  Ties keep the simpler
 *   choice (native, then the gather, one-way, fewer chunks).
 */
cm_status cm_einsum_cost(int n_ranks, int chunks, cm_direction dir, int decompose, int64_t m, int64_t K, int64_t n,
                         const cm_rates *rates, double *us);
cm_status cm_plan_choose_einsum(int n_ranks, int64_t m, int64_t K, int64_t n, const cm_rates *rates, int max_chunks,
                                int *decompose, int *chunks, cm_direction *dir, double *us);

/* Library version string. */
const char *cm_version(void);

/*
 * cm_ag_gemm_noalloc -- cm_ag_gemm without a workspace argument, for callers
 * that cannot allocate device memory (for example a plugin that is handed
 * only its input and output buffers by a framework owning all device memory,
 * or a loop that must not call cudaMalloc).  The pages have no counterpart:
 * this is a packaging of the same operation.
 *  Scratch: one device array of CM_NOALLOC_SCRATCH_BYTES defined in the
 *  library and held by every GPU that loads it until the process exits.
 *  Arguments, layouts and results are those of cm_ag_gemm.
 *  Errors: CM_ERR_WORKSPACE if the call needs more scratch than the array
 *  holds (checked before any device work); otherwise as cm_ag_gemm.
 *  The first call on a device looks up the array's address with that device
 *  current; make it outside any stream capture.  Every call shares the array:
 *  its status word, flags and counters are cleared on `stream` at the start
 *  of each call, and calls that may overlap on the GPU race on it.  Argument
 *  and launch errors are returned; a device-side wait that expires (which
 *  leaves the outputs undefined) is recorded in the array's status word, which
 *  cm_ag_gemm_noalloc_check_status reads.  Never allocates.
 */
#define CM_NOALLOC_SCRATCH_BYTES (64u << 20)
cm_status cm_ag_gemm_noalloc(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout, void *y,
                             cm_dtype y_dtype, int64_t m, int64_t K, int64_t n, cm_stream_t stream);

/*
 * cm_ag_gemm_noalloc_check_status -- cm_check_status for the allocation-free
 * entry point: synchronise `stream` and read the status word of the last
 * cm_ag_gemm_noalloc call on the current device (the library's scratch array
 * is that call's workspace).  Returns CM_OK, CM_ERR_TIMEOUT (a bounded wait
 * expired; that call's outputs are undefined) or CM_ERR_CUDA; info as for
 * cm_check_status.  Call it with the same device current as the call it
 * checks.  Never allocates.  No counterpart on the pages: like the entry
 * point it checks, it only repackages the library for callers that cannot
 * allocate.
 */
cm_status cm_ag_gemm_noalloc_check_status(cm_stream_t stream, int32_t info[4]);

#ifdef __cplusplus
}
#endif

#endif /* CM_H_ */
