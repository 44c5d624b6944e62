/*
 * tbe.h -- C ABI of libtbe: table-batched embedding bags (TBE) on one GB300.
 *
 * The operator is the one described on the page "FBTriton table-batched
 * embeddings: the backward win is a threshold moved from 32 to 256":
 *
 *  - Layout ([FBT] "A lookup table that is most of the model"): every table
 *    sits in one weight buffer; every feature's bags share one flat
 *    `indices` array and one `offsets` array laid out feature-major, so bag
 *    (t, b) is indices[offsets[t*B + b] : offsets[t*B + b + 1]].  The output
 *    is one [B, sum_t D_t] matrix with feature t at column D_offsets[t].  An
 *    empty bag leaves its slot zero; a repeated id is added twice.
 *  - Forward ([FBT] "The forward: a general gather and one clever special
 *    case"): sum pooling of the rows a bag names, optionally scaled by
 *    per-sample weights, accumulated in FP32; a small-table path counts ids
 *    per bag and multiplies the count matrix by the table on tensor cores.
 *  - Backward ([FBT] "Why the backward is the hard half" and "Three tiers,
 *    routed by run length"): every lookup gets the key
 *    table_row_base[t] + id, the keys are sorted, equal keys form runs, and
 *    each run's row gradient is the sum of the output-gradient slices of the
 *    bags that read it (times their per-sample weights).  Short runs are
 *    reduced by one warp each; long runs are cut into chunks whose partial
 *    sums are combined by the last chunk to finish (fence + counter).
 *  - Exact optimizer ([FBT] "Why the backward is the hard half"): SGD or
 *    row-wise Adagrad applied once per distinct row to its finished
 *    gradient, in place on the tables (tbe_exact_update).
 *
 * Conventions for every entry point
 *  - Pointers named dev_* or documented "device" are CUDA device pointers;
 *    all others are host pointers.  The caller owns every buffer.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work on it: they never synchronise and
 *    never allocate device memory.
 *  - Return value: TBE_OK or a TBE_ERR_* code for errors found on the host
 *    (bad arguments, unsupported shapes, CUDA launch failures).  Errors that
 *    depend on the data (ids outside their table, broken offsets, a
 *    workspace-capacity shortfall, a bounded wait that gave up) are OR-ed
 *    into the optional device word `dev_status` as TBE_DEV_* bits; kernels
 *    never trap.  A lookup whose id is outside [0, rows_t) contributes
 *    nothing, forward or backward.
 *  - Sizes: N (lookups) < 2^30, T*B < 2^31, sum of table rows < 2^32 - 1,
 *    rows of one table < 2^31, T <= TBE_MAX_TABLES.  Every table's row must
 *    be a multiple of 16 bytes and every table must start on a 16-byte
 *    boundary of `weights`.
 */
#ifndef TBE_H_
#define TBE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes (host) ------------------------------------------------ */
#define TBE_OK 0
#define TBE_ERR_INVALID_ARG 1 /* null pointer, negative size, inconsistent layout */
#define TBE_ERR_UNSUPPORTED 2 /* a shape or dtype outside the stated limits      */
#define TBE_ERR_CUDA 3        /* a CUDA runtime call or kernel launch failed      */
#define TBE_ERR_WORKSPACE 4   /* workspace smaller than the size query returned   */

/* ---- device status bits (OR-ed into *dev_status by kernels) --------------- */
#define TBE_DEV_BAD_INDEX 0x1   /* an id outside [0, rows_t); it was skipped          */
#define TBE_DEV_BAD_OFFSETS 0x2 /* offsets[0] != 0, decreasing, or offsets[T*B] != N */
#define TBE_DEV_TIMEOUT 0x4     /* a bounded wait gave up; outputs are not valid      */
#define TBE_DEV_CAPACITY 0x8    /* row_grads_capacity too small; outputs truncated    */

/* ---- element types ------------------------------------------------------- */
#define TBE_F32 0
#define TBE_F16 1
#define TBE_BF16 2

#define TBE_MAX_TABLES 4096

/* ---- forward path selection ---------------------------------------------- */
#define TBE_PATH_AUTO 0      /* histogram path where eligible, else gather */
#define TBE_PATH_GATHER 1    /* always the gather kernel                   */
#define TBE_PATH_HISTOGRAM 2 /* histogram path; TBE_ERR_UNSUPPORTED if not eligible */

/* ---- pooling ------------------------------------------------------------- */
#define TBE_POOL_SUM 0  /* a bag's output is the (weighted) sum of its rows     */
#define TBE_POOL_MEAN 1 /* ... divided by the bag's number of lookups (empty: 0) */

/*
 * Description of the packed tables (all HOST arrays; copied by
 * tbe_plan_create, so they may be freed afterwards).
 *   T                : number of tables (features), 1..TBE_MAX_TABLES
 *   table_row_base   : [T+1] running sum of table row counts (the page's
 *                      hash_size_cumsum); rows_t = diff; global row of id in
 *                      table t is table_row_base[t] + id
 *   D_offsets        : [T+1] running sum of table widths; D_t = diff; also
 *                      the output column offset of feature t
 *   weights_offsets  : [T] byte offset of table t inside `weights`
 *                      (row-major [rows_t, D_t] in its dtype)
 *   weights_dtype    : [T] TBE_F32 / TBE_F16 / TBE_BF16
 *   table_weighted   : [T] 1 if table t uses per_sample_weights; NULL means
 *                      every table does when per_sample_weights is given
 *   out_dtype        : forward output element type
 *   pooling          : TBE_POOL_SUM or TBE_POOL_MEAN.  Mean pooling divides
 *                      each bag's fp32 sum by its number of lookups L (one
 *                      IEEE division; an empty bag stays 0); its backward
 *                      gives each lookup (w_i / L) * grad_out[b]
 */
typedef struct tbe_layout {
  int32_t T;
  const int64_t* table_row_base;
  const int32_t* D_offsets;
  const int64_t* weights_offsets;
  const int32_t* weights_dtype;
  const uint8_t* table_weighted;
  int32_t out_dtype;
  int32_t pooling;
} tbe_layout;

/* Opaque plan: validated layout, packed per-table metadata and kernel
 * choices.  The packed metadata lives in caller-provided device memory. */
typedef struct tbe_plan tbe_plan;

/* Bytes of device memory a plan for T tables needs (256-byte multiple). */
size_t tbe_plan_device_bytes(int32_t T);

/* Validate `L`, pack its per-table metadata and copy it (asynchronously, on
 * `stream`) into `dev_meta` (device, >= tbe_plan_device_bytes(T) bytes,
 * 16-byte aligned, owned by the caller and kept alive while the plan is in
 * use).  The host-side plan object is returned in *plan_out (heap memory of
 * the host; release with tbe_plan_destroy).
 * Errors: TBE_ERR_INVALID_ARG (nulls, T out of range, decreasing
 * table_row_base or D_offsets, unknown dtype), TBE_ERR_UNSUPPORTED (a row
 * that is not a multiple of 16 bytes, an unaligned table, row counts beyond
 * the limits), TBE_ERR_CUDA. */
int tbe_plan_create(const tbe_layout* L, void* dev_meta, size_t dev_meta_bytes, void* stream,
                    tbe_plan** plan_out);
void tbe_plan_destroy(tbe_plan* plan);

/*
 * Forward: out[b, D_offsets[t] + c] = sum_{i in bag(t,b)} w_i * W_t[id_i, c]
 * accumulated in FP32 and rounded once (nearest-even) to out_dtype.
 *   weights            : device, the packed table buffer
 *   indices            : device int64 [N], table-local ids
 *   offsets            : device int64 [T*B + 1], feature-major
 *   per_sample_weights : device fp32 [N] or NULL (unweighted); applies to
 *                        the tables the layout marks weighted
 *   out                : device [B, D_offsets[T]] of out_dtype, row-major;
 *                        every element is written (empty bags give 0)
 *   dev_status         : device int32 word or NULL
 * B == 0 or T*B == 0 is a no-op. */
int tbe_forward(const tbe_plan* plan, const void* weights, const int64_t* indices, int64_t N,
                const int64_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                int32_t* dev_status, void* stream);

/* Forward with an explicit path (TBE_PATH_*).  The histogram path ([FBT]
 * "The forward: a general gather and one clever special case": pooled sums
 * as per-bag counts times the table on the tensor cores) needs every table
 * of the plan to be fp16 or bf16 with 1..TBE_HIST_MAX_ROWS rows and D a
 * multiple of 16 up to 256; otherwise TBE_ERR_UNSUPPORTED.  It takes all T
 * tables in one launch, and per-sample weights on weighted tables (their
 * "counts" are fp32 sums of the weights).  TBE_PATH_AUTO additionally
 * requires the mean bag length N / (T * B) to reach the tuned threshold. */
#define TBE_HIST_MAX_ROWS 64
int tbe_forward_path(const tbe_plan* plan, const void* weights, const int64_t* indices, int64_t N,
                     const int64_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                     int32_t* dev_status, void* stream, int32_t path);

/* The forward with 32-bit ids and offsets (indices: device int32 [N];
 * offsets: device int32 [T*B + 1]; everything else as tbe_forward_path).
 * Half the index traffic of the int64 layout ([FBT] "A lookup table that is
 * most of the model": the jagged indices / offsets pair); results are
 * identical to tbe_forward_path on the same values. */
int tbe_forward_i32(const tbe_plan* plan, const void* weights, const int32_t* indices, int64_t N,
                    const int32_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                    int32_t* dev_status, void* stream, int32_t path);

/* Per-bag id histograms of every table of a histogram-eligible plan, the
 * count matrices the histogram path multiplies by the tables (device int32,
 * caller-owned, B * table_row_base[T] entries):
 *   counts[table_row_base[t] * B + b * rows_t + r] = #{i in bag(t, b) : id_i = r}.
 * Per-sample weights play no part.  Produced by the same kernel code as the
 * histogram forward. */
int tbe_histogram_counts(const tbe_plan* plan, const int64_t* indices, int64_t N,
                         const int64_t* offsets, int32_t B, int32_t* counts, int32_t* dev_status,
                         void* stream);

/*
 * Backward (row gradients).  For every global row r read by a valid lookup:
 *   row_grad[r, c] = sum_{i : table_row_base[t_i] + id_i = r} w_i * G[b_i, D_offsets[t_i] + c]
 * summed in FP32.
 *   grad_out          : device fp32 [B, D_offsets[T]]
 *   indices, offsets, per_sample_weights : as for tbe_forward
 *   unique_rows       : device int64 [N]; the first U entries receive the
 *                       ascending distinct global rows
 *   run_starts        : device int32 [N + 1] or NULL; entries 0..U receive
 *                       the start of each row's run in sorted order and the
 *                       number of valid lookups
 *   sorted_positions  : device int32 [N] or NULL; the lookup positions
 *                       ordered by (row, position) -- valid lookups first,
 *                       then those with a bad id in position order
 *   row_grads         : device fp32, capacity row_grads_capacity floats;
 *                       run u of table t is written at float offset
 *                       sum_{t'<t} U_t' * D_t' + (u - unique_count[t]) * D_t
 *                       (table-major blocks)
 *   unique_count      : device int64 [T + 1]; unique_count[t] = number of
 *                       distinct rows of tables < t, so unique_count[T] = U
 *   workspace         : device, >= tbe_backward_workspace_bytes(plan, B, N)
 *                       bytes, 256-byte aligned; contents need no
 *                       initialisation and are scratch after the call
 * If the row gradients need more than row_grads_capacity floats,
 * TBE_DEV_CAPACITY is set and the excess is not written. */
size_t tbe_backward_workspace_bytes(const tbe_plan* plan, int32_t B, int64_t N);
int tbe_backward(const tbe_plan* plan, const float* grad_out, const int64_t* indices, int64_t N,
                 const int64_t* offsets, int32_t B, const float* per_sample_weights,
                 int64_t* unique_rows, int32_t* run_starts, int32_t* sorted_positions,
                 float* row_grads, int64_t row_grads_capacity, int64_t* unique_count,
                 void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* The backward with 32-bit ids and offsets (int32 [N] and [T*B + 1]);
 * everything else, and every result, as tbe_backward. */
int tbe_backward_i32(const tbe_plan* plan, const float* grad_out, const int32_t* indices, int64_t N,
                     const int32_t* offsets, int32_t B, const float* per_sample_weights, int64_t* unique_rows,
                     int32_t* run_starts, int32_t* sorted_positions, float* row_grads, int64_t row_grads_capacity,
                     int64_t* unique_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream);

/*
 * Backward without a caller-provided workspace (the page has no counterpart;
 * this is an entry point for callers that cannot allocate device memory,
 * such as a plugin that an engine hands only a stream and its tensors).
 * Same arguments and results as tbe_backward, minus the workspace: the
 * scratch space is one array of TBE_STATIC_WORKSPACE_BYTES compiled into the
 * library, held on every GPU that loads it until the process exits.
 *   - Allocates nothing (no cudaMalloc / cudaFree, no allocating library
 *     call); inputs and outputs are still the caller's.
 *   - The first call on a device looks up the array's device address with
 *     that device current.
 *   - Batches whose scratch exceeds TBE_STATIC_WORKSPACE_BYTES (check with
 *     tbe_backward_workspace_bytes) are refused with TBE_ERR_WORKSPACE.
 *   - Every call on a device shares the array; calls whose work overlaps on
 *     the GPU (on other streams) race and must be serialised by the caller.
 */
#define TBE_STATIC_WORKSPACE_BYTES (32u << 20)
int tbe_backward_static_workspace(const tbe_plan* plan, const float* grad_out, const int64_t* indices,
                                  int64_t N, const int64_t* offsets, int32_t B,
                                  const float* per_sample_weights, int64_t* unique_rows,
                                  int32_t* run_starts, int32_t* sorted_positions, float* row_grads,
                                  int64_t row_grads_capacity, int64_t* unique_count,
                                  int32_t* dev_status, void* stream);

/*
 * Exact optimizer step ([FBT] "Why the backward is the hard half": the
 * update runs once per distinct row, on the row's finished gradient, so it
 * sees the whole sum).  Applies, in place, to every row a tbe_backward call
 * on the same stream produced (its outputs are passed unchanged):
 *   TBE_OPT_EXACT_SGD:
 *       W[r] <- W[r] - learning_rate * g
 *   TBE_OPT_EXACT_ROWWISE_ADAGRAD (one FP32 momentum scalar per row):
 *       m[r] <- m[r] + (sum_c g_c^2) / D_t
 *       W[r] <- W[r] - learning_rate / (sqrt(m[r]) + eps) * g
 * with g the row's gradient (D_t floats), computed in FP32 and stored
 * rounded to nearest-even in the table's dtype.
 *   weights            : device, the packed table buffer, updated in place
 *   momentum           : device fp32 [table_row_base[T]], one scalar per
 *                        global row, updated in place; Adagrad only (may be
 *                        NULL for SGD)
 *   unique_rows        : device int64, the backward's distinct rows
 *   max_unique         : capacity of unique_rows (the backward's N); runs at
 *                        or beyond it are never read
 *   row_grads, row_grads_capacity, unique_count : the backward's outputs
 *   dev_status         : device int32 word or NULL
 * Data errors skip the row and set a bit: TBE_DEV_BAD_INDEX for a row
 * outside its table, TBE_DEV_CAPACITY for a gradient beyond
 * row_grads_capacity or unique_count[T] > max_unique.
 * Errors: TBE_ERR_INVALID_ARG (nulls, an unknown kind, a learning rate or
 * eps that is not finite, a negative eps), TBE_ERR_UNSUPPORTED (row_grads
 * or weights not 16-byte aligned, a table width that is not a multiple
 * of 4). */
#define TBE_OPT_EXACT_SGD 0
#define TBE_OPT_EXACT_ROWWISE_ADAGRAD 1
typedef struct tbe_optimizer {
  int32_t kind;
  float learning_rate;
  float eps;
} tbe_optimizer;
int tbe_exact_update(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                     const int64_t* unique_rows, int64_t max_unique, const float* row_grads,
                     int64_t row_grads_capacity, const int64_t* unique_count, int32_t* dev_status,
                     void* stream);

/*
 * Backward with the exact optimizer fused into it ([FBT] "Why the backward
 * is the hard half": the update runs once per distinct row, on its finished
 * gradient, inside the backward; "Three tiers, routed by run length": the
 * long-run tier's last chunk applies it).  Same inputs and indexing outputs
 * as tbe_backward, but no row gradients are emitted: where a row's gradient
 * is finished -- the short-run tier's end of run, a one-chunk long run, or
 * the root of a long run's combine -- the row of `weights` (and its momentum)
 * is updated in place exactly as tbe_exact_update would update it, bit for
 * bit (same FP32 operations in the same order).
 *   opt, weights, momentum : as for tbe_exact_update (momentum may be NULL for
 *                            SGD)
 *   everything else        : as for tbe_backward (workspace size from
 *                            tbe_backward_workspace_bytes)
 * Every table's width must be at most 128 columns (a row gradient is one
 * quad per lane of one warp), else TBE_ERR_UNSUPPORTED; wider layouts use
 * tbe_backward followed by tbe_exact_update.
 * Errors: as tbe_backward, plus TBE_ERR_INVALID_ARG for an invalid optimizer
 * or a missing weights / momentum buffer. */
int tbe_backward_update(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                        const float* grad_out, const int64_t* indices, int64_t N, const int64_t* offsets,
                        int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                        int32_t* sorted_positions, int64_t* unique_count, void* workspace,
                        size_t workspace_bytes, int32_t* dev_status, void* stream);

/* tbe_backward_update with 32-bit ids and offsets (indices: device int32
 * [N]; offsets: device int32 [T*B + 1]; everything else as
 * tbe_backward_update); results identical to it on the same values. */
int tbe_backward_update_i32(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                            const float* grad_out, const int32_t* indices, int64_t N, const int32_t* offsets,
                            int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                            int32_t* sorted_positions, int64_t* unique_count, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * The backward in two calls ([FBT] "Using it, and the import that stops you":
 * the index transpose hoisted ahead of the gradient).  Everything up to the
 * reduction -- linearize, sort, segmentation, classification -- reads only
 * the ids, offsets and per-sample weights, so it can run before grad_out
 * exists, e.g. on a second stream beside the forward:
 *   tbe_backward_index  : those stages; writes unique_rows, run_starts,
 *                         sorted_positions (each optional as in
 *                         tbe_backward), unique_count and the workspace.
 *                         row_grads_capacity is the capacity the reduction
 *                         will get (INT64_MAX when it applies an optimizer);
 *                         a shortfall is reported here (TBE_DEV_CAPACITY).
 *   tbe_backward_reduce : the reduction, on the same plan, N, B, presence of
 *                         per-sample weights, unique_rows, run_starts,
 *                         unique_count and workspace, launched after the
 *                         index call has completed or on the same stream
 *                         after it.  With opt == NULL it writes row_grads
 *                         as tbe_backward; with an optimizer it updates
 *                         weights (and momentum) in place as
 *                         tbe_backward_update and writes no row gradients.
 * The pair gives exactly tbe_backward's (or tbe_backward_update's) results.
 * Errors: as tbe_backward / tbe_backward_update. */
int tbe_backward_index(const tbe_plan* plan, const int64_t* indices, int64_t N, const int64_t* offsets, int32_t B,
                       const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                       int32_t* sorted_positions, int64_t row_grads_capacity, int64_t* unique_count, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/* tbe_backward_index with 32-bit ids and offsets. */
int tbe_backward_index_i32(const tbe_plan* plan, const int32_t* indices, int64_t N, const int32_t* offsets,
                           int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                           int32_t* sorted_positions, int64_t row_grads_capacity, int64_t* unique_count,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

int tbe_backward_reduce(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                        const float* grad_out, int64_t N, int32_t B, const float* per_sample_weights,
                        int64_t* unique_rows, int32_t* run_starts, float* row_grads, int64_t row_grads_capacity,
                        int64_t* unique_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

/*
 * Tuning knobs (process-wide; set them before launching work that should
 * use them, not concurrently with launches).
 *   long_run_threshold : runs with at least this many lookups take the
 *                        long-run (chunked, multi-warp) tier; shorter runs
 *                        are reduced by one warp each
 *   long_chunk         : lookups per chunk of a long run (a multiple of 32,
 *                        or 0: chosen from the batch size, 64..256)
 *   fwd_unroll         : 16-byte row chunks in flight per lane in the
 *                        forward gather (4 or 8)
 *   fwd_lanes_per_row  : most lanes that share one row in the forward gather
 *                        (1, 2, 4, 8, 16 or 32); fewer lanes pool more bags
 *                        per warp at once
 *   red_unroll         : gradient slices in flight per lane in the backward
 *                        reduction (4: more resident warps, 8: deeper)
 *   fwd_ring           : forward kernel for layouts whose rows are at most
 *                        512 bytes: 2 = stream (a warp pools a run of
 *                        consecutive bags as one stream of rows copied into
 *                        a shared-memory ring; for tables of one shape with
 *                        D <= 192 and a batch that fits one wave of blocks at
 *                        <= 32 bags per block, a block's four warps pool equal
 *                        quarters of one run of bags), 1 = per-bag ring (16 rows in
 *                        flight per lane group), 0 = rows loaded into
 *                        registers, 3 = automatic (stream when every row
 *                        is at most 256 bytes, or at most 512 bytes with a
 *                        mean bag under 32 lookups; else per-bag ring);
 *                        rows wider than 512 bytes always use the register
 *                        kernel
 *   fwd_blocks_per_sm  : resident blocks per SM of the gather grid (0 = as
 *                        many as fit; 4 with fwd_unroll 4 selects a build
 *                        of the kernel with a smaller register budget)
 *   hist_min_mean_bag  : TBE_PATH_AUTO takes the histogram path only when
 *                        N / (T * B) reaches this; 0 (default) = the
 *                        measured gate: 16, or 32 when weighted tables get
 *                        per-sample weights
 *   short_item_lookups : lookups per work item of the short-run tier (runs
 *                        are grouped by 32 and cut into parts of about this
 *                        many lookups; raised to long_run_threshold if lower)
 * Values outside their ranges are rejected with TBE_ERR_INVALID_ARG. */
typedef struct tbe_tuning {
  int32_t long_run_threshold;
  int32_t long_chunk;
  int32_t fwd_unroll;
  int32_t fwd_blocks_per_sm;
  int32_t hist_min_mean_bag;
  int32_t short_item_lookups;
  int32_t fwd_lanes_per_row;
  int32_t red_unroll;
  int32_t fwd_ring;
} tbe_tuning;
int tbe_get_tuning(tbe_tuning* out);
int tbe_set_tuning(const tbe_tuning* in);

/* Stage timing: when enabled, each tbe_forward / tbe_backward records a CUDA
 * event after each of its kernels on its stream.  tbe_trace_read waits for
 * the last recorded call and returns up to max_stages stage durations in
 * milliseconds (stage k = time between events k-1 and k; stage 0 starts at
 * the call) plus their names.  Returns the number of stages (>= 0) or a
 * negative TBE_ERR_* code. */
int tbe_trace_enable(int32_t on);
int tbe_trace_read(float* stage_ms, const char** stage_names, int32_t max_stages);

/*
 * Failure-reporting self-test ([FBT] "Three tiers, routed by run length":
 * the fused tier's arrival counter is a wait between kernels' blocks; here
 * every such wait is bounded and reports a status instead of hanging).
 * Runs one of the library's bounded waits on something that never
 * completes and lets it give up after `polls` polls:
 *   kind 0 : the look-back word wait of the backward's scans, on a word no
 *            kernel publishes;
 *   kind 1 : the mbarrier wait of the histogram path, on a barrier that
 *            expects one arrival that never comes (no copy is in flight).
 * The kernel then OR-s TBE_DEV_TIMEOUT into *dev_status (device int32) and
 * returns; nothing traps, and the device stays usable.
 * Errors: TBE_ERR_INVALID_ARG (kind not 0/1, polls outside 1..2^20, null
 * dev_status), TBE_ERR_CUDA. */
int tbe_wait_selftest(int32_t kind, int32_t polls, int32_t* dev_status, void* stream);

/* Human-readable text for a return code. */
const char* tbe_status_string(int32_t code);

/* Library version string. */
const char* tbe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TBE_H_ */
