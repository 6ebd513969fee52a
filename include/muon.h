/*
 * muon.h -- C ABI of libmuon: the Muon optimizer step on one GB300 GPU.
 *
 * The step is the data-parallel hot path described by three DeepSpeed pull
 * requests about Muon under ZeRO:
 *   [BF16]  "Support Muon in BF16_Optimizer with FP32 gradient accumulation"
 *   [ONCE]  "Run Muon once per optimizer step under ZeRO-3, not once per
 *            micro-batch"
 *   [OFFL]  "Fix Muon optimizer under ZeRO CPU offload and bound gather
 *            buffers"
 *
 * Data model.  Every optimizer buffer (accumulated gradient, momentum, FP32
 * master weights, and each micro-batch's BF16 gradient) is one flat array
 * cut into partitions, one per emulated data-parallel rank ([BF16], PR
 * description: flat, rank-partitioned buffers with alignment padding).
 * Flat index i of partition p lives at storage element
 *     storage_offset[p] + (i - flat_begin[p])
 * of each buffer; the same mapping holds for all buffers.  A parameter is a
 * rows x cols row-major matrix occupying flat indices
 * [offset, offset + rows*cols).  Flat indices inside a partition that no
 * parameter covers are padding: no call reads or writes them.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device; host pointers are ordinary host memory and are only read
 *     during the call (tables are copied; the caller may free them after).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     GPU work is enqueued asynchronously on it.  Only calls that create a
 *     plan (below) and the diagnostic calls muon_device_error,
 *     muon_profile_read and muon_release_workspace synchronise the host.
 *     Once its plans exist, a sequence of muon_accumulate / muon_step /
 *     muon_step_ex calls may be captured into a CUDA graph and replayed.
 *   - Return value: MUON_OK (0) or a negative MUON_ERR_* code.  On error
 *     nothing has been enqueued, and muon_last_error() describes it.
 *   - The caller owns every buffer it passes.  The library owns a per-table
 *     workspace (device memory) and plans, created on the first muon_step
 *     with a given table set (and on the first call with new NS settings or
 *     a new workspace budget; muon_newton_schulz per shape) and freed by
 *     muon_release_workspace().  Creating a plan calls cudaMalloc and copies
 *     tables to the device, so such a call synchronises and must not be
 *     stream-captured.
 *   - Calls serialise on one library-wide lock; muon_last_error() reports
 *     the last error of any thread.
 */
#ifndef MUON_H
#define MUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

#define MUON_OK 0
#define MUON_ERR_INVALID (-1)     /* inconsistent tables or arguments */
#define MUON_ERR_UNSUPPORTED (-2) /* valid request outside what is built */
#define MUON_ERR_CUDA (-3)        /* a CUDA runtime/driver call failed */
#define MUON_ERR_OOM (-4)         /* workspace allocation failed */

/* One parameter.  use_muon = 0 marks an auxiliary (non-Muon) parameter:
 * it is counted in the global norm and clipped, but not orthogonalised
 * ([BF16], PR description: auxiliary Adam groups keep their own path).
 * num_heads > 1 splits the rows into num_heads contiguous blocks that are
 * normalised and orthogonalised independently (per-head Muon, [ONCE]
 * review thread, muon_num_heads); rows % num_heads must be 0.
 * 24 bytes, 8-byte aligned. */
typedef struct muon_param {
  int64_t offset;   /* flat index of element (0,0) */
  int32_t rows;     /* >= 1 */
  int32_t cols;     /* >= 1 */
  int32_t num_heads;
  int32_t use_muon; /* 1 = Muon matrix, 0 = auxiliary */
} muon_param_t;

/* One partition: flat indices [flat_begin, flat_end) stored at
 * storage_offset.  Partitions must be sorted by flat_begin, must not
 * overlap in flat space or in storage, and together must cover every
 * parameter.  24 bytes. */
typedef struct muon_partition {
  int64_t flat_begin;
  int64_t flat_end;
  int64_t storage_offset;
} muon_partition_t;

typedef enum {
  MUON_NS_STANDARD = 0, /* X <- aX + (bA + cA^2)X, A = XX^T            */
  MUON_NS_GRAM = 1      /* same map through R = X0 X0^T, Y = Q X0       */
} muon_ns_method_t;

typedef enum {
  MUON_OPERANDS_BF16 = 0, /* BF16 operands, FP32 accumulation (tensor cores) */
  MUON_OPERANDS_FP32 = 1  /* FP32 operands and accumulation                   */
} muon_operand_mode_t;

typedef enum { MUON_DTYPE_BF16 = 0, MUON_DTYPE_FP32 = 1 } muon_dtype_t;

/* Written on the device by muon_step (read it after synchronising). */
typedef struct muon_result {
  int32_t applied;   /* 1 = step applied, 0 = skipped (non-finite gradient) */
  int32_t ns_calls;  /* Newton-Schulz problems run this step (0 if skipped) */
  float global_norm; /* sqrt(sum ||u_muon||^2 + sum ||g_aux||^2)           */
  float clip_coef;   /* min(1, clip / (global_norm + 1e-6)); 1 if clip <= 0 */
} muon_result_t;

/* Host-side counters. */
typedef struct muon_stats {
  int64_t steps;                  /* muon_step calls enqueued */
  int64_t ns_calls_last_step;     /* NS problems enqueued by the last step */
  int64_t muon_matrices;          /* Muon parameters in the last step */
  int64_t kernel_launches_last_call; /* kernels the last call launched */
  int64_t kernel_launches_total;  /* kernels launched since load */
  size_t workspace_bytes;         /* device bytes held by all plans */
} muon_stats_t;

/* S1, FP32 gradient accumulation of one BF16 micro-batch ([BF16], PR
 * description; [ONCE], "The change": partitions accumulate the raw
 * gradient and Muon runs only at the step):
 *     accum[s] = (overwrite ? 0 : accum[s]) + scale * float(grad[s])
 * with scale*grad rounded to FP32 before the sum.  scale is normally
 * 1/gradient_accumulation_steps.
 *   accum : device float[storage size], in/out
 *   grad  : device bfloat16 bit patterns (uint16) with accum's layout
 *   n     : storage elements; used only when params == NULL, in which case
 *           all n elements are processed (padding included)
 *   params/nparams, parts/nparts : host tables; when given, only elements
 *           some parameter covers are touched (padding is left alone)
 * Errors: MUON_ERR_INVALID for bad tables or n < 0 with params == NULL. */
MUON_API int muon_accumulate(float* accum, const uint16_t* grad, int64_t n, float scale,
                    int overwrite, const muon_param_t* params, int nparams,
                    const muon_partition_t* parts, int nparts, void* stream);

/* S1 for several micro-batches in one pass over accum: bit for bit the
 * result of muon_accumulate called on grads[0], ..., grads[count - 1] in
 * that order, the first call with `overwrite` and the others adding:
 *     a = overwrite ? 0 : accum[s];
 *     for j in 0 .. count-1:  a = a + scales[j] * float(grads[j][s])
 *     accum[s] = a
 * (each product rounded to FP32 before its sum), reading accum at most once
 * and writing it once instead of once per micro-batch.
 *   grads  : host array of `count` device pointers, each bf16 bit patterns
 *            with accum's layout, 8-byte aligned; read during the call's
 *            work on `stream`
 *   scales : host array of `count` floats
 *   count  : 1 .. MUON_ACCUMULATE_MAX
 *   the other arguments as muon_accumulate.
 * Errors: as muon_accumulate; MUON_ERR_INVALID for count out of range or a
 * NULL or misaligned grads[j]. */
#define MUON_ACCUMULATE_MAX 8
MUON_API int muon_accumulate_n(float* accum, const uint16_t* const* grads, const float* scales,
                               int count, int64_t n, int overwrite, const muon_param_t* params,
                               int nparams, const muon_partition_t* parts, int nparts,
                               void* stream);

/* S2-S4, the optimizer step, once per accumulation boundary ([ONCE], "The
 * change"; [BF16], PR description):
 *   1. overflow check: any non-finite accum element of any parameter
 *      skips the step -- accum, momentum and master are left bit-identical
 *      and d_result->applied = 0;
 *   2. per Muon parameter (per head block): m <- beta*m + g (FP32, in
 *      place), X0 = m / (||m||_F + 1e-7), transposed if rows > cols,
 *      ns_steps Newton-Schulz steps (quintic 3.4445, -4.7750, 2.0315) by
 *      ns_method in operand_mode precision, transposed back: u;
 *   3. global norm over the Muon updates and the auxiliary gradients,
 *      coef = min(1, clip / (norm + 1e-6)) (clip <= 0: coef = 1);
 *   4. owned-slice write-back: Muon: accum = coef*u, master -= lr*coef*u;
 *      auxiliary: accum = coef*g, master untouched.  Padding untouched.
 *   accum, momentum, master : device float storage buffers, in/out
 *   d_result : device muon_result_t, written at the end of the step
 * Errors: MUON_ERR_INVALID (overlapping parameters, a parameter not covered
 * by the partitions, unsorted or overlapping partitions, overlapping
 * storage, rows/cols < 1, rows % num_heads != 0, NULL buffers),
 * MUON_ERR_UNSUPPORTED (ns_steps < 1 or > 64, unknown method or mode),
 * MUON_ERR_OOM, MUON_ERR_CUDA. */
MUON_API int muon_step(float* accum, float* momentum, float* master,
              const muon_param_t* params, int nparams,
              const muon_partition_t* parts, int nparts, float beta, float lr,
              int ns_method, int ns_steps, float clip, int operand_mode,
              muon_result_t* d_result, void* stream);

/* Options of muon_step_ex.  Zero-initialise, set struct_size, then set
 * what differs from the defaults (the defaults reproduce muon_step).
 *   clip_mode  MUON_CLIP_UPDATE (default): the global norm is taken over the
 *              Muon updates and the auxiliary gradients and scales every
 *              update ([ONCE], "The change").  MUON_CLIP_GRAD: the norm is
 *              taken over all gradients and the gradients are clipped
 *              before the momentum and Newton-Schulz ([BF16], PR
 *              description: Muon runs after reduction and global clipping);
 *              result.global_norm is then the gradient norm.
 *   grad_scale multiplies accum before anything else (0 means 1): pass
 *              1/S to undo a loss scale S, so neither the overflow check
 *              nor the clip norm sees it ([OFFL], loss-scaling commit).
 *   aux_adam   1: auxiliary parameters also get an Adam step on their
 *              clipped gradient, in place on master, exp_avg and exp_avg_sq
 *              (device float buffers with accum's layout; only auxiliary
 *              elements are touched): m = b1 m + (1-b1) g,
 *              v = b2 v + (1-b2) g g, w += -(lr/(1-b1^t)) m /
 *              (sqrt(v)/sqrt(1-b2^t) + eps) (Kingma & Ba); t = adam_step
 *              >= 1.  ([BF16], PR description: auxiliary Adam groups keep
 *              their own update path; fusing it is optional.)
 *   workspace_budget  bytes; 0 = unbounded.  Otherwise the Newton-Schulz
 *              blocks run in waves whose workspace fits the budget (a
 *              block larger than the budget runs alone), the unclipped
 *              update is parked in accum, and a final pass applies the clip
 *              coefficient (with MUON_CLIP_GRAD the coefficient is known
 *              before the waves and updates are written directly).  Results
 *              are bit-identical to the unbounded step.
 *   last_grad  non-NULL: the last micro-batch's gradients, folded into the
 *              step: on every element some parameter covers, the step's
 *              gradient is g[s] = (last_grad_overwrite ? 0 : accum[s]) +
 *              last_grad_scale * float(last_grad[s]), the arithmetic of
 *              muon_accumulate with those arguments.  accum, momentum,
 *              master and the result are bit-identical to that call
 *              followed by the step (a skipped step leaves g in accum).
 *              When a folded micro-batch overwrites accum's old value
 *              (last_grad_overwrite, or prev_grad_overwrite below), the
 *              step's kernels form g wherever they read it, so accum is
 *              written once per element (by the write-back) instead of
 *              twice; otherwise the step's first pass writes g into accum
 *              and the rest read it there.  Either way last_grad may be
 *              read by any of the step's kernels: it must stay unchanged
 *              until the step's work on `stream` has completed.  8-byte
 *              aligned.
 *   prev_grad  non-NULL (with last_grad): one more micro-batch folded in
 *              before last_grad: g[s] = (prev_grad_overwrite ? 0 :
 *              accum[s]) + prev_grad_scale * float(prev_grad[s]), then
 *              last_grad added as above -- the arithmetic of two
 *              muon_accumulate calls (prev, then last) followed by the
 *              step, bit for bit; accum is read only when neither
 *              overwrites it.  Same lifetime as last_grad; 8-byte aligned.
 *   stats_out  non-NULL: device double[4], written at the end of the step:
 *              [0] the sum of squares the clip norm was taken over (the
 *              Muon updates and the auxiliary gradients), [1] 1 if the step
 *              was skipped (non-finite gradient, or a device error) else 0,
 *              [2] the Newton-Schulz problems run, [3] 0.  A caller that
 *              splits the parameters over ranks adds these up across ranks
 *              (see muon_dp_finish).  8-byte aligned.
 * struct_size is sizeof(muon_step_options_t), MUON_STEP_OPTIONS_V2_SIZE for
 * callers built against the layout that ends at last_grad_overwrite, or
 * MUON_STEP_OPTIONS_V1_SIZE for the one that ends at workspace_budget. */
typedef enum { MUON_CLIP_UPDATE = 0, MUON_CLIP_GRAD = 1 } muon_clip_mode_t;

typedef struct muon_step_options {
  int32_t struct_size;   /* sizeof(muon_step_options_t) */
  int32_t clip_mode;     /* muon_clip_mode_t */
  float grad_scale;      /* 0 or 1 = no scaling */
  int32_t aux_adam;      /* 0 / 1 */
  float adam_lr, adam_beta1, adam_beta2, adam_eps;
  int64_t adam_step;     /* >= 1 when aux_adam */
  float* exp_avg;        /* device, when aux_adam */
  float* exp_avg_sq;     /* device, when aux_adam */
  uint64_t workspace_budget;
  /* -- absent when struct_size == MUON_STEP_OPTIONS_V1_SIZE -- */
  const uint16_t* last_grad;    /* device bf16, accum's layout, or NULL */
  float last_grad_scale;
  int32_t last_grad_overwrite;
  /* -- absent when struct_size <= MUON_STEP_OPTIONS_V2_SIZE -- */
  double* stats_out;            /* device double[4], or NULL */
  const uint16_t* prev_grad;    /* device bf16, accum's layout, or NULL */
  float prev_grad_scale;
  int32_t prev_grad_overwrite;
} muon_step_options_t;
#define MUON_STEP_OPTIONS_V1_SIZE 64   /* struct_size of the layout without last_grad */
#define MUON_STEP_OPTIONS_V2_SIZE 80   /* struct_size of the layout without stats_out */

/* muon_step with options (NULL = defaults).  Errors as muon_step, plus
 * MUON_ERR_INVALID for a bad struct_size, a non-finite or negative
 * grad_scale, aux_adam without state buffers or with adam_step < 1. */
MUON_API int muon_step_ex(float* accum, float* momentum, float* master,
                          const muon_param_t* params, int nparams,
                          const muon_partition_t* parts, int nparts, float beta,
                          float lr, int ns_method, int ns_steps, float clip,
                          int operand_mode, const muon_step_options_t* opts,
                          muon_result_t* d_result, void* stream);

/* ---------------------------------------------------------------------
 * Data parallelism across ranks (one process per GPU).
 *
 * The pages run the step on ranks that each hold only their partitions of
 * the flat buffers: each Muon matrix needs its slices from every rank that
 * holds one, Newton-Schulz runs on whole matrices, and every rank writes
 * back its owned intersection ("Support Muon in BF16_Optimizer with FP32
 * gradient accumulation", PR description and review thread on
 * all_to_all_single: static send/recv split tables computed once, only the
 * slices that cross partitions exchanged; "Run Muon once per optimizer step
 * under ZeRO-3, not once per micro-batch", "The change": Muon round-robin
 * over ranks, each rank's slice written back).  Here:
 *   1. a plan assigns every parameter (Muon and auxiliary) to one owner
 *      rank and derives the exchange tables (host only, no GPU);
 *   2. muon_dp_pack gathers each rank's slices (gradient, and momentum for
 *      Muon parameters) into a send buffer, ordered by owner; the caller
 *      runs one all-to-all with the plan's split sizes;
 *   3. muon_dp_unpack places the received slices into the owner's packed
 *      buffers of its whole parameters, and muon_step_ex runs on them with
 *      the plan's owned tables, clip = 0, lr = 0 and stats_out set: the
 *      packed accum then holds the unclipped update u (the auxiliary
 *      gradient for auxiliary parameters) and the packed momentum m';
 *   4. the caller adds stats_out up over the ranks (one all-reduce of four
 *      doubles: the global sum of squares, the skip count, the NS count);
 *   5. muon_dp_pack in the receive direction gathers u and m' back into the
 *      receive layout; the caller runs the reverse all-to-all (split sizes
 *      swapped), which lands every slice in its holder's send layout;
 *   6. muon_dp_finish computes coef = min(1, clip / (sqrt(sum) + 1e-6)) on
 *      the device and writes each held slice: Muon accum = coef u, master
 *      -= lr coef u, momentum = m'; auxiliary accum = coef g.  A step that
 *      any rank skipped writes nothing.
 * A plan's partition table lists every rank's partitions (global flat
 * ranges), part_rank[p] names the rank that holds partition p, and each
 * storage_offset is an index into that rank's own buffers.
 * ------------------------------------------------------------------- */
typedef struct muon_dp_plan muon_dp_plan_t;   /* opaque */

typedef enum {
  MUON_DP_BALANCED = 0,   /* largest first onto the least loaded rank */
  MUON_DP_ROUND_ROBIN = 1 /* parameter k on rank k mod world (the pages' order) */
} muon_dp_assign_t;

/* One slice of one parameter held by one rank and owned by another (or the
 * same) rank.  The send list of a rank is ordered by (owner, parameter,
 * position); the receive list by (holder, parameter, position). */
typedef struct muon_dp_segment {
  int32_t param;    /* parameter index in the table */
  int32_t peer;     /* send list: the owner; receive list: the holder */
  int32_t is_muon;  /* 1: the momentum slice follows the gradient slice */
  int32_t pad;
  int64_t len;      /* elements */
  int64_t local;    /* send list: storage index in this rank's buffers;
                       receive list: index in the packed owned buffers */
  int64_t buf;      /* offset of the slice in the exchange buffer; a Muon
                       slice's momentum (or m') follows at buf + len */
} muon_dp_segment_t;   /* 40 bytes */

typedef struct muon_dp_sizes {
  int32_t world, rank;
  int32_t owned_params;   /* parameters this rank owns */
  int32_t nparams;
  int64_t owned_elems;    /* elements of each packed owned buffer */
  int64_t send_segments, recv_segments;
  int64_t send_elems;     /* elements of the send buffer (sum of send counts) */
  int64_t recv_elems;     /* elements of the receive buffer */
  double owned_cost;      /* this rank's share of the assignment's cost model */
  double max_cost;        /* the most loaded rank's */
} muon_dp_sizes_t;

/* Builds the plan of `rank` (host only; no CUDA call).  ns_method feeds the
 * cost model (formula flops of the NS iteration plus the streaming passes,
 * 12500 flop-equivalents per element: ~50 bytes per element at the tensor
 * rate per HBM byte of a GB300).
 * Errors: MUON_ERR_INVALID for overlapping or uncovered parameters,
 * unsorted or overlapping partitions, overlapping storage within a rank,
 * part_rank outside [0, world), rank outside [0, world), world < 1. */
MUON_API int muon_dp_plan_create(const muon_param_t* params, int nparams,
                                 const muon_partition_t* parts, const int32_t* part_rank,
                                 int nparts, int world, int rank, int ns_method, int assign,
                                 muon_dp_plan_t** out);
MUON_API void muon_dp_plan_destroy(muon_dp_plan_t* plan);
MUON_API int muon_dp_plan_sizes(const muon_dp_plan_t* plan, muon_dp_sizes_t* out);
/* Copies the plan's tables into caller arrays (any may be NULL):
 *   owner[nparams]            owner rank of every parameter
 *   send_counts[world]        elements this rank sends to each rank
 *   recv_counts[world]        elements it receives from each rank
 *   owned_params[owned_params] the owned parameters with offsets in the
 *                             packed owned buffers (one partition covers
 *                             [0, owned_elems), storage offset 0)
 *   send_segs[send_segments], recv_segs[recv_segments] */
MUON_API int muon_dp_plan_tables(const muon_dp_plan_t* plan, int32_t* owner,
                                 int64_t* send_counts, int64_t* recv_counts,
                                 muon_param_t* owned_params, muon_dp_segment_t* send_segs,
                                 muon_dp_segment_t* recv_segs);

/* Exchange buffers (device float).  direction MUON_DP_SEND: for every send
 * segment, buf[seg.buf + i] = a[seg.local + i] and, for Muon slices,
 * buf[seg.buf + seg.len + i] = b[seg.local + i] (a = accum, b = momentum,
 * this rank's storage buffers).  MUON_DP_RECV: the same over the receive
 * segments (a, b = the packed owned buffers).  muon_dp_unpack is the
 * inverse copy.  The first device call of a plan uploads its segments
 * (cudaMalloc; must not be stream-captured).  Errors: MUON_ERR_INVALID for
 * NULL buffers, MUON_ERR_CUDA. */
typedef enum { MUON_DP_SEND = 0, MUON_DP_RECV = 1 } muon_dp_direction_t;
MUON_API int muon_dp_pack(muon_dp_plan_t* plan, int direction, float* buf, const float* a,
                          const float* b, void* stream);
MUON_API int muon_dp_unpack(muon_dp_plan_t* plan, int direction, const float* buf, float* a,
                            float* b, void* stream);

/* The write-back of step 6 above, on this rank's storage buffers, from the
 * reverse exchange's buffer (send layout: u, then m' for Muon slices) and
 * the all-reduced stats (device double[4], as muon_step_ex's stats_out
 * summed over the ranks).  Writes d_result (applied = 0 when stats[1] > 0,
 * ns_calls = stats[2], global_norm, clip_coef) for every rank alike. */
MUON_API int muon_dp_finish(muon_dp_plan_t* plan, const float* buf, float* accum,
                            float* momentum, float* master, const double* stats, float lr,
                            float clip, muon_result_t* d_result, void* stream);

/* Newton-Schulz orthogonalisation of one rows x cols row-major matrix:
 * normalise by the Frobenius norm (+1e-7), transpose if rows > cols,
 * ns_steps quintic steps by ns_method, transpose back.
 *   X, Y     : device arrays of io_dtype (muon_dtype_t), rows*cols each;
 *              X is read only; Y may not alias X
 *   operand_mode : arithmetic precision (muon_operand_mode_t)
 * Uses a library workspace sized for the shape (kept until
 * muon_release_workspace).  Errors as muon_step. */
MUON_API int muon_newton_schulz(const void* X, void* Y, int rows, int cols, int io_dtype,
                       int ns_method, int ns_steps, int operand_mode, void* stream);

/* Newton-Schulz of one matrix (the arguments and the computation of
 * muon_newton_schulz) with no device allocation, for callers that cannot
 * call cudaMalloc: processes whose device memory is handed out by another
 * allocator that reserves it up front (a framework's caching allocator,
 * which a direct cudaMalloc would bypass or find exhausted), and runtimes
 * that forbid allocation once they serve (cudaMalloc may synchronise the
 * device and stall a latency-bound loop).  It calls no cudaMalloc/cudaFree
 * and no allocating library routine; all of its scratch (norm partials,
 * the X and m x m work matrices, GEMM and TMA descriptors) sits in one
 * fixed 16 MiB __device__ array inside the library, which every GPU that
 * loads the library holds until the process exits.  The pages have no
 * counterpart of this entry point.
 *   Kernels: BF16-operand products run on the single-SM tensor-core
 *   kernel; FP32-operand products and gram's m x m recurrence run on the
 *   CUDA-core FP32 GEMM (muon_newton_schulz uses SM pairs and the split-3
 *   tensor-core products there), so the two entries agree within the
 *   operand mode's tolerance, not bit for bit.
 *   Limits: rows * cols <= MUON_NOALLOC_MAX_ELEMS, min(rows, cols) <=
 *   MUON_NOALLOC_MAX_MIN_DIM, max(rows, cols) <= MUON_NOALLOC_MAX_DIM;
 *   larger matrices return MUON_ERR_UNSUPPORTED (see muon_last_error()).
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it; make
 *   that first call before any stream capture.
 *   All calls share the one array and leave their contents in it: two
 *   calls whose work overlaps on the GPU (different streams) race and
 *   corrupt each other's results.  Host threads may call concurrently: a
 *   call holds the library lock while it builds its descriptors and copies
 *   them (from host arrays that the next call reuses) onto `stream`.
 *   A bounded wait that runs out in its tensor-core products records a
 *   code that muon_device_error reports. */
#define MUON_NOALLOC_MAX_ELEMS 1048576
#define MUON_NOALLOC_MAX_MIN_DIM 512
#define MUON_NOALLOC_MAX_DIM 16384
MUON_API int muon_newton_schulz_noalloc(const void* X, void* Y, int rows, int cols,
                                        int io_dtype, int ns_method, int ns_steps,
                                        int operand_mode, void* stream);

/* Host-side counters (no GPU work).  Returns MUON_OK. */
MUON_API int muon_get_stats(muon_stats_t* out);

/* What a step over these tables would do, computed on the host alone (no
 * CUDA call, no GPU needed): the tables are validated as muon_step
 * validates them (same errors), and the Newton-Schulz grouping is the one
 * the tensor-core path of a GB300 uses for ns_method and operand_mode. */
typedef struct muon_table_info {
  int64_t muon_params;      /* parameters with use_muon = 1 */
  int64_t muon_blocks;      /* their head blocks: Newton-Schulz calls per step */
  int64_t ns_problems;      /* after stacking equal consecutive blocks */
  int32_t pair_engine;      /* 1: BF16 products on SM pairs (256-row tiles) */
  int32_t stack_rows;       /* rows cap of a stack (0: no stacking) */
  int64_t muon_elements;    /* elements of the Muon parameters */
  int64_t aux_elements;     /* elements of the auxiliary parameters */
  int64_t padding_elements; /* flat indices inside partitions no parameter covers */
  int64_t segments;         /* (block or auxiliary parameter) x partition runs */
  uint64_t workspace_bytes; /* the unbounded plan's Newton-Schulz work regions */
} muon_table_info_t;
MUON_API int muon_describe_tables(const muon_param_t* params, int nparams,
                                  const muon_partition_t* parts, int nparts, int ns_method,
                                  int operand_mode, muon_table_info_t* out);

/* Cross-checks for tests (not a production setting): plans built after
 * the call route the Newton-Schulz products through another kernel or
 * schedule, so tests can compare them with the product path.  Existing
 * plans keep what they were built with (muon_release_workspace drops them).
 * Every knob's default is the product path.
 *   MUON_TEST_GEMM        0 default; 1 CUDA-core GEMM for every product;
 *                         2 single-SM tensor-core kernel instead of SM pairs
 *   MUON_TEST_STACK       1 default (equal consecutive blocks stacked); 0 off
 *   MUON_TEST_FLOW        1 default (one SM-pair launch per iteration);
 *                         0 one launch per product
 *   MUON_TEST_FLOW_LAG    0 default (half the problems); k >= 1
 *   MUON_TEST_FLOW_WAVES  1 default; k >= 1 groups of problems
 *   MUON_TEST_RASTER      0 default (large products with an MN-major B run
 *                         their tiles in groups of 4 column tiles); 1
 *                         row-major order; k in [2, 64]: groups of k
 *   MUON_TEST_EXTENT_SHRINK  0 default; k > 0: a library built with
 *                         MUON_DEBUG checks its streaming kernels' tiles
 *                         against a storage extent k elements smaller than
 *                         the partitions describe (to see the check report)
 * Errors: MUON_ERR_INVALID for an unknown knob or value. */
typedef enum {
  MUON_TEST_GEMM = 0,
  MUON_TEST_STACK = 1,
  MUON_TEST_FLOW = 2,
  MUON_TEST_FLOW_LAG = 3,
  MUON_TEST_FLOW_WAVES = 4,
  MUON_TEST_RASTER = 5,
  MUON_TEST_EXTENT_SHRINK = 6
} muon_test_knob_t;
MUON_API int muon_testing_set(int knob, int value);

/* Message for the last error on this thread ("" if none). */
MUON_API const char* muon_last_error(void);

/* Frees every plan and workspace (synchronises the device first). */
MUON_API void muon_release_workspace(void);

/* Synchronises the device and returns the first error code a kernel
 * recorded since the last query (0 = none), clearing it.  The tensor-core
 * kernels bound every wait; a wait that runs out records a positive code
 * here instead of hanging (1 = TMA producer, 2 = MMA issuer, 3 = epilogue,
 * 4 = a dependency of the SM-pair kernel).  A library built with MUON_DEBUG
 * also checks every streaming-kernel tile against the extents its tables
 * describe and records 16 for a tile that would leave them (and skips it).
 * A step whose products hit such an error also reports applied = -1. */
MUON_API int muon_device_error(void);

/* Phase timing with CUDA events on the launching stream, for benchmarks.
 * muon_profile_enable(1) makes every later call record an event pair
 * around each kernel launch; muon_profile_read() synchronises those events
 * and returns, per phase, the launch count and total device milliseconds
 * accumulated since the last reset, plus the algorithmic bytes moved or
 * flops executed.  Phases are indexed by muon_phase_t. */
typedef enum {
  MUON_PHASE_ACCUMULATE = 0, /* S1 */
  MUON_PHASE_REDUCE = 1,     /* S2 pass 1: overflow check + sums of squares */
  MUON_PHASE_GATHER = 2,     /* S2 pass 2: momentum write + X0 */
  MUON_PHASE_NS_GEMM = 3,    /* S3: the Newton-Schulz matrix products */
  MUON_PHASE_NORM = 4,       /* S4a: update sums of squares, norm, clip */
  MUON_PHASE_SCATTER = 5,    /* S4b: owned-slice write-back */
  MUON_PHASE_COUNT = 6
} muon_phase_t;

typedef struct muon_phase_time {
  int64_t launches;
  double total_ms;
  double algorithmic_bytes;
  double algorithmic_flops;
} muon_phase_time_t;

MUON_API int muon_profile_enable(int on);
/* As muon_profile_enable, for the phases whose bit (1 << muon_phase_t) is
 * set in mask only (0 = off); fewer events perturb a timed run less.  Calls
 * issued while their stream is captured into a CUDA graph record the events
 * as nodes of the graph, timed again by every replay. */
MUON_API int muon_profile_enable_phases(uint32_t mask);
MUON_API int muon_profile_read(muon_phase_time_t* out, int nphases, int reset);

#ifdef __cplusplus
}
#endif
#endif /* MUON_H */
