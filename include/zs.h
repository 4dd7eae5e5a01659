/*
 * zs.h - C ABI of the sharded mixed-precision AdamW step over a flat, padded
 * parameter buffer (ZeRO-1/2/3, FSDP1 FlatParameter), for one sm_103a GPU on
 * which the N_d data-parallel ranks are simulated as separate device buffers.
 *
 * The method is the one described in "Infra: Data Parallel" (F. Pu):
 *   - section "Naive Data Parallelism": gradient buckets, gradient accumulation
 *     over micro-batches with the loss divided by their number;
 *   - section "Zero Redundancy Optimizer (ZeRO)": Reduce-Scatter with
 *     averaging, an element-wise AdamW update of each rank's shard with fp32
 *     master weights and moments (k = 12 bytes per parameter), All-Gather of
 *     the updated 16-bit parameters; ZeRO-2 bucket-wise reduction; ZeRO-3
 *     per-layer gather / reduce-scatter with no gather after the update;
 *   - section "Fully Sharded Data Parallel (FSDP)", subsection "FSDP1": the
 *     FlatParameter (flatten + concatenate the parameters of one unit, pad,
 *     cut into N_d equal contiguous shards that may cross parameter
 *     boundaries; a rank holding nothing of a parameter sees an empty view).
 *
 * ---------------------------------------------------------------------------
 * Conventions (all entry points)
 *
 * Types.      Parameters and gradients are bf16 (16-bit, stored as 2-byte
 *             words); master weights, m and v are fp32.
 * Indices.    Every element has one GLOBAL FLAT INDEX i in [0, padded_numel):
 *             the units' padded FlatParameters laid one after another in
 *             unit order.  Unit u covers [base_u, base_u + padded_u); rank r
 *             owns [base_u + r*S_u, base_u + (r+1)*S_u) of it, S_u =
 *             padded_u / N_d.  Padding elements are zero in every buffer.
 * Buffer kinds (how a pointer argument maps global index i of rank q):
 *   ZS_RANK_FULL   N_d pointers; ptrs[q][i]              (whole flat space)
 *   ZS_SHARDED     1 pointer;    ptrs[0][i]              (each rank's shard of
 *                  every unit at its owned position: the concatenation of all
 *                  ranks' shards; on separate GPUs each rank would hold only
 *                  its own piece)
 *   ZS_RANK_BUCKET N_d pointers; ptrs[q][i - bucket_begin] (one bucket)
 *   ZS_RANK_UNIT   N_d pointers; ptrs[q][i - unit_base]    (one unit)
 *             master, m and v are ZS_SHARDED fp32 arrays of padded_numel
 *             elements, except in zs_rank_shard_step, which takes one rank's
 *             own state in that rank's local layout (its shard of every unit,
 *             back to back) for the mode with one rank per process and GPU.
 * Ownership.  The caller owns all device memory and all streams.  The library
 *             never allocates device memory; its module memory holds a status
 *             word (zs_device_status), 1024 counter pairs for the dynamic tile
 *             order of the launches over ranges of 2^24 elements and more (the
 *             fused steps, the ZeRO-3 gathers and updates, the update alone, the
 *             naive-DP all-reduce and step: one pair per such launch in flight,
 *             drawn in turn, so at most 1024 of those launches may run at once
 *             on a device) and the staging array of zs_zero2_step_host_noalloc.
 *             The step calls never
 *             synchronise and enqueue work only on the streams they are given
 *             (a cudaStream_t; NULL is the legacy default stream); calls that
 *             use a second stream order it after the first with events.  The
 *             checkpoint calls are the exception: they synchronise their stream
 *             and return with the data in place.  A plan owns host tables only.
 * Alignment.  Every device pointer must be 16-byte aligned.
 * Aliasing.   Inputs and outputs must not overlap unless a call says so.
 * Step.       The AdamW step t is 1-based.
 * Errors.     Every entry point returns ZS_OK or a negative status.  Argument
 *             errors are found before anything is enqueued (nothing is
 *             written); zs_last_error() then returns a message (thread-local,
 *             valid until the next call on that thread).  Launch failures
 *             return ZS_ERR_CUDA.  Faults inside kernels surface at the
 *             caller's next synchronisation, as with any CUDA launch.
 * Threads.    A plan is immutable after creation and may be shared by
 *             threads; calls on different streams may run concurrently when
 *             their buffers do not overlap.
 * Graphs.     Because the step calls only enqueue work, a sequence of them
 *             (including the two-stream ones) may be captured into a CUDA
 *             graph and replayed, which removes the host's per-call time
 *             between short kernels (e.g. per-group FSDP2 conversions).  The
 *             step number, hyper-parameters and pointers are kernel arguments:
 *             a replay repeats the values it was captured with.  The
 *             checkpoint calls synchronise and cannot be captured.
 */
#ifndef ZS_H
#define ZS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */
#define ZS_OK               0
#define ZS_ERR_INVALID     (-1)   /* bad argument: nothing was enqueued              */
#define ZS_ERR_CUDA        (-2)   /* a CUDA runtime call or launch failed            */
#define ZS_ERR_OOM_HOST    (-3)   /* host allocation for plan tables failed          */
#define ZS_ERR_UNSUPPORTED (-5)   /* valid request the library does not implement     */

#define ZS_STAGE_DP     0         /* naive data parallel (no sharding)               */
#define ZS_STAGE_ZERO1  1         /* optimizer state sharded                         */
#define ZS_STAGE_ZERO2  2         /* + gradients sharded                             */
#define ZS_STAGE_ZERO3  3         /* + parameters sharded (FSDP full shard)          */

#define ZS_RANK_FULL    0
#define ZS_SHARDED      1
#define ZS_RANK_BUCKET  2
#define ZS_RANK_UNIT    3

#define ZS_MAX_RANKS    64        /* largest N_d accepted                            */

#define ZS_LAYOUT_FSDP1 0         /* FlatParameter: units flattened, padded, cut evenly   */
#define ZS_LAYOUT_FSDP2 1         /* per-parameter Shard(0), rank-major group buffer      */

#define ZS_FUSED_AUTO   0         /* staged kernel for large 8-aligned ranges, else streaming */
#define ZS_FUSED_LDG    1         /* register-streaming kernel (16-byte loads/stores)   */
#define ZS_FUSED_TMA    2         /* bulk-copy staged kernel wherever it applies       */

#define ZS_DEVERR_NONE          0u
#define ZS_DEVERR_PRODUCER_WAIT 1u   /* a staged kernel's producer gave up waiting for a free stage */
#define ZS_DEVERR_CONSUMER_WAIT 2u   /* a staged kernel's consumer gave up waiting for its data     */
#define ZS_DEVERR_SELFTEST      3u   /* zs_selftest_wait_timeout ran its wait out (expected)         */
#define ZS_DEVERR_GATHER_WAIT   4u   /* a bulk-store gather gave up waiting for its tile             */

typedef struct zs_plan_s* zs_plan_t;

/* AdamW hyper-parameters, as fp32 values. */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
} zs_adamw_hparams;

/* ------------------------------------------------------------------ plan (host only) */

/* Build the FlatParameter plan.  "Infra: Data Parallel", FSDP section, FSDP1
 * layout figure and subsection "FSDP1"; buckets from section "Naive Data
 * Parallelism".
 *   n_params        number of parameters (>= 1), in module order.
 *   ndims[k]        rank of parameter k's shape (0..8; 0 = scalar, one element).
 *   dims            all shapes concatenated (sum of ndims entries), each >= 1.
 *   unit_of_param   unit id of each parameter, ids 0..U-1 all used; NULL puts
 *                   every parameter in unit 0.  Parameters of a unit keep their
 *                   relative order; unit u's FlatParameter is padded on its own
 *                   with the fewest zeros that make its length a multiple of n_d.
 *   n_d             number of data-parallel ranks, 1..ZS_MAX_RANKS.
 *   stage           ZS_STAGE_* (recorded; used as the default for accounting).
 *   bucket_bytes    gradient bucket size in bytes of bf16 gradients; a bucket is
 *                   floor(bucket_bytes/2) consecutive elements of one unit (the
 *                   last bucket of a unit is shorter).  <= 0 means one bucket per unit.
 *   out             receives the plan; release it with zs_plan_destroy.
 * Errors: ZS_ERR_INVALID for any out-of-range argument; ZS_ERR_OOM_HOST. */
int zs_plan_create(int32_t n_params, const int32_t* ndims, const int64_t* dims,
                   const int32_t* unit_of_param, int32_t n_d, int32_t stage,
                   int64_t bucket_bytes, zs_plan_t* out);
void zs_plan_destroy(zs_plan_t plan);

/* Same arguments as zs_plan_create, FSDP2 layout ("Infra: Data Parallel", FSDP
 * section, FSDP2 layout figure and subsection "FSDP2": every parameter keeps its
 * global shape and is cut along dimension 0; a group's parameters are still
 * gathered and reduce-scattered together).  Parameter k (d0 rows of `row`
 * elements; a 0-d parameter is one row of one element) gives rank r the rows
 * [r*c_k, min((r+1)*c_k, d0)), c_k = ceil(d0 / N_d).  Rank r's shard of a unit is
 * its pieces of the unit's parameters in order, each padded with zero rows to c_k
 * rows, so S_u = sum of c_k * row_k and the unit's flat range is the N_d shards one
 * after another (padded_u = N_d * S_u).  Every other call of this header works on
 * such a plan unchanged (the step is element-wise); zs_fsdp2_chunk_cat and
 * zs_fsdp2_copy_out convert to and from the parameters' own layout.  For an FSDP2
 * plan zs_plan_param's flat_offset is rank 0's piece; zs_plan_param_segment gives
 * each rank's piece (real rows only).  Errors as zs_plan_create. */
int zs_plan_create_fsdp2(int32_t n_params, const int32_t* ndims, const int64_t* dims,
                         const int32_t* unit_of_param, int32_t n_d, int32_t stage,
                         int64_t bucket_bytes, zs_plan_t* out);

/* ZS_LAYOUT_FSDP1 or ZS_LAYOUT_FSDP2. */
int zs_plan_layout(zs_plan_t plan, int32_t* layout);

/* Dimension-0 split of parameter k on rank r (FSDP2 subsection: local shape =
 * (nrows, rest of the global shape)): first row, number of rows (0 when the rank
 * holds none), rows per rank c_k, elements per row.  Valid for both layouts (the
 * FSDP1 layout does not use it). */
int zs_plan_param_rows(zs_plan_t plan, int32_t k, int32_t rank, int64_t* row_begin, int64_t* nrows,
                       int64_t* rows_per_rank, int64_t* row_elems);

/* Global flat ranges [begin, end) that hold padding (zeros in every buffer), in
 * increasing order: the tail of each unit for FSDP1, the padding rows of every
 * rank's piece for FSDP2.  Writes at most `capacity` ranges and sets *count to the
 * total number (call with capacity 0 to size the arrays). */
int zs_plan_pad_ranges(zs_plan_t plan, int64_t* begins, int64_t* ends, int64_t capacity, int64_t* count);

/* Totals.  Any output pointer may be NULL. */
int zs_plan_info(zs_plan_t plan, int64_t* numel, int64_t* padded_numel,
                 int64_t* shard_numel_per_rank, int32_t* n_units, int32_t* n_buckets,
                 int32_t* n_d, int32_t* stage);
/* Unit u: global base index, real and padded element counts, shard size S_u. */
int zs_plan_unit(zs_plan_t plan, int32_t u, int64_t* base, int64_t* numel,
                 int64_t* padded_numel, int64_t* shard_numel);
/* Bucket b (0..n_buckets-1, ordered by global index): its unit and global range [begin, end). */
int zs_plan_bucket(zs_plan_t plan, int32_t b, int32_t* unit, int64_t* begin, int64_t* end);
/* The part [begin, end) of bucket b that the reduce-scatter hands to rank r (begin == end: none). */
int zs_plan_bucket_rank_slice(zs_plan_t plan, int32_t b, int32_t rank, int64_t* begin, int64_t* end);
/* Parameter k: unit and global flat range [flat_offset, flat_offset + numel). */
int zs_plan_param(zs_plan_t plan, int32_t k, int32_t* unit, int64_t* flat_offset, int64_t* numel);
/* The view of parameter k on rank r ("use_orig_params", subsection "FSDP1"):
 * global flat_begin, offset inside the rank's shard of the unit, and length.
 * A rank holding no element of the parameter gets len = 0 and zeros for the
 * other two (the empty view). */
int zs_plan_param_segment(zs_plan_t plan, int32_t k, int32_t rank, int64_t* flat_begin,
                          int64_t* shard_offset, int64_t* len);
/* Model-state bytes one rank holds under `stage` ("Infra: Data Parallel", ZeRO
 * memory figure): parameters and gradients at 2 bytes, master/m/v at 4 bytes
 * each (k = 12); sharded stages hold the padded FlatParameter. */
int zs_plan_memory_bytes(zs_plan_t plan, int32_t stage, int64_t* bytes_per_rank);
/* Bytes one rank sends in one step under `stage` (ZeRO section, communication
 * paragraphs; 16-bit elements, every bucket and unit summed): DP ring
 * all-reduce, ZeRO-1/2 reduce-scatter + all-gather, ZeRO-3 reduce-scatter +
 * one or two all-gathers (two when reshard_after_forward != 0, FSDP2
 * subsection). */
int zs_plan_comm_bytes(zs_plan_t plan, int32_t stage, int32_t reshard_after_forward,
                       int64_t* bytes_sent_per_rank);

/* The eight fp32 scalars AdamW uses at step t (host only), in this order:
 * beta1, beta2, eps, decay = 1 - lr*wd, c1 = 1 - beta1, c2 = 1 - beta2,
 * step_size = lr / (1 - beta1^t), sqrt_bc2 = sqrt(1 - beta2^t); each computed
 * in double from the fp32 hyper-parameters, then rounded to fp32. */
int zs_adamw_scalars(const zs_adamw_hparams* hp, int64_t step, float* out8);

/* Message for the last non-OK return on this thread ("" if none). */
const char* zs_last_error(void);

/* Selects the kernel behind zs_fused_step, zs_fused_step_buckets,
 * zs_zero3_rs_step_unit and zs_dp_step for the whole process (ZS_FUSED_AUTO,
 * ZS_FUSED_LDG or ZS_FUSED_TMA).  Every variant
 * computes bit-identical results; they differ in how data reaches the SMs.  The
 * staged kernel exists for N_d in {2, 4, 8, 16, 32} and needs the range's buffers
 * on the 8-element grid; elsewhere the streaming kernel runs.  Set it before
 * enqueueing work from other threads.  Errors: ZS_ERR_INVALID for an unknown value. */
int zs_set_fused_variant(int32_t variant);

/* Programmatic dependent launch (sm_90 and later) for every kernel of the
 * library, for the whole process: enable != 0 (the default) launches each kernel
 * so that it may be scheduled while the previous kernel on its stream drains;
 * the kernel waits for that kernel to complete, with its memory visible, before
 * it touches global memory, so stream order holds for every byte and results
 * are identical either way.  It shortens the gap between back-to-back launches
 * (bucket-by-bucket steps, per-group calls).  enable = 0 launches plainly.
 * Set it before enqueueing work from other threads.  Never fails (ZS_OK). */
int zs_set_dependent_launch(int32_t enable);

/* Device-side status of the current device (ZS_DEVERR_*): a staged kernel whose
 * bounded wait ran out records a code here, stops, waits (bounded) for its
 * copies in flight and returns, leaving the context usable.  This call copies
 * the word to the host, so it waits for the device's prior work; clear != 0
 * resets it to ZS_DEVERR_NONE.  Errors: ZS_ERR_CUDA. */
int zs_device_status(uint32_t* code, int32_t clear);

/* Self-test of the bounded wait used by the staged kernels: one block waits on
 * a barrier nothing will complete, gives up after limit_cycles SM cycles
 * (1 .. 2^32) and records ZS_DEVERR_SELFTEST.  Nothing else is touched.
 * Errors: ZS_ERR_INVALID for a limit out of range; ZS_ERR_CUDA. */
int zs_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/* ------------------------------------------------------------------ device operations */

/* Gradient accumulation without synchronisation ("Infra: Data Parallel",
 * section "Naive Data Parallelism", gradient-accumulation paragraph): for
 * every rank q and element i,
 *     acc[q][i] = bf16( fp32(acc[q][i]) + fp32(micro[q][i]) * scale )
 * with acc taken as +0 when `first` != 0 (acc is then write-only).  `scale`
 * is 1/n_micro for n_micro equal micro-batches whose losses are sample means.
 * acc, micro: ZS_RANK_FULL bf16, N_d pointers each; acc may equal micro
 * (in place). */
int zs_accumulate_grad(zs_plan_t plan, void* const* acc, const void* const* micro,
                       float scale, int32_t first, void* stream);

/* Reduce-Scatter with averaging (ZeRO section, ZeRO-1 paragraph; ZeRO-1 and
 * ZeRO-2 flow figures): for every element i of bucket `bucket` (or of every
 * bucket when bucket = -1), owned by rank r,
 *     out_r[i] = bf16( (sum over q = 0..N_d-1, ascending, of fp32 grads[q][i]) / N_d )
 * The sum starts from +0 and is fp32.
 *   grads_kind  ZS_RANK_FULL, or ZS_RANK_BUCKET (then bucket >= 0).
 *   out_kind    ZS_RANK_FULL: out[r] is rank r's full buffer and only its
 *               owned elements are written (ZeRO-1 keeps the full gradient
 *               buffer; out may be the same array of pointers as grads, in
 *               place);  ZS_SHARDED: out[0] is the sharded reduced gradient
 *               (ZeRO-2). */
int zs_reduce_scatter_mean(zs_plan_t plan, int32_t bucket, const void* const* grads,
                           int32_t grads_kind, void* const* out, int32_t out_kind, void* stream);

/* AdamW on shards (ZeRO section: AdamW is element-wise, each rank updates only
 * its own shard with its own moments): for every element i owned by `rank`
 * (every rank when rank = -1), with g = fp32(grad_r[i]) and the scalars of
 * zs_adamw_scalars, each operation rounded once in fp32 and none fused:
 *     p = master[i] * decay
 *     m[i] = beta1*m[i] + c1*g
 *     v[i] = beta2*v[i] + c2*(g*g)
 *     p = p - step_size * (m[i] / (sqrt(v[i]) / sqrt_bc2 + eps))
 *     master[i] = p;   param_r[i] = bf16(p)
 *   grad_kind   ZS_SHARDED, or ZS_RANK_FULL (ZeRO-1: rank r's reduced slice in
 *               its full gradient buffer).
 *   params_kind ZS_RANK_FULL: written into rank r's replica at its owned
 *               position (the source of an in-place all-gather);  ZS_SHARDED. */
int zs_adamw_shard_step(zs_plan_t plan, int32_t rank, const void* const* grad, int32_t grad_kind,
                        float* master, float* m, float* v, void* const* params,
                        int32_t params_kind, const zs_adamw_hparams* hp, int64_t step,
                        void* stream);

/* All-Gather of the updated bf16 parameters (ZeRO section, ZeRO-1 paragraph
 * and flow figure): every rank's replica receives every rank's shard.
 *   src_kind  ZS_SHARDED: src[0] is the sharded parameter array;
 *             ZS_RANK_FULL: in place, src must equal replicas and rank r's
 *             shard is read from its own replica.
 *   replicas  ZS_RANK_FULL, N_d pointers. */
int zs_all_gather(zs_plan_t plan, const void* const* src, int32_t src_kind,
                  void* const* replicas, void* stream);

/* FSDP2 layout conversions for one unit of an FSDP2 plan (see
 * zs_plan_create_fsdp2).  `params` holds one pointer per parameter of the unit,
 * in parameter order, each the parameter in its own (row-major, natural) layout
 * as bf16; `flat` is the unit's flat buffer of padded_u bf16 elements (rank-major,
 * e.g. a ZS_RANK_UNIT buffer, or a ZS_RANK_FULL buffer advanced to the unit's base).
 * zs_fsdp2_chunk_cat: params -> flat, padding rows written as zeros (building one
 *   rank's reduce-scatter input from its gradients).
 * zs_fsdp2_copy_out: flat -> params (after a gather: each rank's rows back into the
 *   full parameters).
 * Pointers must be 2-byte aligned; runs that share their 16-byte phase move 16
 * bytes per access.  Errors: ZS_ERR_INVALID (not an FSDP2 plan, bad unit, NULL or
 * misaligned pointer; nothing enqueued), ZS_ERR_CUDA. */
int zs_fsdp2_chunk_cat(zs_plan_t plan, int32_t unit, const void* const* params, void* flat, void* stream);
int zs_fsdp2_copy_out(zs_plan_t plan, int32_t unit, const void* flat, void* const* params, void* stream);

/* Naive data parallelism ("Infra: Data Parallel", section "Naive Data
 * Parallelism": every rank keeps a full replica of parameters, gradients and
 * optimizer state, all-reduces the gradients to their mean and applies the same
 * update; per-rank model-state memory 16 bytes per parameter, ~4 Psi bytes sent).
 * zs_all_reduce_mean: in place, every rank's buffer (ZS_RANK_FULL) gets
 *   bf16((sum over q ascending of fp32 grads[q][i]) / N_d) for every element of
 *   bucket `bucket` (-1: all).
 * zs_dp_step: the all-reduce and each rank's full AdamW in one pass: master, m,
 *   v are N_d full fp32 arrays (one per rank, padded_numel elements each, the
 *   rank's own replicated state); replicas[q] receives bf16 of rank q's master.
 *   Same arithmetic as zs_fused_step; every rank's copy ends bit-identical.
 * Errors: ZS_ERR_INVALID (before anything is enqueued), ZS_ERR_CUDA. */
int zs_all_reduce_mean(zs_plan_t plan, int32_t bucket, void* const* grads, void* stream);
int zs_dp_step(zs_plan_t plan, const void* const* grads, float* const* master, float* const* m,
               float* const* v, void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
               void* stream);

/* The three steps above in one pass over HBM: reduce-scatter with averaging,
 * AdamW on the shard, all-gather into every replica.  Results are bit-identical
 * to zs_reduce_scatter_mean + zs_adamw_shard_step + zs_all_gather (the reduced
 * gradient is rounded to bf16 before the update as there).
 * Gradient and replica buffers may also be pinned host memory (cudaHostAlloc /
 * cudaMallocHost, reachable from the device under unified addressing): the kernel
 * then reads or writes them over the host link directly, with no copy-engine
 * transfer (the register-streaming kernel is used for such calls).
 *   bucket      -1 = the whole flat space, else one bucket (the update is
 *               element-wise, so a bucket can be stepped as soon as its
 *               gradients are complete).
 * A range of at least 2^24 elements (device buffers, N_d of 2, 4, 8, 16 or
 * 32) is stepped by one persistent launch whose CTAs take their tiles in
 * order from a counter; a shorter range is stepped as a walk: cut at
 * multiples of 4 Mi elements, one launch per piece; the launches after the
 * first start on their own pieces while the previous one drains and complete
 * after it, so stream order holds at the call's end (pinned host buffers: one
 * launch, nothing cut).
 *   grads_kind  ZS_RANK_FULL, or ZS_RANK_BUCKET (bucket >= 0; ZeRO-2 staging).
 *   replicas    ZS_RANK_FULL; must not overlap grads. */
int zs_fused_step(zs_plan_t plan, int32_t bucket, const void* const* grads, int32_t grads_kind,
                  float* master, float* m, float* v, void* const* replicas,
                  const zs_adamw_hparams* hp, int64_t step, void* stream);

/* zs_fused_step with the last micro-batch's gradient accumulation done inside
 * the step ("Infra: Data Parallel", section "Naive Data Parallelism",
 * gradient-accumulation paragraph: the micro-batch gradients are summed, each
 * scaled, before the data-parallel reduction; ZeRO section for the rest).  For every element i of the range and
 * every rank q, rank q's gradient is
 *     g_q[i] = bf16( fp32(acc[q][i]) + fp32(micro[q][i]) * scale )
 * - exactly what zs_accumulate_grad(acc, micro, scale, first = 0) would store -
 * and the step then runs on g_q as zs_fused_step does.  The results (master, m,
 * v, replicas) are bit-identical to zs_accumulate_grad followed by
 * zs_fused_step on acc; acc and micro are only read (the accumulated gradient is
 * consumed by the step, not stored), which saves writing and re-reading it:
 * 24 + 6 N_d bytes per element against 24 + 10 N_d for the two calls.
 *   acc, micro  N_d pointers each, both of kind grads_kind (ZS_RANK_FULL, or
 *               ZS_RANK_BUCKET with bucket >= 0); acc holds the earlier
 *               micro-batches' sum (zs_accumulate_grad), micro the last
 *               micro-batch's gradients; either may be pinned host memory (the
 *               streaming kernel then runs, as in zs_fused_step).
 *   scale       finite; 1/n_micro for n_micro equal micro-batches.
 *   bucket, master, m, v, replicas, hp, step as in zs_fused_step; replicas must
 *               not overlap acc or micro.  Walked as zs_fused_step walks a short
 *               range, at every length.
 * Errors: ZS_ERR_INVALID (nothing enqueued), ZS_ERR_CUDA. */
int zs_fused_step_accumulate(zs_plan_t plan, int32_t bucket, const void* const* acc, const void* const* micro,
                             int32_t grads_kind, float scale, float* master, float* m, float* v,
                             void* const* replicas, const zs_adamw_hparams* hp, int64_t step, void* stream);

/* zs_fused_step for a list of buckets (ZS_RANK_FULL gradients) in the order
 * given - e.g. the buckets whose gradients became ready together, last layer
 * first.  Same results as calling zs_fused_step once per bucket, with the
 * argument checks, the pointer-kind queries and the per-call overhead paid
 * once.  The update is element-wise and the buckets are disjoint, so the
 * launches need no order among themselves: the list is walked as in
 * zs_fused_step (pieces of at most ~4 Mi elements, each launch starting while
 * the previous one drains; the first waits for everything enqueued before the
 * call, and the call's work completes in stream order).
 *   launch_mode  ZS_BUCKETS_ONE_WALK: listed buckets that touch are merged
 *                into one range (a run of neighbours, in either order) before
 *                the walk (when they merge into one range of at least 2^24
 *                elements, it is stepped as zs_fused_step steps a long range:
 *                one dynamic-order launch); disjoint runs shorter than 2^16 elements share
 *                persistent launches of a list kernel (128 runs per launch)
 *                instead of a launch each; where only the streaming kernel
 *                applies (host buffers, other rank counts) one launch per
 *                range.
 *                ZS_BUCKETS_PER_BUCKET: the buckets are walked one after
 *                another in the order given (a list of one bucket of at least
 *                2^24 elements: one dynamic-order launch), no launch spanning two buckets,
 *                as when each is stepped as soon as backward has made it
 *                ready; with a side_stream other than stream, the buckets at
 *                odd positions are walked on side_stream (which first waits
 *                for all work enqueued on stream); before returning, stream
 *                is made to wait for side_stream.  The two-stream form creates
 *                and releases two CUDA events (no device memory).
 *   side_stream  used by ZS_BUCKETS_PER_BUCKET only; NULL or equal to stream:
 *                one stream.
 * Errors: ZS_ERR_INVALID (bad or repeated bucket index, unknown launch_mode,
 * or any check of zs_fused_step; nothing enqueued), ZS_ERR_CUDA. */
#define ZS_BUCKETS_ONE_WALK 0
#define ZS_BUCKETS_PER_BUCKET 1
int zs_fused_step_buckets(zs_plan_t plan, int32_t n_buckets, const int32_t* buckets,
                          const void* const* grads, float* master, float* m, float* v,
                          void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                          int32_t launch_mode, void* stream, void* side_stream);

/* One rank's local share of the ZeRO-1/2 step when every data-parallel rank is
 * its own process on its own GPU ("Infra: Data Parallel", ZeRO section,
 * communication paragraphs and ZeRO-1/2 flow figures: the reduce-scatter hands
 * rank r every rank's gradients for the part of the bucket it owns, rank r
 * averages them and updates its own shard of the optimizer state, and the
 * all-gather then spreads the updated shards).  The exchanges are the caller's
 * collectives (an all-to-all of each bucket before this call, an all-gather of
 * the parameter shards after it); this call is the part between them: over
 * rank r's part of `bucket`, fold the N_d received gradient slices in
 * ascending rank order from +0, average, round to bf16, run AdamW on the
 * rank's own fp32 state and write the rank's bf16 parameter shard.  Results
 * equal rank r's shard of zs_fused_step bit for bit.
 *   rank         0 .. N_d-1, the calling rank.
 *   bucket       a bucket index, or -1 for the rank's whole shard (every unit).
 *   slices       N_d device pointers (16-byte aligned); slices[q] holds rank
 *                q's bf16 gradients for the elements rank r owns in the bucket,
 *                contiguous, in flat-index order: the receive buffer of an
 *                all-to-all in which every rank sends its bucket
 *                [begin, end), split by owner (zs_plan_bucket_rank_slice gives
 *                each owner's part).  For bucket -1: rank r's pieces of every
 *                unit back to back, in unit order.
 *   master, m, v rank r's own fp32 state, in its local layout: its shard of
 *                every unit, units in order (shard_numel_per_rank elements);
 *                the bucket's part starts at the unit's offset in that layout
 *                (sum of the earlier units' shard sizes) plus the part's offset
 *                in the rank's shard of the unit.
 *   param_shard  rank r's bf16 parameters in the same local layout (written).
 * Runs on `stream` (the staged kernel when the local offsets keep 16-byte
 * alignment, else the streaming kernel; the values are the same).
 * Errors: ZS_ERR_INVALID (bad plan, rank or bucket, a NULL or misaligned
 * pointer, bad hyper-parameters or step; nothing enqueued), ZS_ERR_CUDA. */
int zs_rank_shard_step(zs_plan_t plan, int32_t rank, int32_t bucket, const void* const* slices,
                       float* master, float* m, float* v, void* param_shard,
                       const zs_adamw_hparams* hp, int64_t step, void* stream);

/* zs_fused_step over the whole flat space with the gradients in HOST memory
 * (pinned for overlap): enqueues one host-to-device copy per rank into
 * dev_grads (ZS_RANK_FULL, caller-owned device staging), the fused step, and a
 * device-to-host copy of rank 0's updated replica into host_replica0 (may be
 * NULL to skip).  Same results as zs_fused_step. */
int zs_fused_step_host(zs_plan_t plan, const void* const* host_grads, void* const* dev_grads,
                       float* master, float* m, float* v, void* const* replicas,
                       const zs_adamw_hparams* hp, int64_t step, void* host_replica0,
                       void* stream);

/* ZeRO-3 gather of one unit (ZeRO section, ZeRO-3 paragraph and flow figure:
 * before forward, and again before backward, each rank borrows the unit's full
 * parameters): full[q][j] = shards[0][base_u + j] for every rank q and j in
 * [0, padded_u).
 *   shards  ZS_SHARDED bf16 parameter shards (1 pointer).
 *   full    ZS_RANK_UNIT, N_d pointers of padded_u elements. */
int zs_zero3_gather_unit(zs_plan_t plan, int32_t unit, const void* shards, void* const* full,
                         void* stream);

/* ZeRO-3 reduce-scatter with averaging of one unit's gradients fused with the
 * AdamW update of every rank's shard of that unit (same arithmetic as
 * zs_reduce_scatter_mean then zs_adamw_shard_step); no gather follows.
 *   grads   ZS_RANK_UNIT, N_d pointers of padded_u elements (each rank's
 *           backward gradients for the unit).
 *   shards  ZS_SHARDED bf16 parameter shards, updated in place. */
int zs_zero3_rs_step_unit(zs_plan_t plan, int32_t unit, const void* const* grads, float* master,
                          float* m, float* v, void* shards, const zs_adamw_hparams* hp,
                          int64_t step, void* stream);

/* Sharded checkpoint ("Infra: Data Parallel", FSDP section, subsection
 * "Checkpoint": each rank writes the shards it owns plus the metadata needed to
 * restore them; loading follows the target layout, so the rank count may differ;
 * optimizer state is saved with the weights; FSDP1 and FSDP2 both support it).
 * zs_checkpoint_save writes dir/meta.txt (format tag, N_d, step, layout, per
 * parameter its element count, dim-0 rows and unit, per unit numel/padded/shard)
 * and one file per simulated rank, dir/rank-NNNNN.bin, holding that rank's shard
 * of the bf16 parameters, then master, m and v (each the rank's piece of every
 * unit, units in order).  zs_checkpoint_load reads such a directory into the
 * ZS_SHARDED arrays of `plan`, which must list the same parameters (element counts
 * and dim-0 sizes) but may use another N_d, another unit grouping and the other
 * layout: every element keeps its place in its parameter, the target's padding is
 * zeroed.  `dir` must exist.  `step` is the number of optimizer steps taken
 * (>= 0); load returns the saved count and rejects a meta.txt whose step is
 * missing or negative.  Arrays are ZS_SHARDED device arrays of plan's
 * padded_numel elements.  Both calls first synchronise `stream`, then move the
 * data on up to 16 worker threads, each with its own non-blocking stream and two
 * 16 MiB pinned host staging buffers (host memory, freed before returning; no
 * device memory), overlapping file I/O with the copies; they return after the
 * data is in place.
 * Errors: ZS_ERR_INVALID (NULL argument, I/O failure, a checkpoint of another
 * model or a malformed one: nothing is written to the device before the metadata
 * and file sizes are checked), ZS_ERR_CUDA. */
int zs_checkpoint_save(zs_plan_t plan, const char* dir, const void* shards, const float* master,
                       const float* m, const float* v, int64_t step, void* stream);
int zs_checkpoint_load(zs_plan_t plan, const char* dir, void* shards, float* master, float* m,
                       float* v, int64_t* step, void* stream);

/* ZeRO-2 step fed from host memory ("Infra: Data Parallel", ZeRO section,
 * ZeRO-2 paragraph and flow figure: gradients are reduced bucket by bucket and
 * no rank keeps a full gradient buffer).  For each bucket, in descending order:
 * one host-to-device copy per rank of the bucket's gradients into one slot of a
 * two-slot staging ring (copy_stream), the fused step on that bucket (stream),
 * which frees the slot, and, when host_replica0 is given, a device-to-host copy
 * of the bucket's slice of rank 0's updated replica (d2h_stream, or copy_stream
 * when NULL).  Copies of the next bucket overlap the update of this one.  Same
 * results as zs_fused_step over the whole flat space.  `stream` waits for all
 * of it at the end; the caller synchronises before reading host_replica0.
 *   host_grads     N_d host pointers (pinned for asynchronous copies), each
 *                  holding the rank's padded_numel gradients.
 *   staging        2 * N_d device pointers; slot k, rank q at [k*N_d + q], each
 *                  at least staging_elems >= the largest bucket's elements.
 *   replicas       ZS_RANK_FULL; master/m/v ZS_SHARDED.
 * Errors: ZS_ERR_INVALID (before anything is enqueued), ZS_ERR_CUDA. */
int zs_zero2_step_host(zs_plan_t plan, const void* const* host_grads, void* const* staging,
                       int64_t staging_elems, float* master, float* m, float* v, void* const* replicas,
                       const zs_adamw_hparams* hp, int64_t step, void* host_replica0, void* stream,
                       void* copy_stream, void* d2h_stream);

/* zs_zero2_step_host without caller-provided staging: a variant for callers
 * that cannot allocate device memory when they run the step (a framework that
 * owns all device memory through its own pool, a latency-critical thread that
 * must not pay cudaMalloc's implicit device synchronisation, a plug-in handed only
 * stream and buffer pointers).  The pages have no counterpart: this is a
 * property of the library, not of the method.
 * The two-slot staging ring is a fixed device array inside the library image,
 * ZS_NOALLOC_STAGING_BYTES (32 MiB) per GPU, held by every GPU that loads the
 * library until the process exits; the call itself allocates nothing (no
 * cudaMalloc, no events).  The first call on a device looks up the array's device
 * address with that device current (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture begins.  Copies, updates and the
 * copy-back of rank 0's replica all run in order on `stream` (no overlap).
 * Every call on a device shares the one array and leaves its last contents in
 * it; nothing in it has to start at zero because each bucket is copied in before
 * it is read.  Calls whose work overlaps on the GPU (other streams, other host
 * threads) race on the array: serialise them.
 * Same arguments and results as zs_zero2_step_host minus the staging.  Plans
 * whose 2 x N_d x largest bucket (rounded up to 8 elements) x 2 bytes exceed
 * ZS_NOALLOC_STAGING_BYTES are rejected with ZS_ERR_INVALID and a message that
 * states the limit.  Errors: ZS_ERR_INVALID (before anything is enqueued),
 * ZS_ERR_CUDA. */
#define ZS_NOALLOC_STAGING_BYTES (32ll << 20)
int zs_zero2_step_host_noalloc(zs_plan_t plan, const void* const* host_grads, float* master, float* m,
                               float* v, void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                               void* host_replica0, void* stream);

/* One ZeRO-3 step over every unit (ZeRO section, ZeRO-3 paragraph and flow
 * figure; FSDP2 subsection for reshard_after_forward), scheduled on two streams:
 * forward in unit order gathers each unit into a pool slot; backward in reverse
 * order gathers it again (only when reshard_after_forward != 0), then reduce-
 * scatters the unit's gradients with averaging and updates every rank's shard
 * (zs_zero3_rs_step_unit).  Gathers and updates run on side_stream; main_stream
 * (the compute stream, where a model's forward/backward would run) only waits
 * for each gather and releases the slot, and at the end waits for the last
 * update.  With two slots the next unit's gather overlaps the current unit's use;
 * in backward the next unit's gather is issued before the current unit's
 * reduce-scatter and update (backward prefetch).
 * side_stream may equal main_stream (everything serialised in stream order, no
 * event used; same results).
 *   shards       ZS_SHARDED bf16 parameter shards (updated in place).
 *   master,m,v   ZS_SHARDED fp32.
 *   unit_grads   n_units * N_d pointers; unit u, rank q at [u*N_d + q], each
 *                ZS_RANK_UNIT (padded_u elements).  Entries may repeat.
 *   pool         pool_slots * N_d pointers; slot k, rank q at [k*N_d + q], each
 *                at least the largest unit's padded size.  pool_slots >= 2 (1 for
 *                a single unit) with reshard_after_forward, >= n_units without;
 *                afterwards each slot holds the last unit gathered into it.
 * With two streams the call creates and releases CUDA events (no device memory).
 * Errors: ZS_ERR_INVALID (checked before anything is enqueued), ZS_ERR_CUDA. */
int zs_zero3_step(zs_plan_t plan, void* shards, float* master, float* m, float* v,
                  const void* const* unit_grads, void* const* pool, int32_t pool_slots,
                  int32_t reshard_after_forward, const zs_adamw_hparams* hp, int64_t step,
                  void* main_stream, void* side_stream);

#ifdef __cplusplus
}
#endif

#endif /* ZS_H */
