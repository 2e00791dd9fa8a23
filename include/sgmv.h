/*
 * sgmv.h -- C ABI of the GB300 (sm_103a) segmented-gather LoRA library (libsgmv_gb300.so).
 *
 * The operation ("Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The
 * Heterogeneous Batching Bottleneck: Why Standard Serving Stalls", equation
 *     y_i = x_i W0 + (alpha/r) x_i A_{k(i)} B_{k(i)};
 * section "The SGMV Mathematical Formulation": tokens grouped into contiguous segments
 * [s_i, s_{i+1}), each bound to one adapter through an array of weight pointers; section
 * "Mathematical Modeling: Throughput Scaling and Kernel Launch Bounds", part 2: one launch for
 * all A projections ("shrink") and one for all B projections ("expand") per layer):
 *
 *   for each segment i in [0, num_segments), k = seg_adapter[i], rows t in
 *   [seg_starts[i], seg_starts[i+1]):
 *       v[t]  = x[t] . A_k[layer_idx]                  (shrink, h_in -> r)
 *       y[t] += scale * v[t] . B_k[layer_idx]          (expand, r -> h_out)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every pointer argument except the host pointer of sgmv_get_error() is DEVICE
 *   memory owned by the caller, on the current CUDA device: the pointer arrays A_ptrs/B_ptrs
 *   themselves, the segment table and all tensors.  The library allocates nothing per call
 *   and keeps no reference after the call is enqueued.
 * Layout.  Row-major, contiguous.
 *   x   [M][h_in]            activations (M >= seg_starts[num_segments]).
 *   y   [M][h_out]           holds the base output x W0 on entry; the LoRA term is added.
 *   v   [M][r]  fp32         shrink output / expand input.
 *   A_ptrs[k] -> adapter k's block [L][h_in][r];   layer l starts at element l*h_in*r.
 *   B_ptrs[k] -> adapter k's block [L][r][h_out];  layer l starts at element l*r*h_out.
 *   seg_starts [num_segments+1] int32, non-decreasing; seg_adapter [num_segments] int32.
 *   x, y, A and B share one element type (dtype); accumulation is fp32 throughout and y is
 *   rounded (to nearest even) once, at the store.
 * Segments.  Rows outside [seg_starts[0], seg_starts[num_segments]) are never read or
 *   written.  A segment with seg_starts[i+1] <= seg_starts[i] is empty.  A negative adapter
 *   id means "no adapter": those rows are left unchanged (shrink leaves their v untouched).
 *   Several segments may use the same adapter; its weights are then streamed once for all of
 *   them.  A row must not belong to two segments.
 * Alignment.  x, y, v, every A_ptrs[k]/B_ptrs[k] block and the pointer arrays must be 16-byte
 *   aligned; h_in and h_out must be multiples of 8; r must be 8, 16, 32 or 64.
 * Asynchrony.  Work is enqueued on `stream` and the call returns without synchronising, so it
 *   can be captured into a CUDA graph (after one uncaptured call with the same dtype/rank on
 *   the device, which sets the kernels' attributes).  Calls on one stream are ordered; calls
 *   on different streams that write the same rows race.
 * Errors.  Host-checkable violations return a negative status and enqueue nothing.  Defects
 *   that only the device can see are not checked on the fast path and are undefined behaviour
 *   there (typically a memory fault): decreasing offsets and adapter ids past the pool (run
 *   sgmv_validate() on untrusted tables), a null or misaligned A_ptrs[k] / B_ptrs[k] of an
 *   adapter the table uses (sgmv_validate_pointers()), and a layer_idx at or past the number
 *   of layers L of the adapter blocks (the library is never told L; the caller checks it).
 *   Every device-side wait is bounded; a wait that runs out sets the library's device error
 *   word, which sgmv_get_error() reads (SGMV_ETIMEOUT), and the kernel returns without
 *   hanging.
 */
#ifndef SGMV_GB300_H
#define SGMV_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; 0 is the legacy default stream. */
typedef struct CUstream_st *sgmv_stream_t;

typedef enum {
    SGMV_F32 = 0,   /* float32                     */
    SGMV_F16 = 1,   /* IEEE binary16               */
    SGMV_BF16 = 2   /* bfloat16                    */
} sgmv_dtype_t;

typedef enum {
    SGMV_OK = 0,
    SGMV_EINVAL = -1,        /* null pointer, negative size, bad enum                       */
    SGMV_EALIGN = -2,        /* pointer not 16-byte aligned, h_in/h_out not multiples of 8  */
    SGMV_EUNSUPPORTED = -3,  /* rank not in {8,16,32,64}, sizes past the documented limits  */
    SGMV_ECUDA = -4,         /* a CUDA runtime call or launch failed                        */
    SGMV_ETIMEOUT = -5,      /* a bounded device-side wait ran out (see sgmv_get_error)     */
    SGMV_EPLAN = -6,         /* a planned call read an invalid plan (see sgmv_get_error)    */
    SGMV_ENOSPACE = -7,      /* the adapter pool has too few free slots for the batch       */
    SGMV_EBUSY = -8          /* the adapter's slot is read by a batch not yet released      */
} sgmv_status_t;

/* Largest num_segments one call accepts (the segment table is staged on chip). */
#define SGMV_MAX_SEGMENTS 4096
/* Largest h_in and h_out one call accepts. */
#define SGMV_MAX_HIDDEN 65536
/* Largest row stride (elements) of x or y that the _strided entry points accept. */
#define SGMV_MAX_LD (1 << 24)
/* Largest number of projections of one lora_apply_multi call. */
#define SGMV_MAX_PROJECTIONS 4
/* Largest row capacity (max_rows) of lora_apply_static_plan. */
#define SGMV_STATIC_PLAN_MAX_ROWS 65536

/*
 * lora_apply -- the fused path: y[t] += scale * (x[t] . A_k) . B_k for every segment row.
 * Source: the y_i equation above (with scale = alpha/r) and the SGMV segment formulation; the
 * fusion keeps the r-wide intermediate on chip, so one launch replaces the two per layer of
 * section "Mathematical Modeling ...", part 2.
 *   y            in/out  [M][h_out], dtype
 *   x            in      [M][h_in],  dtype
 *   A_ptrs       in      [num_adapters] device pointers to [L][h_in][r] blocks, dtype
 *   B_ptrs       in      [num_adapters] device pointers to [L][r][h_out] blocks, dtype
 *   seg_starts   in      [num_segments+1] int32
 *   seg_adapter  in      [num_segments] int32 (negative: no adapter; may be null when
 *                        num_segments == 0)
 *   num_segments         0 <= num_segments <= SGMV_MAX_SEGMENTS (0: returns SGMV_OK, no-op)
 *   layer_idx            0 <= layer_idx < L (the layer count of every adapter block the
 *                        table uses; only the sign is checked), selects the layer
 *   h_in, h_out          multiples of 8, <= SGMV_MAX_HIDDEN
 *   r                    8, 16, 32 or 64
 *   scale                alpha / r, applied in fp32 to the intermediate before the expand
 *   dtype                element type of x, y, A and B
 *   stream               CUDA stream the work is enqueued on
 * Execution: one kernel launch.  For fp16 / bf16 and r >= 16, an adapter group (all rows of
 * one adapter in the call) runs on the tensor cores (tcgen05.mma; section "Hardware-Level
 * Optimizations in SGMV": tensor-core tiles for long segments) when it has at least 64 rows
 * (half a 128-row tile) and the CUDA-core path would re-read at least 32 MB of its weights
 * (ceil(rows / 4) x the bytes of A_k and B_k); there the intermediate is kept as a 16-bit high
 * part plus a 16-bit low part, about 16 significant bits.  Every other group runs on the CUDA
 * cores in fp32.
 * Returns SGMV_OK or a negative sgmv_status_t (nothing enqueued on a negative status other
 * than SGMV_ECUDA from the launch itself).
 */
int lora_apply(void *y, const void *x, const void *const *A_ptrs, const void *const *B_ptrs,
               const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
               int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
               sgmv_dtype_t dtype, sgmv_stream_t stream);

/* Flags of lora_apply_ex. */
#define SGMV_OVERLAP_PRIOR 1u
#define SGMV_NO_TENSOR_CORES 2u
#define SGMV_TENSOR_CORES_ALWAYS 4u
#define SGMV_LONG_BATCH 8u
#define SGMV_DENSE_GRID 16u

/*
 * lora_apply_ex -- lora_apply with launch flags.
 *   flags = 0: identical to lora_apply.
 *   flags = SGMV_OVERLAP_PRIOR: the kernel is launched as a programmatic dependent of the
 *     kernel enqueued before it on `stream` (CUDA programmatic dependent launch).  It may start,
 *     read the segment table and the pointer arrays and stream adapter weights while that
 *     previous kernel is still running; it waits for the previous kernel to complete before it
 *     reads x or y and before it writes y.  Use it for back-to-back layer calls (for example a
 *     CUDA graph of a layer sweep): the weight streaming of one call then overlaps the tail of
 *     the previous one.  Precondition: the immediately preceding kernel on the stream does not
 *     write the segment table, A_ptrs/B_ptrs or any adapter weights.  The pages describe no
 *     counterpart; it is launch mechanics for the same operation.
 *   flags |= SGMV_NO_TENSOR_CORES: every adapter group runs on the CUDA cores, however many
 *     rows it has (the results agree within rounding; used to check one path against the
 *     other and by callers that know a batch holds only decode rows).
 *   flags |= SGMV_TENSOR_CORES_ALWAYS: every adapter group of at least 64 rows runs on the
 *     tensor cores, without the cost rule described under lora_apply (fp16 / bf16, r >= 16).
 *     Not combinable with SGMV_NO_TENSOR_CORES (SGMV_EINVAL).
 *   flags |= SGMV_LONG_BATCH: the caller declares a long call (a prefill batch, or adapter
 *     groups of hundreds of rows).  The kernel then runs one CTA per SM with up to 227 KB of
 *     shared memory instead of two co-resident CTAs of 112 KB: deeper rings of weight and
 *     activation stages for both the CUDA-core and the tensor-core paths.  The results agree
 *     with a launch without the flag within rounding (the routing of groups and the chunking
 *     of h_in are the same; the grid, and with it the split of work over CTAs, may differ).
 *     With SGMV_OVERLAP_PRIOR the next call's CTAs can only start where this call's CTAs have
 *     left, so the overlap of short calls is lost: do not use it for decode batches.
 *   flags |= SGMV_DENSE_GRID: the caller declares a decode batch with many work items (many
 *     rows spread over many adapter groups, for example 256 tokens over 60 or more adapters).
 *     The kernel then runs two CTAs of this call per SM in the default geometry instead of
 *     one, so that each SM streams two items at once; the next kernel of the stream can start
 *     only as this call's CTAs finish, so the overlap that hides a short call's start-up is
 *     lost.  Measured on GB300 (256 tokens, h = 4096, r = 16): 256 ids over 1024 adapters
 *     25.7 -> 17.3 us per chained call, Zipf-drawn ids 16.0 -> 12.0 us; 64 one-token segments
 *     of 64 adapters 6.0 -> 9.2 us (do not use it there).  Ignored with SGMV_LONG_BATCH (whose
 *     CTAs take a whole SM).  The results agree with a launch without the flag within
 *     rounding (the split of work over CTAs differs).
 * Other arguments, layout and errors: as for lora_apply (SGMV_EINVAL for unknown flags).
 */
int lora_apply_ex(void *y, const void *x, const void *const *A_ptrs, const void *const *B_ptrs,
                  const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                  int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
                  sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * lora_apply_strided -- lora_apply_ex on x and y whose rows are ldx and ldy elements apart:
 * row t of x is x + t * ldx (its first h_in elements are read), row t of y is y + t * ldy (its
 * first h_out elements are read and written; the elements past h_out in a row are never
 * touched).  This lets the delta apply to column slices of wider activations, for example the
 * q, k or v part of a fused projection output, in place.  The pages describe dense [M][h]
 * activations; the row stride is the common leading-dimension generalisation.
 *   ldx   h_in <= ldx <= SGMV_MAX_LD, a multiple of 8 (SGMV_EINVAL if below h_in,
 *         SGMV_EALIGN if not a multiple of 8, SGMV_EUNSUPPORTED above SGMV_MAX_LD)
 *   ldy   the same with h_out
 * Other arguments, layout, flags and errors: as for lora_apply_ex.  lora_apply_ex is this call
 * with ldx = h_in and ldy = h_out.
 */
int lora_apply_strided(void *y, int32_t ldy, const void *x, int32_t ldx,
                       const void *const *A_ptrs, const void *const *B_ptrs,
                       const int32_t *seg_starts, const int32_t *seg_adapter,
                       int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                       int32_t r, float scale, sgmv_dtype_t dtype, uint32_t flags,
                       sgmv_stream_t stream);

/*
 * sgmv_shrink -- v[t] = x[t] . A_k for every segment row (overwrites those rows of v; other
 * rows of v are not written).  Source: the first factor x_i A_{k(i)} of the y_i equation and
 * the "one launch for all A projections" of section "Mathematical Modeling ...", part 2.
 *   v      out  [M][r] float32
 *   x      in   [M][h_in] dtype;  A_ptrs, seg_starts, seg_adapter, num_segments, layer_idx,
 *   h_in, r, dtype, stream: as for lora_apply.
 */
int sgmv_shrink(float *v, const void *x, const void *const *A_ptrs, const int32_t *seg_starts,
                const int32_t *seg_adapter, int32_t num_segments, int32_t layer_idx,
                int32_t h_in, int32_t r, sgmv_dtype_t dtype, sgmv_stream_t stream);

/*
 * sgmv_shrink_ex -- sgmv_shrink with the flags of lora_apply_ex (SGMV_OVERLAP_PRIOR,
 * SGMV_NO_TENSOR_CORES, SGMV_TENSOR_CORES_ALWAYS; SGMV_EINVAL for others).  As in lora_apply,
 * fp16 / bf16 groups of at least 64 rows whose CUDA-core items would re-read at least 32 MB of
 * A_k run on the tensor cores (v is then exact up to fp32 accumulation order).
 */
int sgmv_shrink_ex(float *v, const void *x, const void *const *A_ptrs,
                   const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                   int32_t layer_idx, int32_t h_in, int32_t r, sgmv_dtype_t dtype,
                   uint32_t flags, sgmv_stream_t stream);

/*
 * sgmv_shrink_strided -- sgmv_shrink_ex with x rows ldx elements apart (ldx as for
 * lora_apply_strided; v stays dense [M][r]).
 */
int sgmv_shrink_strided(float *v, const void *x, int32_t ldx, const void *const *A_ptrs,
                        const int32_t *seg_starts, const int32_t *seg_adapter,
                        int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t r,
                        sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * sgmv_expand -- y[t] += scale * v[t] . B_k for every segment row.  Source: the second factor
 * (x_i A_k) B_k of the y_i equation, times alpha/r, and the "one launch for all B projections"
 * of section "Mathematical Modeling ...", part 2.
 *   y      in/out [M][h_out] dtype
 *   v      in     [M][r] float32 (as written by sgmv_shrink)
 *   B_ptrs, seg_starts, seg_adapter, num_segments, layer_idx, r, h_out, scale, dtype, stream:
 *   as for lora_apply.
 */
int sgmv_expand(void *y, const float *v, const void *const *B_ptrs, const int32_t *seg_starts,
                const int32_t *seg_adapter, int32_t num_segments, int32_t layer_idx, int32_t r,
                int32_t h_out, float scale, sgmv_dtype_t dtype, sgmv_stream_t stream);

/*
 * sgmv_expand_ex -- sgmv_expand with the flags of lora_apply_ex.  On the tensor cores (same
 * routing rule, weights = B_k) scale * v enters the MMA as a 16-bit high part plus a 16-bit low
 * part (about 16 significant bits), as in the fused path.
 */
int sgmv_expand_ex(void *y, const float *v, const void *const *B_ptrs,
                   const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                   int32_t layer_idx, int32_t r, int32_t h_out, float scale, sgmv_dtype_t dtype,
                   uint32_t flags, sgmv_stream_t stream);

/*
 * sgmv_expand_strided -- sgmv_expand_ex with y rows ldy elements apart (ldy as for
 * lora_apply_strided; the elements past h_out in a row are never touched).
 */
int sgmv_expand_strided(void *y, int32_t ldy, const float *v, const void *const *B_ptrs,
                        const int32_t *seg_starts, const int32_t *seg_adapter,
                        int32_t num_segments, int32_t layer_idx, int32_t r, int32_t h_out,
                        float scale, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * ---- Plans: the segment table grouped once, reused by every layer and projection ----------
 * Source: section "Mathematical Modeling: Throughput Scaling and Kernel Launch Bounds", part 2
 * (every layer's adapter work in a fixed number of launches) and section "Hardware-Level
 * Optimizations in SGMV" (segment descriptors pre-sorted by adapter so that each adapter's
 * weights are streamed once).  The grouping of a batch's table by adapter does not depend on
 * the layer or on the projection; the unplanned calls above redo it in every CTA of every call.
 * sgmv_plan does it once, on the device, into a buffer the caller owns; the *_planned calls and
 * lora_apply_multi read it instead of the table.
 *
 * Plan contents (int32 words; the buffer is opaque to callers but its layout is fixed):
 * a 16-word header (magic, status, num_segments, groups G, rows listed, max_rows), the group
 * row offsets [num_segments + 1], the group adapters [num_segments] and the row list
 * [max_rows].  Groups are the distinct adapter ids >= 0 of the non-empty segments, in the
 * order of their first segment; a group's rows are its segments' rows, segment after segment.
 * Negative ids and empty segments are dropped (their rows are never touched).
 */

/* Bytes of a plan for a table of num_segments segments holding at most max_rows rows (0 for
 * negative sizes or num_segments > SGMV_MAX_SEGMENTS). */
size_t sgmv_plan_size(int32_t num_segments, int32_t max_rows);

/*
 * sgmv_plan -- groups the device segment table into `plan` (one kernel launch of one CTA,
 * asynchronous on `stream`).
 *   seg_starts, seg_adapter  in   device table as for lora_apply (validate untrusted tables
 *                                 first: decreasing offsets count as empty segments here)
 *   num_segments                  0 <= num_segments <= SGMV_MAX_SEGMENTS
 *   max_rows                      capacity of the row list (>= the rows of the table that have
 *                                 an adapter; the caller knows M and passes it)
 *   plan                     out  device buffer of plan_bytes >= sgmv_plan_size(), 16-byte
 *                                 aligned, owned by the caller; valid until overwritten
 * A table with more than max_rows rows yields a plan marked invalid (status word 1): every
 * planned call that reads it returns without touching y or v and sets the library's device
 * error word to SGMV_EPLAN.  Returns SGMV_OK, SGMV_EINVAL (null pointers, negative sizes,
 * plan_bytes too small), SGMV_EALIGN, SGMV_EUNSUPPORTED or SGMV_ECUDA.
 * Ordering: a planned call launched with SGMV_OVERLAP_PRIOR reads the plan before it waits for
 * the kernel enqueued just before it, so that kernel must not be the sgmv_plan that writes the
 * plan (the same rule as for the segment table); without the flag any order on one stream is
 * fine.
 */
int sgmv_plan(const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
              int32_t max_rows, void *plan, size_t plan_bytes, sgmv_stream_t stream);

/*
 * lora_apply_planned -- lora_apply_strided with the segment table replaced by a plan.
 *   plan           in   from sgmv_plan (device, 16-byte aligned)
 *   num_segments        the num_segments the plan was built with (its capacity; checked
 *                       against the plan on the device: a mismatch is SGMV_EPLAN)
 * Other arguments, flags, layout and errors: as for lora_apply_strided (x and y rows ldx and
 * ldy elements apart; ldx = h_in and ldy = h_out for dense activations).  The results equal
 * the unplanned call's within rounding (the same routing rule and chunking; the rows of a group
 * are visited in the plan's order).
 */
int lora_apply_planned(void *y, int32_t ldy, const void *x, int32_t ldx,
                       const void *const *A_ptrs, const void *const *B_ptrs, const void *plan,
                       int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                       int32_t r, float scale, sgmv_dtype_t dtype, uint32_t flags,
                       sgmv_stream_t stream);

/* sgmv_shrink_strided with a plan (arguments as for lora_apply_planned). */
int sgmv_shrink_planned(float *v, const void *x, int32_t ldx, const void *const *A_ptrs,
                        const void *plan, int32_t num_segments, int32_t layer_idx, int32_t h_in,
                        int32_t r, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/* sgmv_expand_strided with a plan (arguments as for lora_apply_planned). */
int sgmv_expand_planned(void *y, int32_t ldy, const float *v, const void *const *B_ptrs,
                        const void *plan, int32_t num_segments, int32_t layer_idx, int32_t r,
                        int32_t h_out, float scale, sgmv_dtype_t dtype, uint32_t flags,
                        sgmv_stream_t stream);

/* One projection of lora_apply_multi: the arguments of lora_apply_planned that differ between
 * projections (device pointers; ldx / ldy in elements). */
typedef struct {
    void *y;
    const void *x;
    const void *const *A_ptrs;
    const void *const *B_ptrs;
    int32_t ldy, ldx;
    int32_t h_in, h_out;
    float scale;
    int32_t reserved;  /* 0 */
} sgmv_projection_t;

/*
 * lora_apply_multi -- the fused LoRA term of up to SGMV_MAX_PROJECTIONS projections of one
 * layer (for example q, k and v of an attention block, or gate and up of an MLP) in ONE
 * kernel launch over one plan: proj[q] gets y_q[t] += scale_q * (x_q[t] . A_{q,k}) . B_{q,k}.
 * Each projection has its own x, y, weights, h_in, h_out and scale; all share the plan (the
 * batch), the layer, the rank r and the element type.  The grid is divided between the
 * projections in proportion to an estimate of their bytes.  proj is a HOST array of num_proj
 * entries, read during the call.  Projections must not write overlapping y rows.
 * Flags, layout and errors as for lora_apply_planned (SGMV_EUNSUPPORTED when num_proj >
 * SGMV_MAX_PROJECTIONS).  Each projection's result equals lora_apply_planned's on its own
 * within rounding.
 */
int lora_apply_multi(const sgmv_projection_t *proj, int32_t num_proj, const void *plan,
                     int32_t num_segments, int32_t layer_idx, int32_t r, sgmv_dtype_t dtype,
                     uint32_t flags, sgmv_stream_t stream);

/*
 * lora_apply_base -- the base projection and the LoRA term in one output pass:
 *     y[t] = x[t] . W0^T + scale * (x[t] . A_k) . B_k   rows t of segments with adapter k >= 0
 *     y[t] = x[t] . W0^T                                 every other row t < M
 * Source: "Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The Heterogeneous
 * Batching Bottleneck": the y_i equation's two terms, and that section's figure in which the
 * base GEMM feeds the fused SGMV kernel; here the LoRA term is added in the base GEMM's
 * epilogue, so y is written once (no read-modify-write of a base output).
 *   y        [M][ldy] output, written (not accumulated) for every row < M, columns < h_out
 *   x        [M][ldx] input rows
 *   M        rows of x and y (segment rows must lie in [0, M))
 *   W0       [h_out][ldw] base weight, one row per output feature (a linear layer's weight:
 *            the equation's x_i W0 is sum_j x[t][j] * W0[n][j])
 *   A_ptrs, B_ptrs, seg_starts, seg_adapter, num_segments, layer_idx, h_in, h_out, r, scale
 *            as for lora_apply (num_segments = 0: y = x . W0^T only)
 *   v_work   caller-owned fp32 workspace of M * r floats, 16-byte aligned (the shrink writes
 *            v = x . A_k there for the rows of segments with an adapter); may be NULL when
 *            num_segments == 0
 *   flags    passed to the shrink, which sends adapter groups of 64 rows or more to its
 *            tensor role unless SGMV_NO_TENSOR_CORES is set (SGMV_OVERLAP_PRIOR also makes the
 *            GEMM wait for the previous kernel of the stream before reading x)
 * Enqueues two kernels: sgmv_shrink_strided into v_work, then the GEMM (tcgen05, 128 x 256
 * output tiles, one CTA per SM), which starts its main loop while the shrink runs and waits
 * for it only before reading v.  Types: SGMV_F16 and SGMV_BF16 (SGMV_F32 -> SGMV_EUNSUPPORTED).
 * Layout rules as for lora_apply_strided (h_in, h_out, ldx, ldy, ldw multiples of 8; y, x, W0,
 * v_work 16-byte aligned).  Errors as for lora_apply; nothing is enqueued on a host-checked
 * error.  The device error word reports SGMV_ETIMEOUT if a bounded wait of either kernel
 * runs out.
 */
int lora_apply_base(void *y, int32_t ldy, const void *x, int32_t ldx, int32_t M, const void *W0,
                    int32_t ldw, const void *const *A_ptrs, const void *const *B_ptrs,
                    const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                    int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
                    float *v_work, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * lora_apply_static_plan -- lora_apply_planned for callers that cannot allocate device memory:
 * the library builds the plan itself (sgmv_plan) into a fixed array inside the library
 * instead of a caller-provided buffer, then applies it; the caller passes only inputs and
 * outputs.  The pages describe no counterpart: it is a deployment variant.  Callers in this
 * position are, for example, an inference runtime that reserves all device memory at start-up
 * through its own allocator and forbids cudaMalloc afterwards (a fixed memory budget, no
 * fragmentation), or a plugin interface that gives an operator no way to request a workspace.
 *   seg_starts, seg_adapter, num_segments  the device table, as for lora_apply
 *   max_rows       the plan's row capacity (>= the rows of the table that have an adapter)
 *   other arguments as for lora_apply_planned (ldx / ldy as for lora_apply_strided)
 * Limits: num_segments <= SGMV_MAX_SEGMENTS and max_rows <= SGMV_STATIC_PLAN_MAX_ROWS, else
 * SGMV_EUNSUPPORTED.  The array holds one plan of that size (about 295 KB), is created on every
 * device that loads the library and stays there until the process exits.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, once per device); make
 * that first call before any stream capture.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 * Sharing: every call, on every stream, uses the same array, which keeps the last call's plan
 * (the plan kernel rewrites every word the apply kernel reads, so nothing needs clearing).
 * Calls that overlap on the GPU -- on two streams, or two host threads -- race on it: order
 * them.  SGMV_OVERLAP_PRIOR is rejected (SGMV_EINVAL): the apply kernel must wait for the
 * plan kernel enqueued just before it.  Errors otherwise as for sgmv_plan and
 * lora_apply_planned; nothing is enqueued on a host-checked error.
 */
int lora_apply_static_plan(void *y, int32_t ldy, const void *x, int32_t ldx,
                           const void *const *A_ptrs, const void *const *B_ptrs,
                           const int32_t *seg_starts, const int32_t *seg_adapter,
                           int32_t num_segments, int32_t max_rows, int32_t layer_idx,
                           int32_t h_in, int32_t h_out, int32_t r, float scale,
                           sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * lora_apply_ranked -- the fused LoRA term with a rank and a scale of its own for every
 * adapter: y[t] += adapter_scale[k] * (x[t] . A_k) . B_k, where adapter k has rank
 * r_k = adapter_rank[k] and its blocks are A_k [L][h_in][r_k] and B_k [L][r_k][h_out]
 * (row-major; layer l at l*h_in*r_k and l*r_k*h_out).  Source: the y_i equation of section
 * "The Heterogeneous Batching Bottleneck" with alpha/r taken per adapter, and section
 * "Operational Checklist" (rank standardisation): a batch can hold adapters of several ranks,
 * and each is read at its own size, not padded.
 *   adapter_rank   in   device int32 [num_adapters]: r_k, a multiple of 8 in [8, r_max].  An
 *                       entry outside that set makes its adapter a no-op (its rows are left
 *                       unchanged): the kernels never read more of a block than its entry
 *                       declares.
 *   adapter_scale  in   device float [num_adapters]: the factor of adapter k's term (alpha_k /
 *                       r_k in the equation)
 *   seg_starts, seg_adapter  the table (as for lora_apply), or null when `plan` is given
 *   plan           in   a plan from sgmv_plan (as for lora_apply_planned), or null
 *   r_max          8, 16, 32 or 64: the largest rank the call may meet (the kernels' capacity)
 * Other arguments, flags, layout and errors: as for lora_apply_strided.  With every rank equal
 * to r_max and every scale equal to `scale` the result equals lora_apply_strided's bit for bit.
 * On the tensor cores the columns of v past r_k are exact zeros; on the CUDA cores B rows past
 * r_k are never read.
 */
int lora_apply_ranked(void *y, int32_t ldy, const void *x, int32_t ldx,
                      const void *const *A_ptrs, const void *const *B_ptrs,
                      const int32_t *adapter_rank, const float *adapter_scale,
                      const int32_t *seg_starts, const int32_t *seg_adapter, const void *plan,
                      int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                      int32_t r_max, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream);

/*
 * ---- Adapter pool: device slots filled on demand from host copies ------------------------
 * Source: section "Core Innovation 2: Decoupled Multi-Tenant Memory Architecture" (dynamic
 * LoRA space allocation: adapter weights stream from host memory into a GPU pool
 * asynchronously, so that loading a cold adapter overlaps the running batch) and the pointer
 * arrays of section "Core Innovation 1".  The pool is host-side bookkeeping over device memory
 * the caller owns: `slots` slots of sgmv_pool_slot_bytes() each in one slab, 256-byte aligned.
 * Adapter k's host copy is its A block [L][h_in][r] and B block [L][r][h_out] (pinned host
 * memory lets the copies overlap compute; pageable memory works but copies synchronously).
 * Per batch: sgmv_pool_acquire (makes its adapters resident, pins their slots, writes the
 * device pointer arrays the compute calls take), then the compute calls on compute_stream,
 * then sgmv_pool_release (unpins; the slots may be refilled once the kernels enqueued before
 * it have completed).  One pool serves one compute stream; calls on one pool are serialised
 * by a mutex.  The pool allocates its host index and four pinned staging tables at creation
 * and nothing afterwards.
 */
typedef struct sgmv_pool sgmv_pool_t;

/* Bytes of one slot: the A and B blocks of one adapter, each rounded up to 256 bytes (0 for
 * bad arguments). */
size_t sgmv_pool_slot_bytes(int32_t layers, int32_t h_in, int32_t h_out, int32_t r,
                            sgmv_dtype_t dtype);

/*
 * sgmv_pool_create -- a pool of `slots` slots in the caller's device slab (>= slots *
 * sgmv_pool_slot_bytes(), 256-byte aligned, on the current device) for adapter ids
 * [0, num_adapters).  *out receives the handle.  Returns SGMV_OK, SGMV_EINVAL, SGMV_EALIGN or
 * SGMV_ECUDA.
 */
int sgmv_pool_create(sgmv_pool_t **out, void *slab, size_t slab_bytes, int32_t slots,
                     int32_t num_adapters, int32_t layers, int32_t h_in, int32_t h_out,
                     int32_t r, sgmv_dtype_t dtype);

/* Waits for the pool's outstanding events and frees its host-side state (not the slab). */
int sgmv_pool_destroy(sgmv_pool_t *pool);

/* Where adapter k's host copy lives (host pointers, read by later acquires).  Re-registering
 * a resident adapter drops its slot so that the next acquire copies the new weights
 * (SGMV_EBUSY while an unreleased batch reads it). */
int sgmv_pool_register(sgmv_pool_t *pool, int32_t adapter, const void *host_A,
                       const void *host_B);

/*
 * sgmv_pool_acquire -- makes the adapters of ids[0..n) (a HOST array; negative ids are skipped,
 * repeats count once) resident and pins their slots until sgmv_pool_release.  Each missing
 * adapter takes the least-recently-used slot that is unpinned and whose last release has
 * completed; its A and B blocks are copied on copy_stream.  compute_stream then waits for
 * those copies, and d_A_ptrs / d_B_ptrs (device arrays of num_adapters pointers, as
 * lora_apply takes them) are rewritten on compute_stream: entries of resident adapters point
 * at their slots, the others are null.  *copied (may be null) receives the number of adapters
 * copied.  Returns SGMV_OK, SGMV_EINVAL (an id past num_adapters or not registered),
 * SGMV_ENOSPACE (more distinct adapters than free slots: nothing is changed), SGMV_EALIGN or
 * SGMV_ECUDA.
 */
int sgmv_pool_acquire(sgmv_pool_t *pool, const int32_t *ids, int32_t n, void *d_A_ptrs,
                      void *d_B_ptrs, sgmv_stream_t copy_stream, sgmv_stream_t compute_stream,
                      int32_t *copied);

/* Unpins the slots of ids[0..n) (host array) after the batch's kernels were enqueued on
 * compute_stream; they become evictable once those kernels complete. */
int sgmv_pool_release(sgmv_pool_t *pool, const int32_t *ids, int32_t n,
                      sgmv_stream_t compute_stream);

/* Counters: acquires that found an adapter resident / copied it, and the slots in use. */
int sgmv_pool_stats(const sgmv_pool_t *pool, uint64_t *hits, uint64_t *misses,
                    int32_t *resident);

/*
 * sgmv_validate -- checks a segment table on the device and writes an OR of these bits to
 * *d_err (device int32, overwritten; 0 = valid):
 *   1  seg_starts decreases somewhere          2  seg_starts[0] < 0
 *   4  seg_starts[num_segments] > M            8  an adapter id >= num_adapters
 * Negative adapter ids are valid (no adapter).  The pages describe no such check; it is the
 * debugging counterpart of the fast path, which trusts the table.
 *   seg_starts, seg_adapter  in   device table as for lora_apply
 *   num_segments             >= 0 (any size)
 *   num_adapters             size of the pointer arrays the table will be used with
 *   M                        rows of x and y
 *   d_err                    out  device int32
 */
int sgmv_validate(const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                  int32_t num_adapters, int32_t M, int32_t *d_err, sgmv_stream_t stream);

/*
 * sgmv_validate_pointers -- checks, on the device, the weight pointers of every adapter that a
 * non-empty segment of the table uses, and writes an OR of these bits to *d_err (device int32,
 * overwritten; 0 = valid):
 *   16  A_ptrs[k] is null or not 16-byte aligned     32  the same for B_ptrs[k]
 * Only the pointer values are read, never the memory they point to, so a bad table cannot
 * fault here.  Adapter ids < 0 (no adapter) or >= num_adapters (reported by sgmv_validate,
 * bit 8) are skipped.  Either pointer array may be null (not checked: a shrink-only or
 * expand-only caller), not both.  The pages' pointer arrays (section "Core Innovation 1",
 * figure "SGMV Kernel Memory Layout & Execution Grid") carry no such check; this is the
 * debugging counterpart of the fast path, which dereferences them unchecked.
 *   A_ptrs, B_ptrs           in   device arrays of num_adapters device pointers (or null)
 *   seg_starts, seg_adapter  in   device table as for lora_apply
 *   num_segments, num_adapters    >= 0
 *   d_err                    out  device int32
 * Returns SGMV_OK, SGMV_EINVAL (null table, both arrays null, negative sizes), SGMV_EALIGN (a
 * pointer array not 8-byte aligned) or SGMV_ECUDA.
 */
int sgmv_validate_pointers(const void *const *A_ptrs, const void *const *B_ptrs,
                           const int32_t *seg_starts, const int32_t *seg_adapter,
                           int32_t num_segments, int32_t num_adapters, int32_t *d_err,
                           sgmv_stream_t stream);

/*
 * sgmv_get_error -- synchronises `stream`, copies the current device's library error word to
 * *host_err (a host int32: 0 or a negative sgmv_status_t: SGMV_ETIMEOUT, SGMV_EPLAN) and, when
 * clear != 0, resets it to 0.  Returns SGMV_OK or SGMV_ECUDA.
 */
int sgmv_get_error(int32_t *host_err, int32_t clear, sgmv_stream_t stream);

/*
 * sgmv_set_wait_limit -- sets the bound, in nanoseconds, of every device-side wait of later
 * launches on the current device (default 2e9 = 2 s; 0 restores the default).  With
 * inject_stall != 0 the next launches also wait once on a barrier that nothing completes, so
 * that the bound runs out: a fault-free way to exercise the timeout path.  Test hook; the
 * pages describe no counterpart.  Returns SGMV_OK or SGMV_ECUDA.
 */
int sgmv_set_wait_limit(uint64_t limit_ns, int32_t inject_stall);

/* Human-readable name of a status code (static string). */
const char *sgmv_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int sgmv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGMV_GB300_H */
