/*
 * fused_adamw.h -- C ABI of the GB300 fused AdamW / AMSGrad step and of the
 * gradient statistics that feed its skip and global-norm clip.
 *
 * Sources (RUDA documentation pages; section names as printed):
 *   [FA-ja] "実験的なデバイス上の融合 AdamW / AMSGrad"   (ja/docs/fused-adamw)
 *   [FA-zh] "实验性融合 AdamW / AMSGrad"                  (zh/docs/fused-adamw)
 *   [TR-zh] "训练与状态保存"                                (zh/docs/training)
 *
 * General contract (applies to every entry point below):
 *   - Pointers named "device" must be CUDA device (or managed) memory of the
 *     current device.  Host pointers are rejected with FA_ERR_POINTER
 *     ([FA-ja] "サポートされている契約": no arbitrary host pointers).
 *   - ``stream`` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  All device work is enqueued on it, in call order.  The merge
 *     kernels and the gated update are launched as programmatic dependents:
 *     they may be scheduled while the kernel before them on the stream is still
 *     running, and wait for it to complete before touching any memory, so the
 *     stream's order is unchanged for the caller.
 *   - FA_OK from an enqueuing call means the work was ENQUEUED, not that it
 *     finished ([FA-ja] "低レベルの使用"; [FA-zh] "用法"): check the stream's
 *     completion before trusting or checkpointing outputs; after a device
 *     failure discard them.
 *   - Validation happens before anything is enqueued or written; on any
 *     error no output (host or device) is modified ([FA-ja] "低レベルの使用").
 *   - The library allocates nothing, on the device or pinned on the host, and
 *     creates no stream or event: buffers (outputs, row statistics, scratch,
 *     report, the report mailbox) belong to the caller.  Its only state is
 *     caches of device properties, a device flag for the update pipeline's
 *     bounded waits (fa_device_error) and one fixed merge scratch array
 *     (fa_merge_gradient_stats_static), all part of the loaded library.
 *   - A stream that is being captured into a CUDA graph is accepted without
 *     the device check (CUDA cannot report a capturing stream's device).
 *     fa_analyze_gradient and fa_merge_gradient_stats (and the chunk merge) may
 *     be captured and replayed.  The update calls take the step count
 *     and the coefficients from the host at every call, so a captured update
 *     would replay one fixed step: do not capture them ([FA-ja]
 *     "サポートされている契約": graph replay with a device step counter is not
 *     supported).
 *   - Parameters and moments are dense contiguous FP32; gradients are dense
 *     contiguous FP32, FP16 or BF16 of the same element count
 *     ([FA-zh] "增加的实际能力").  Strides, broadcasts and sparse gradients
 *     cannot be expressed through this ABI; the Python binding rejects them.
 */
#ifndef FUSED_ADAMW_H
#define FUSED_ADAMW_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 2

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_NULL = 1,      /* a required pointer is NULL, or state pointers disagree with t  */
    FA_ERR_DTYPE = 2,     /* unknown gradient dtype                                          */
    FA_ERR_SIZE = 3,      /* negative count, or a buffer too small for the request           */
    FA_ERR_OPTION = 4,    /* option/control out of range (non-finite lr, beta outside [0,1),  */
                          /* eps < 0, scale <= 0, t would overflow, ...)                     */
    FA_ERR_ALIAS = 5,     /* buffers that must be distinct overlap                           */
    FA_ERR_POINTER = 6,   /* host pointer, or device memory of another device/stream device  */
    FA_ERR_ALIGN = 7,     /* pointer not aligned to its element size                         */
    FA_ERR_PLAN = 8,      /* statistics rows outside 1..4,194,304                            */
    FA_ERR_CUDA = 9,      /* a CUDA call failed (launch error, copy error)                   */
    FA_ERR_SEGMENTS = 10  /* segment table not non-decreasing from 0 to n                    */
} fa_status;

typedef enum fa_dtype { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

/* Hyper-parameters, as doubles ([FA-ja] "低レベルの使用": AdamWOptions).
 * Valid ranges: lr >= 0, 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0,
 * weight_decay >= 0, all finite; amsgrad and maximize are 0 or 1. */
typedef struct fa_options {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    int32_t amsgrad;
    int32_t maximize;
} fa_options;

/* Per-call control ([FA-ja] "低レベルの使用": StepControl).  gradient_scale
 * divides the stored gradient (finite, > 0); skip_update is the caller's
 * found_inf flag -- this call does not compute it. */
typedef struct fa_step_control {
    double gradient_scale;
    int32_t skip_update;
} fa_step_control;

/* 12-byte statistics record ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练": a 12-byte
 * report).  Row records, intermediate merge records and the final report all
 * use it.  nonfinite counts stored NaN and +-Inf values exactly (saturating
 * at 2^32-1).  When nonfinite == 0 the record holds the sum of squares of the
 * STORED (still scaled) gradient values in one of two forms:
 *   sum_sq >= 0: the sum is sum_sq + sum_sq_lo (added in FP64);
 *   sum_sq <  0: the sum is -(sum_sq + sum_sq_lo) * 2^192 -- the form taken
 *                when the sum would overflow FP32 (a finite value above about
 *                1.8e19 has a square beyond FP32's range): the values are
 *                multiplied by 2^-96 before they are squared.
 * fa_stats_sum_sq decodes either form.  When nonfinite > 0 the sum is
 * unspecified (it may be Inf or NaN) -- the step is skipped then and the sum
 * is never used. */
typedef struct fa_stats {
    float sum_sq;
    uint32_t nonfinite;
    float sum_sq_lo;
} fa_stats;

/* A report mailbox: 16 bytes of pinned host memory that the device can write
 * (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped; with unified
 * addressing every pinned allocation qualifies), 4-byte aligned, owned by the
 * caller.  The kernel that produces a step's final record (the last merge, or the
 * per-segment decision kernel) also stores it here and then, after a system-wide
 * fence, its sequence number, so that the host can read the record without a copy
 * or an event on the stream.  One mailbox serves one call at a time; its initial
 * contents do not matter. */
typedef struct fa_report_mailbox {
    fa_stats report;
    uint32_t seq;
} fa_report_mailbox;

/* Outcome of a step that ran the statistics path. */
typedef struct fa_step_report {
    int32_t updated;           /* 1 when the update kernel was enqueued                 */
    int32_t skipped_nonfinite; /* 1 when the step was skipped for a non-finite gradient */
    uint64_t nonfinite;        /* non-finite stored gradient values found               */
    double grad_norm;          /* global L2 norm of the unscaled gradient               */
    double clip_coef;          /* factor applied to the unscaled gradient (1 = none)    */
} fa_step_report;

/* ---- host-only helpers ---------------------------------------------------- */

/* The sum of squares a statistics record stands for ([TR-zh] "在 ruda:0 上进行原生
 * PyTorch 训练": the 12-byte report; the pages fix its size, not its encoding):
 * either form above, in FP64, into *sum_sq -- the value that fa_clip_decision
 * takes (the total of several ranks' or segments' records is the sum of these).
 * Host only; FA_ERR_NULL for a NULL pointer. */
fa_status fa_stats_sum_sq(const fa_stats *record, double *sum_sq);

/* FA_ABI_VERSION of the loaded library, for a caller to check against the
 * header it was built with (library bookkeeping; the pages have no counterpart). */
int32_t fa_abi_version(void);

/* A static English description of a status code, never NULL (the status codes
 * follow the error classes of [FA-ja] "低レベルの使用": invalid options, sizes,
 * pointers and overlaps are rejected before anything runs). */
const char *fa_status_string(fa_status status);

/* Some large updates (steady steps decided on the device with a gradient scale
 * that is not a power of two, or per segment from the reports in each launch)
 * stage tiles through shared memory with TMA bulk copies; every
 * wait in that pipeline is bounded (about a second), and a wait that gives up
 * sets a device flag, drains its own copies and ends the kernel early (its
 * outputs are then incomplete: discard them, as [FA-ja] "低レベルの使用" asks of
 * any device failure).  This reads the flag of the current device into *flag
 * (0 = no wait ever gave up) and clears it when clear != 0.  Waits for the
 * device; FA_ERR_CUDA if it cannot be read.  The pipeline is this library's;
 * the pages have no counterpart. */
fa_status fa_device_error(int32_t *flag, int32_t clear);

/* Bounds-checked build (a test variant of the library compiled with
 * -DFA_BOUNDS_CHECK=1; the pages have no counterpart): every kernel checks the
 * element range it is about to touch against its array's length, and counts
 * and skips an access outside it instead of performing it.  *enabled is 1 in
 * that build and 0 in the normal one.  When violations is not NULL it receives
 * the number of out-of-range accesses on the current device since the last
 * clear (always 0 in the normal build, which touches no device for this);
 * clear != 0 resets the count.  Waits for the device in the checked build;
 * FA_ERR_CUDA if the count cannot be read. */
fa_status fa_bounds_check_report(int32_t *enabled, uint64_t *violations, int32_t clear);

/* Self-test of the bounded waits above (the pages have no counterpart), with no
 * fault: one steady-state update
 * of the n-element p, m, v (device, FP32) with gradient g, launched so that
 * every shared-memory stage waits for 16 bytes that never arrive.  Each wait
 * gives up after its limit (about a second), the kernel drains its own
 * copies and returns without writing p, m or v; the call waits for it and
 * stores the flag in *flag (1 when the waits gave up, as they must), then
 * clears it.  n must be large enough for the shared-memory path (at least two
 * tiles per SM; FA_ERR_SIZE else) and the pointers 16-byte co-aligned
 * (FA_ERR_ALIGN else).  Not part of the update path. */
fa_status fa_pipeline_selftest(int64_t n, float *p, const void *g, fa_dtype gdt, float *m,
                               float *v, int32_t *flag, void *stream);

/* Defaults ([FA-ja] "この演算子を使用する理由": betas (0.9, 0.999), eps 1e-5,
 * weight_decay 1e-4, matching RUDA's AdamWConfig).  The pages state no default
 * learning rate; 1e-3 is used.  amsgrad = maximize = 0. */
fa_options fa_options_default(void);

/* Host coefficients of one update, FP64 then cast to FP32 ([FA-ja]
 * "この演算子を使用する理由": the host computes the bias corrections once per call
 * from FP64 integer powers and casts them to FP32).  ``t`` is the 1-based step
 * of the update; ``grad_mult`` an extra factor on the unscaled gradient.
 * Writes 9 floats: beta1, 1-beta1, beta2, 1-beta2, lr/(1-beta1^t),
 * 1/(1-beta2^t), eps, 1-lr*weight_decay, (maximize ? -1 : 1)*grad_mult/scale. */
fa_status fa_step_coefficients(const fa_options *options, uint64_t t, double gradient_scale,
                               double grad_mult, float coef_out[9]);

/* ---- the fused update ----------------------------------------------------- */

/*
 * Out-of-place step ([FA-ja] "低レベルの使用" adamw_step and "割り当てとパフォーマンスの
 * モデル"; [FA-zh] "增加的实际能力").  Per element, one HBM pass:
 *   g = stored/gradient_scale, negated if maximize;
 *   m = beta1*m + (1-beta1)*g;  v = beta2*v + (1-beta2)*g*g;
 *   AMSGrad: vmax = max(vmax, v) (uncorrected) and v_used = vmax, else v_used = v;
 *   p = p*(1-lr*wd) - lr*(m/(1-beta1^t)) / (sqrt(v_used/(1-beta2^t)) + eps).
 *
 *   n               element count (>= 0)
 *   p, g, gdt       device inputs: FP32 parameters, gradient of type gdt
 *   m, v, vmax      device state; all NULL iff t_in == 0 (no state yet: the
 *                   first update writes the moments without reading them);
 *                   vmax NULL unless options->amsgrad
 *   t_in            completed updates so far
 *   p_out, m_out, v_out, vmax_out
 *                   device outputs (vmax_out NULL unless amsgrad); distinct,
 *                   and overlapping no input
 *   t_out, updated  host outputs: t_in+1 and 1 when an update was enqueued;
 *                   t_in and 0 when n == 0 or ctl.skip_update: then nothing is
 *                   launched, no buffer is checked or touched, and the output
 *                   pointers may be NULL (the caller need not allocate them).
 */
fa_status fa_adamw_step(int64_t n, const float *p, const void *g, fa_dtype gdt,
                        const float *m, const float *v, const float *vmax, uint64_t t_in,
                        const fa_options *options, fa_step_control ctl,
                        float *p_out, float *m_out, float *v_out, float *vmax_out,
                        uint64_t *t_out, int32_t *updated, void *stream);

/*
 * In-place step on caller-owned storage ([FA-ja] "ネイティブ PyTorch ストレージと
 * 階層統計": adamw_scaled on framework-preallocated storage).  Same arithmetic as
 * fa_adamw_step; p, m, v (and vmax with AMSGrad) are read and rewritten in
 * place and must not overlap each other or g.  ``*t`` is the completed step
 * count on entry and is advanced on an update; when *t == 0 the moments are
 * only written.  ``grad_mult`` multiplies the unscaled gradient (the global
 * clip coefficient; 1 = none; finite, >= 0).  n == 0 or ctl.skip_update:
 * nothing is launched or checked, *t is unchanged and *updated = 0.
 */
fa_status fa_adamw_step_inplace(int64_t n, float *p, const void *g, fa_dtype gdt,
                                float *m, float *v, float *vmax, uint64_t *t,
                                const fa_options *options, fa_step_control ctl,
                                double grad_mult, int32_t *updated, void *stream);

/*
 * Pre-flattened multi-tensor bucket ([FA-ja] "サポートされている契約": a flattened
 * bucket is valid only when every element shares the options and the step
 * count).  ``seg_offsets`` (host, nseg+1 entries, non-decreasing from 0 to
 * n_total) records the tensors packed in the bucket; the update itself is ONE
 * launch over the flat buffers, identical element by element to updating
 * each tensor on its own.  Other arguments as fa_adamw_step_inplace.
 */
fa_status fa_bucket_step(const int64_t *seg_offsets, int32_t nseg, int64_t n_total,
                         float *p, const void *g, fa_dtype gdt, float *m, float *v,
                         float *vmax, uint64_t *t, const fa_options *options,
                         fa_step_control ctl, double grad_mult, int32_t *updated,
                         void *stream);

/*
 * One update of a pre-flattened bucket in any of its variants, described by
 * one record (fa_bucket_update_args): where the gradient multiplier comes from,
 * and whether the low-precision model copy is written in the same pass.  Every variant is the
 * per-element update of fa_bucket_step over the flat buffers, identical to
 * updating each tensor on its own ([FA-ja] "サポートされている契約").
 *
 * The multiplier of the unscaled gradient, from exactly one source:
 *   - grad_mult (host): one factor, the global clip coefficient (1 = none;
 *     finite, >= 0).  It must be 1 when another source is given.
 *   - seg_grad_mult (host, nseg doubles, finite, >= 0): one factor per segment
 *     ([TR-zh] "FP32 主参数与混合参数存储": Fp32MasterOptimizer clips each
 *     parameter by its own rule).  One launch per 240 segments.
 *   - report (device, one fa_stats as written by fa_merge_gradient_stats earlier
 *     on the same stream): the decision is taken in the update kernel
 *     ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练": a non-finite gradient skips the
 *     whole step; the global L2 clip of the unscaled gradient).  The kernel skips
 *     when the report counts a non-finite value, and otherwise multiplies by the
 *     coefficient fa_clip_decision computes (max_grad_norm <= 0: no clip), with
 *     the same FP64 operations in the same order.  The results are therefore
 *     bit-identical to reading the report back and passing that coefficient as
 *     grad_mult.  The update is launched as a programmatic dependent of the kernel
 *     before it.
 *   - seg_reports (device, nseg fa_stats as written by
 *     fa_merge_gradient_stats_chunks earlier on the same stream): the same per
 *     segment.  Any non-finite count skips the whole update; segment k takes the
 *     coefficient of record k.  With seg_decided (device scratch of
 *     seg_decided_elements >= nseg + 1 FP32 elements, FA_ERR_SIZE when fewer,
 *     overlapping no other buffer; only with seg_reports, else FA_ERR_OPTION),
 *     one small kernel first takes every segment's decision there, once for the
 *     bucket, and the update kernels read it instead of each deciding from the
 *     reports: the same bits, and faster on large buckets.  Its contents are
 *     scratch.
 *
 * p_model (device, n_total elements of model_dtype = FA_F16 or FA_BF16, 2-byte
 * aligned, overlapping no other buffer): each updated FP32 p rounded to nearest,
 * ties to even, written in the same HBM pass; +2 bytes per parameter instead of a
 * separate 6-byte cast pass ([TR-zh] "FP32 主参数与混合参数存储": the FP32 master
 * is updated in FP32 and the parameters come back in their storage dtype).  Not
 * with the per-segment sources (FA_ERR_OPTION).  FA_ERR_DTYPE for another dtype.
 *
 * ``t`` is the completed step count; the update is step t + 1.  This call changes
 * no count.  On return *enqueued is 1 when an update kernel was enqueued, and 0
 * for n_total == 0 or ctl.skip_update: then nothing is launched and no buffer is
 * checked or touched.  With a host multiplier the caller advances its count by one
 * when *enqueued.  With a device decision it reads the report and advances the
 * count unless the report counts a non-finite value.  The reports and the model copy
 * must not overlap the state, the gradient or each other (FA_ERR_ALIAS).
 */
typedef struct fa_bucket_update_args {
    const int64_t *seg_offsets;   /* host, nseg + 1 offsets from 0 to n_total (NULL, 0: one) */
    int32_t nseg;
    int64_t n_total;
    float *p;                     /* device FP32 parameters, updated in place        */
    const void *g;                /* device gradient of type gdt                      */
    fa_dtype gdt;
    float *m, *v, *vmax;          /* device FP32 state; vmax only with AMSGrad        */
    uint64_t t;                   /* completed updates                                */
    double grad_mult;             /* host factor (1 = none)                           */
    const double *seg_grad_mult;  /* host, one factor per segment, or NULL            */
    const fa_stats *report;       /* device report: decision in the kernel, or NULL   */
    const fa_stats *seg_reports;  /* device, one report per segment, or NULL          */
    double max_grad_norm;         /* clip threshold of the device decisions (<= 0: none) */
    void *p_model;                /* device FP16/BF16 copy of the updated p, or NULL  */
    fa_dtype model_dtype;         /* FA_F16 or FA_BF16 when p_model is set            */
    float *seg_decided;           /* with seg_reports: device scratch for the decisions, or NULL */
    int64_t seg_decided_elements; /* its FP32 elements (at least nseg + 1)            */
} fa_bucket_update_args;

/* Enqueues the bucket update that ``update`` describes ([FA-ja] "サポートされている
 * 契約": a flattened bucket shares the options and the step count; the variants and
 * their rules above).  *enqueued: 1 when an update kernel was enqueued. */
fa_status fa_bucket_update(const fa_bucket_update_args *update, const fa_options *options,
                           fa_step_control ctl, int32_t *enqueued, void *stream);

/*
 * The staged comparison, for benchmarks only ([FA-ja] "割り当てとパフォーマンスのモデル";
 * [FA-zh] "优化点与边界": an explicit staged baseline of 4 kernels, 5 with AMSGrad,
 * with repeated gradient reads and a delta buffer: 48 and 60 bytes per
 * parameter for FP32 gradients in steady state, against 28 and 36 fused).
 * Stages: m; v; (vmax); delta = lr/bc1*m/(sqrt(v_used/bc2)+eps) into the
 * caller's FP32 buffer ``delta`` (n elements, overlapping nothing); p.  Each
 * stage evaluates the fused kernel's FP32 operations, so the results equal
 * fa_adamw_step_inplace's bit for bit.  Arguments as fa_adamw_step_inplace;
 * p, m, v, vmax and delta must be 16-byte aligned and g 16-byte (FP32) or
 * 8-byte (FP16/BF16) aligned, else FA_ERR_ALIGN.
 */
fa_status fa_adamw_step_staged(int64_t n, float *p, const void *g, fa_dtype gdt, float *m,
                               float *v, float *vmax, uint64_t *t, const fa_options *options,
                               fa_step_control ctl, double grad_mult, float *delta,
                               int32_t *updated, void *stream);

/*
 * fa_bucket_step_clipped with the update gated on the device: the analysis
 * and the merge are enqueued, the merge that writes report_dev also posting the
 * report to ``mailbox`` (see fa_report_mailbox), then the gated update, which
 * starts as the merge's programmatic dependent: nothing waits for the host.
 * The host waits only for the posted report, takes the same decision from it
 * ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练": the report is read back and a
 * non-finite gradient skips the whole step) and advances *t unless the step
 * was skipped.  Returns once the report is read; the update may still run
 * (FA_OK means enqueued).  Results are bit-identical to
 * fa_bucket_step_clipped.  The wait for the report gives up with FA_ERR_CUDA
 * when the stream reports an error or finishes without posting it (and after
 * five minutes in any case).  mailbox: pageable or device memory is
 * FA_ERR_POINTER, NULL FA_ERR_NULL.  Other arguments as fa_bucket_step_clipped.
 */
fa_status fa_bucket_step_clipped_gated(const int64_t *seg_offsets, int32_t nseg, int64_t n_total,
                                       float *p, const void *g, fa_dtype gdt, float *m, float *v,
                                       float *vmax, uint64_t *t, const fa_options *options,
                                       fa_step_control ctl, double max_grad_norm,
                                       int32_t row_len, fa_stats *rows_buf,
                                       int64_t rows_capacity, float *scratch,
                                       int64_t scratch_elements, fa_stats *report_dev,
                                       fa_report_mailbox *mailbox, fa_step_report *out,
                                       void *stream);

/* ---- gradient statistics -------------------------------------------------- */

/*
 * Reduction plan ([FA-ja] "ネイティブ PyTorch ストレージと階層統計": StatsPlan::new(rows)
 * accepts 1..=4,194,304 rows at fan-in 1024; scratch_elements counts FP32
 * elements, excluding the initial statistics and the final report; at most
 * 49,200 bytes).  Each merge kernel reduces groups of 1024 records, until one
 * record is left.  merge_kernels is 1 for rows <= 1024, 2 up to 1,048,576 and
 * 3 above ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练": at most two extra merge
 * kernels, none at <= 1024 rows).  FA_ERR_PLAN outside 1..4,194,304.
 */
fa_status fa_stats_plan(int64_t rows, int32_t *merge_kernels, int64_t *scratch_elements);

/* Row count of an analysis ([FA-ja] "ネイティブ PyTorch ストレージと階層統計":
 * analyze_gradient works in rows): each segment [seg[k], seg[k+1]) is cut into rows
 * of row_len elements, its last row possibly shorter; rows never span
 * segments.  seg_offsets NULL / nseg 0 means one segment [0, n).  Host only. */
fa_status fa_stats_rows(int64_t n, int32_t row_len, const int64_t *seg_offsets, int32_t nseg,
                        int64_t *rows);

/*
 * Read-only gradient analysis ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练":
 * read-only gradient analysis; [FA-ja] "ネイティブ PyTorch ストレージと階層統計":
 * analyze_gradient).  Writes one fa_stats per row (rows as fa_stats_rows) to the
 * device array rows_out (capacity rows_capacity >= rows; FA_ERR_SIZE else).
 * The row count must be a valid plan size (FA_ERR_PLAN else).  The gradient
 * is not modified.
 */
fa_status fa_analyze_gradient(const void *g, fa_dtype gdt, int64_t n, int32_t row_len,
                              const int64_t *seg_offsets, int32_t nseg, fa_stats *rows_out,
                              int64_t rows_capacity, void *stream);

/*
 * Hierarchical merge ([FA-ja] "ネイティブ PyTorch ストレージと階層統計":
 * merge_gradient_stats; [TR-zh]: fan-in 1024, changes the reduction order, not
 * the clip policy).  Reduces ``rows`` device records to one device report, in
 * fa_stats_plan's merge kernels.  ``scratch`` is caller-owned device memory of
 * at least fa_stats_plan's scratch_elements floats (may be NULL when that is
 * 0); its contents on entry do not matter.  Sums are carried as double-float
 * values (an FP32 value and its FP32 residual, added with error-free
 * transformations) and passed between levels as (sum_sq, sum_sq_lo) pairs.
 */
fa_status fa_merge_gradient_stats(const fa_stats *rows_in, int64_t rows, float *scratch,
                                  int64_t scratch_elements, fa_stats *report, void *stream);

/*
 * fa_merge_gradient_stats without a caller-supplied scratch buffer.  The pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory: for example a plugin whose host framework owns
 * every device allocation and does not let extensions call cudaMalloc, or
 * code on a latency-critical path where cudaMalloc/cudaFree, which may
 * synchronise the device, are not allowed.  Inputs and output stay the
 * caller's (rows_in and report, as in fa_merge_gradient_stats).
 *
 * The intermediate records go to one fixed scratch array inside the library
 * (12,300 floats = 49,200 bytes: the largest reduction plan, 4,194,304 rows).
 * Every GPU that loads the library holds that array until the process exits.
 * rows outside 1..4,194,304 are rejected with FA_ERR_PLAN before anything is
 * enqueued.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  A call on a stream that is being captured, on a
 * device where no earlier call has looked the address up, returns FA_ERR_CUDA
 * with nothing enqueued and the capture left intact.  All calls share the one array: the merge
 * writes every scratch record before reading it, so leftovers from an
 * earlier call never leak into a result, but calls whose kernels overlap on
 * the GPU (different streams without ordering between them) race on the
 * array and must be serialised by the caller.
 */
fa_status fa_merge_gradient_stats_static(const fa_stats *rows_in, int64_t rows,
                                         fa_stats *report, void *stream);

/* ---- per-parameter statistics and clipping ---------------------------------- */

/* Scratch (FP32 elements) for fa_merge_gradient_stats_chunks ([FA-ja]
 * "ネイティブ PyTorch ストレージと階層統計": merge_gradient_stats_chunks): 3 words for each
 * group of at most 1024 rows within a chunk.  chunk_rows (host, nchunks+1
 * entries) are row offsets, non-decreasing from 0; their total must be a
 * valid plan size (FA_ERR_PLAN else).  Host only. */
fa_status fa_stats_chunk_scratch(const int64_t *chunk_rows, int32_t nchunks,
                                 int64_t *scratch_elements);

/*
 * One report per chunk of rows ([FA-ja] "ネイティブ PyTorch ストレージと階層統計":
 * merge_gradient_stats_chunks; chunks here are the rows of one bucket segment,
 * i.e. one parameter).  Rows [chunk_rows[k], chunk_rows[k+1]) of rows_in merge
 * into chunk_reports[k] (device, nchunks records; an empty chunk gives a zero
 * record): first groups of at most 1024 rows that never span two chunks, into
 * the caller's scratch (fa_stats_chunk_scratch elements), then one merge per
 * chunk.  Double-float sums as in fa_merge_gradient_stats; a fixed order, so
 * results are reproducible.
 */
fa_status fa_merge_gradient_stats_chunks(const fa_stats *rows_in, const int64_t *chunk_rows,
                                         int32_t nchunks, float *scratch,
                                         int64_t scratch_elements, fa_stats *chunk_reports,
                                         void *stream);

/*
 * The statistics-guarded step with per-parameter clipping ([TR-zh] "FP32 主参数与
 * 混合参数存储": Fp32MasterOptimizer clips each parameter by its own rule; [TR-zh]
 * "在 ruda:0 上进行原生 PyTorch 训练": the report is read back first and a non-finite
 * gradient skips the whole step): analyse the bucket
 * in segment-aligned rows, merge one report per segment into seg_reports
 * (device, nseg records), read them back (nseg * 12 bytes; synchronises),
 * skip the whole step when any value is non-finite, else clip each segment
 * by its own norm (coef_k = max_grad_norm / norm_k when above it, 1 otherwise;
 * max_grad_norm <= 0: no clipping) and update with those multipliers.
 * seg_norms / seg_coefs (host, nseg doubles, may be NULL) receive each
 * segment's unscaled norm and coefficient; out->grad_norm is the whole
 * gradient's norm and out->clip_coef the smallest coefficient.  Scratch is
 * fa_stats_chunk_scratch's size for the segment rows; other arguments as
 * fa_bucket_step_clipped.
 */
fa_status fa_bucket_step_clipped_per_segment(
    const int64_t *seg_offsets, int32_t nseg, int64_t n_total, float *p, const void *g,
    fa_dtype gdt, float *m, float *v, float *vmax, uint64_t *t, const fa_options *options,
    fa_step_control ctl, double max_grad_norm, int32_t row_len, fa_stats *rows_buf,
    int64_t rows_capacity, float *scratch, int64_t scratch_elements, fa_stats *seg_reports,
    double *seg_norms, double *seg_coefs, fa_step_report *out, void *stream);

/*
 * fa_bucket_step_clipped_per_segment with the decision on the device ([FA-ja]
 * "ネイティブ PyTorch ストレージと階層統計": merge_gradient_stats_chunks; [TR-zh]
 * "FP32 主参数与混合参数存储": per-parameter clipping): the
 * segment-aligned analysis, the per-segment merges into seg_reports and the
 * update deciding per segment on the device are enqueued back to back;
 * nothing waits for the host.  Once the merges are done with ``scratch``, and
 * when it holds at least nseg + 1 elements, one small kernel takes every
 * segment's decision there and the update reads it; otherwise the update
 * decides from seg_reports itself (as fa_bucket_update with seg_reports).
 * Either way the results are bit-identical to fa_bucket_step_clipped_per_segment.
 * ``t`` is the completed step count and is not changed: the caller advances
 * its count unless the step counted a non-finite value.
 *
 * mailbox (optional, as in fa_bucket_step_clipped_gated): NULL returns once
 * everything is enqueued, and the caller reads seg_reports after the stream
 * reaches them.  Otherwise the kernel that takes the decisions, which runs
 * before the update, posts the bucket's record to the mailbox: the exact count
 * of non-finite values over all segments (saturating) and the FP64 total of
 * the segments' sums of squares (decoded by fa_stats_sum_sq).  The call returns
 * once that record is posted, while the update may still run, and the caller
 * decides from mailbox->report.nonfinite.  The wait gives up with FA_ERR_CUDA
 * as fa_bucket_step_clipped_gated's does; pageable or device memory is
 * FA_ERR_POINTER.
 *
 * For n_total == 0 or ctl.skip_update nothing is enqueued, and neither
 * seg_reports nor the mailbox is written.  Other arguments as
 * fa_bucket_step_clipped_per_segment.
 */
fa_status fa_bucket_step_clipped_per_segment_gated(
    const int64_t *seg_offsets, int32_t nseg, int64_t n_total, float *p, const void *g,
    fa_dtype gdt, float *m, float *v, float *vmax, uint64_t t, const fa_options *options,
    fa_step_control ctl, double max_grad_norm, int32_t row_len, fa_stats *rows_buf,
    int64_t rows_capacity, float *scratch, int64_t scratch_elements, fa_stats *seg_reports,
    fa_report_mailbox *mailbox, void *stream);

/* Copies the 12-byte device report to host memory and waits for the stream
 * ([TR-zh]: the report is read back before any update).  Synchronises. */
fa_status fa_read_report(const fa_stats *report_dev, fa_stats *report_host, void *stream);

/*
 * Host decision ([TR-zh] "在 ruda:0 上进行原生 PyTorch 训练": any non-finite gradient
 * skips the whole step; optional global L2 clipping after unscale).
 * sum_sq_stored is the sum of squares of the stored gradient (a report's
 * fa_stats_sum_sq, or the sum of several ranks' reports).  Outputs:
 * skip = nonfinite > 0; grad_norm = sqrt(sum_sq_stored)/gradient_scale;
 * clip_coef = max_grad_norm/grad_norm when max_grad_norm > 0 and the norm
 * exceeds it, else 1.  Host only.
 */
fa_status fa_clip_decision(double sum_sq_stored, uint64_t nonfinite, double gradient_scale,
                           double max_grad_norm, int32_t *skip, double *grad_norm,
                           double *clip_coef);

/* fa_read_report followed by fa_clip_decision ([TR-zh] "在 ruda:0 上进行原生 PyTorch
 * 训练": the 12-byte report is read back, then the skip and the clip are decided).
 * Synchronises the stream. */
fa_status fa_clip_decide(const fa_stats *report_dev, double gradient_scale, double max_grad_norm,
                         int32_t *skip, double *grad_norm, double *clip_coef, void *stream);

/*
 * The whole statistics-guarded step on a bucket ([TR-zh] "在 ruda:0 上进行原生
 * PyTorch 训练": ruda_torch.AdamW(fused_step=True, max_grad_norm, hierarchical_stats
 * =True) -- analyse, merge, read back 12 bytes, then update or skip).
 *   1. ctl.skip_update or n_total == 0: nothing is launched; t unchanged.
 *   2. fa_analyze_gradient over segment-aligned rows of row_len into rows_buf.
 *   3. fa_merge_gradient_stats into report_dev, using scratch.
 *   4. fa_clip_decide (synchronises the stream).
 *   5. Non-finite found: skip, t unchanged.  Else one fa_bucket_step with
 *      grad_mult = clip_coef (max_grad_norm <= 0: no clipping).
 * ``out`` (host) receives the decision.  Buffers as in the calls above.
 */
fa_status fa_bucket_step_clipped(const int64_t *seg_offsets, int32_t nseg, int64_t n_total,
                                 float *p, const void *g, fa_dtype gdt, float *m, float *v,
                                 float *vmax, uint64_t *t, const fa_options *options,
                                 fa_step_control ctl, double max_grad_norm, int32_t row_len,
                                 fa_stats *rows_buf, int64_t rows_capacity, float *scratch,
                                 int64_t scratch_elements, fa_stats *report_dev,
                                 fa_step_report *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FUSED_ADAMW_H */
