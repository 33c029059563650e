/*
 * ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain FP64 restatement of the gradient statistics that drive the
 * non-finite skip and the optional global-norm clip, and of the reduction
 * plan's sizes.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load this code.  It shares no source with the CUDA library.
 *
 * Passages followed (RUDA documentation pages):
 *   - "训练与状态保存" (zh/docs/training), section "在 ruda:0 上进行原生 PyTorch 训练":
 *     read-only gradient analysis, global L2 clipping after unscale, a 12-byte
 *     report read back before any update, the whole step skipped on any
 *     non-finite gradient; hierarchical statistics at fan-in 1024 add at most
 *     two merge kernels and 49,200 bytes of reusable space, none at <= 1024
 *     rows, and change the reduction order but not the clip policy.
 *   - "実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw), section
 *     "ネイティブ PyTorch ストレージと階層統計": StatsPlan::new(rows) accepts
 *     1..=4,194,304 rows at fan-in 1024; scratch_elements counts FP32 elements
 *     and excludes the initial statistics and the final report.
 *
 * The statistic is defined on the whole gradient: the sum of squares of the
 * unscaled gradient and the number of stored values that are NaN or +-Inf.
 * Rows are a grouping only; this file sums in plain index order in FP64.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

static int is_nonfinite(double x)
{
    return isnan(x) || isinf(x);
}

/* Whole-gradient statistics: sum of (stored / scale)^2 and the non-finite count
 * ("训练与状态保存", "在 ruda:0 上进行原生 PyTorch 训练": the global L2 norm after
 * unscale, and any non-finite value skips the step). */
void oracle_gradient_stats(int64_t n, const void *g, int gdtype, double gradient_scale,
                           double *sum_sq, uint64_t *nonfinite)
{
    double s = 0.0;
    uint64_t c = 0;
    for (int64_t i = 0; i < n; ++i) {
        double x = oracle_widen(g, gdtype, i);
        if (is_nonfinite(x)) {
            ++c;
            continue;
        }
        double u = x / gradient_scale;
        s += u * u;
    }
    *sum_sq = s;
    *nonfinite = c;
}

/*
 * Per-row statistics of the stored gradient ("実験的なデバイス上の融合 AdamW / AMSGrad",
 * "ネイティブ PyTorch ストレージと階層統計": analyze_gradient).  The buffer is split into
 * segments [seg[k], seg[k+1]) (one segment [0, n) when nseg == 0); each
 * segment is cut into rows of row_len elements, its last row possibly
 * shorter.  Rows never span two segments.  Returns the number of rows, or -1
 * on a malformed segment table.  Non-finite values are counted and left out
 * of the row's sum.
 */
int64_t oracle_row_stats(int64_t n, const void *g, int gdtype, int64_t row_len,
                         const int64_t *seg, int64_t nseg,
                         double *row_sum_sq, uint64_t *row_nonfinite)
{
    int64_t one[2] = {0, n};
    if (nseg == 0) {
        seg = one;
        nseg = 1;
    }
    if (row_len <= 0 || seg[0] != 0 || seg[nseg] != n)
        return -1;
    int64_t r = 0;
    for (int64_t k = 0; k < nseg; ++k) {
        if (seg[k + 1] < seg[k])
            return -1;
        for (int64_t start = seg[k]; start < seg[k + 1]; start += row_len) {
            int64_t end = start + row_len < seg[k + 1] ? start + row_len : seg[k + 1];
            double s = 0.0;
            uint64_t c = 0;
            for (int64_t i = start; i < end; ++i) {
                double x = oracle_widen(g, gdtype, i);
                if (is_nonfinite(x)) {
                    ++c;
                    continue;
                }
                s += x * x;
            }
            if (row_sum_sq)
                row_sum_sq[r] = s;
            if (row_nonfinite)
                row_nonfinite[r] = c;
            ++r;
        }
    }
    return r;
}

/*
 * Reduction plan ("実験的なデバイス上の融合 AdamW / AMSGrad", "ネイティブ PyTorch
 * ストレージと階層統計": StatsPlan; "训练与状态保存", "在 ruda:0 上进行原生 PyTorch
 * 训练": at most two extra merge kernels and 49,200 bytes) for ``rows`` row
 * records at fan-in ``fan_in``: each merge
 * kernel turns its input records into ceil(count / fan_in) records, until
 * one record -- the report -- is left.  Every record is three 4-byte words
 * (12 bytes).  The intermediate records live in scratch; the initial rows and
 * the final report do not count.  Returns 0, or -1 when rows is outside
 * 1..max_rows.
 */
int oracle_stats_plan(int64_t rows, int64_t fan_in, int64_t max_rows,
                      int *merge_kernels, int64_t *scratch_elements,
                      int64_t *level_records /* at least 64 entries */)
{
    if (rows < 1 || rows > max_rows || fan_in < 2)
        return -1;
    int kernels = 0;
    int64_t scratch_records = 0;
    int64_t count = rows;
    do {
        count = (count + fan_in - 1) / fan_in;
        level_records[kernels++] = count;
        if (count > 1)
            scratch_records += count;
    } while (count > 1);
    *merge_kernels = kernels;
    *scratch_elements = 3 * scratch_records;
    return 0;
}

/*
 * The host decision after the report is read back ("训练与状态保存", "在 ruda:0 上
 * 进行原生 PyTorch 训练"): skip on any non-finite
 * value; otherwise the global L2 norm of the unscaled gradient and the clip
 * coefficient min(1, max_grad_norm / norm) (max_grad_norm <= 0: no clip).
 */
void oracle_clip_decision(double sum_sq, uint64_t nonfinite, double max_grad_norm,
                          int *skip, double *norm, double *coef)
{
    *skip = nonfinite > 0;
    *norm = sqrt(sum_sq);
    *coef = 1.0;
    if (!*skip && max_grad_norm > 0.0 && *norm > max_grad_norm)
        *coef = max_grad_norm / *norm;
}
