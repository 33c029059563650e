/*
 * A plain C program that uses the library through include/fused_adamw.h only:
 * device buffers from the CUDA runtime, three statistics-guarded steps of the
 * fused AdamW update (analysis, merge, report, skip/clip decision, update) on
 * n FP32 parameters with FP32 gradients, the second call carrying a +Inf, then
 * the final p, m, v and the three step reports written to a binary file.
 *
 * Inputs are integer hashes scaled by powers of two, exact in FP32, so the test
 * that runs this program can rebuild them bit for bit.  With "gated", every step
 * goes through fa_bucket_step_clipped_gated (the update decides on the device)
 * instead of fa_bucket_step_clipped; with "descriptor", every step is composed
 * from the separate calls: fa_analyze_gradient, fa_merge_gradient_stats,
 * fa_bucket_update with the device report, fa_read_report, fa_stats_sum_sq and
 * fa_clip_decision.  The results must be the same bits in every mode.
 *
 *   consumer <n> <output file> [gated | descriptor]
 */
#include <string.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "fused_adamw.h"

static uint32_t mix(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

/* a value in [-scale, scale) with 16 significant bits: exact in FP32 */
static float sample(uint32_t stream, uint32_t i, float scale) {
    const int32_t u = (int32_t)(mix(mix(stream) ^ i) >> 16) - 32768;
    return (float)u / 32768.0f * scale;
}

#define CHECK_CUDA(x)                                                          \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));           \
            return 2;                                                          \
        }                                                                      \
    } while (0)

#define CHECK_FA(x)                                                            \
    do {                                                                       \
        fa_status s_ = (x);                                                    \
        if (s_ != FA_OK) {                                                     \
            fprintf(stderr, "%s: %s\n", #x, fa_status_string(s_));             \
            return 3;                                                          \
        }                                                                      \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 3 && !(argc == 4 && (strcmp(argv[3], "gated") == 0 ||
                                     strcmp(argv[3], "descriptor") == 0))) {
        fprintf(stderr, "usage: consumer <n> <output file> [gated | descriptor]\n");
        return 1;
    }
    const int gated = argc == 4 && strcmp(argv[3], "gated") == 0;
    const int descriptor = argc == 4 && strcmp(argv[3], "descriptor") == 0;
    const int64_t n = atoll(argv[1]);
    if (n < 2) return 1;
    const int32_t row_len = 256;
    if (fa_abi_version() != FA_ABI_VERSION) return 4;

    int64_t rows = 0, scratch_elems = 0;
    int32_t merge_kernels = 0;
    CHECK_FA(fa_stats_rows(n, row_len, NULL, 0, &rows));
    CHECK_FA(fa_stats_plan(rows, &merge_kernels, &scratch_elems));

    float *h = (float *)malloc((size_t)n * sizeof(float));
    float *p, *g, *m, *v, *scratch = NULL;
    fa_stats *rows_buf, *report;
    CHECK_CUDA(cudaMalloc((void **)&p, (size_t)n * 4));
    CHECK_CUDA(cudaMalloc((void **)&g, (size_t)n * 4));
    CHECK_CUDA(cudaMalloc((void **)&m, (size_t)n * 4));
    CHECK_CUDA(cudaMalloc((void **)&v, (size_t)n * 4));
    CHECK_CUDA(cudaMalloc((void **)&rows_buf, (size_t)rows * sizeof(fa_stats)));
    CHECK_CUDA(cudaMalloc((void **)&report, sizeof(fa_stats)));
    if (scratch_elems > 0) CHECK_CUDA(cudaMalloc((void **)&scratch, (size_t)scratch_elems * 4));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    fa_report_mailbox *mailbox = NULL; /* pinned host memory the device posts the report to */
    CHECK_CUDA(cudaHostAlloc((void **)&mailbox, sizeof *mailbox, cudaHostAllocDefault));

    for (int64_t i = 0; i < n; ++i) h[i] = sample(1u, (uint32_t)i, 0.03125f);
    CHECK_CUDA(cudaMemcpy(p, h, (size_t)n * 4, cudaMemcpyHostToDevice));

    fa_options o = fa_options_default();
    o.lr = 1e-3;
    o.amsgrad = 0;
    fa_step_control ctl;
    ctl.gradient_scale = 4.0;
    ctl.skip_update = 0;
    uint64_t t = 0;
    fa_step_report reps[3];
    for (int call = 1; call <= 3; ++call) {
        for (int64_t i = 0; i < n; ++i) h[i] = sample(100u + (uint32_t)call, (uint32_t)i, 0.0625f);
        if (call == 2) h[n / 2] = 1.0f / 0.0f; /* +Inf: this step is skipped */
        CHECK_CUDA(cudaMemcpy(g, h, (size_t)n * 4, cudaMemcpyHostToDevice));
        if (descriptor) {
            /* the step from the separate calls; the update decides on the device */
            CHECK_FA(fa_analyze_gradient(g, FA_F32, n, row_len, NULL, 0, rows_buf, rows, stream));
            CHECK_FA(fa_merge_gradient_stats(rows_buf, rows, scratch, scratch_elems, report,
                                             stream));
            fa_bucket_update_args u;
            memset(&u, 0, sizeof u);
            u.n_total = n;
            u.p = p;
            u.g = g;
            u.gdt = FA_F32;
            u.m = m;
            u.v = v;
            u.t = t;
            u.grad_mult = 1.0;
            u.report = report;
            u.max_grad_norm = 0.5;
            u.model_dtype = FA_BF16;
            int32_t enqueued = 0;
            CHECK_FA(fa_bucket_update(&u, &o, ctl, &enqueued, stream));
            fa_stats h;
            double sum = 0.0, norm = 0.0, coef = 1.0;
            int32_t skip = 0;
            CHECK_FA(fa_read_report(report, &h, stream));
            CHECK_FA(fa_stats_sum_sq(&h, &sum));
            CHECK_FA(fa_clip_decision(sum, h.nonfinite, ctl.gradient_scale, 0.5, &skip, &norm,
                                      &coef));
            fa_step_report r;
            memset(&r, 0, sizeof r);
            r.updated = enqueued && !skip;
            r.skipped_nonfinite = skip;
            r.nonfinite = h.nonfinite;
            r.grad_norm = norm;
            r.clip_coef = coef;
            reps[call - 1] = r;
            if (!skip) t += 1;
        } else if (gated)
            CHECK_FA(fa_bucket_step_clipped_gated(NULL, 0, n, p, g, FA_F32, m, v, NULL, &t, &o,
                                                  ctl, 0.5, row_len, rows_buf, rows, scratch,
                                                  scratch_elems, report, mailbox,
                                                  &reps[call - 1], stream));
        else
            CHECK_FA(fa_bucket_step_clipped(NULL, 0, n, p, g, FA_F32, m, v, NULL, &t, &o, ctl,
                                            0.5, row_len, rows_buf, rows, scratch,
                                            scratch_elems, report, &reps[call - 1], stream));
    }
    CHECK_CUDA(cudaStreamSynchronize(stream));

    FILE *f = fopen(argv[2], "wb");
    if (!f) return 5;
    fwrite(&t, sizeof t, 1, f);
    fwrite(reps, sizeof reps, 1, f);
    float *bufs[3] = {p, m, v};
    for (int k = 0; k < 3; ++k) {
        CHECK_CUDA(cudaMemcpy(h, bufs[k], (size_t)n * 4, cudaMemcpyDeviceToHost));
        fwrite(h, 4, (size_t)n, f);
    }
    fclose(f);
    cudaFree(p);
    cudaFree(g);
    cudaFree(m);
    cudaFree(v);
    cudaFree(rows_buf);
    cudaFree(report);
    cudaFree(scratch);
    cudaStreamDestroy(stream);
    cudaFreeHost(mailbox);
    free(h);
    return 0;
}
