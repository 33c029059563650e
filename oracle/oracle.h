/* ORACLE -- TEST INFRASTRUCTURE ONLY.  Declarations shared by the two oracle C files. */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int32_t amsgrad, maximize;
} oracle_options;

double oracle_widen(const void *g, int dtype, int64_t i);
double oracle_int_pow(double beta, uint64_t t);

void oracle_adamw_update(int64_t n, const void *g, int gdtype,
                         const oracle_options *o, double gradient_scale,
                         double clip_coef, uint64_t t, int have_state, int round_fp32,
                         double *p, double *m, double *v, double *vmax);

uint16_t oracle_to_bf16(float x);
uint16_t oracle_to_f16(float x);
void oracle_model_copy(int64_t n, const float *p, int dtype, uint16_t *out);

void oracle_gradient_stats(int64_t n, const void *g, int gdtype, double gradient_scale,
                           double *sum_sq, uint64_t *nonfinite);
int64_t oracle_row_stats(int64_t n, const void *g, int gdtype, int64_t row_len,
                         const int64_t *seg, int64_t nseg,
                         double *row_sum_sq, uint64_t *row_nonfinite);
int oracle_stats_plan(int64_t rows, int64_t fan_in, int64_t max_rows,
                      int *merge_kernels, int64_t *scratch_elements,
                      int64_t *level_records);
void oracle_clip_decision(double sum_sq, uint64_t nonfinite, double max_grad_norm,
                          int *skip, double *norm, double *coef);

#endif
