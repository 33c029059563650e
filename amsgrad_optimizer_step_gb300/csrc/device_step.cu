// The decision of a step whose count lives on the device (fa_device_step).
//
// One thread reads the step count and, when given, the 12-byte report of the
// gradient statistics, and takes the host path's decision with the host
// path's FP64 operations in the same order: a report that counts a non-finite
// value skips the step ("训练与状态保存", section "在 ruda:0 上进行原生 PyTorch
// 训练": the report is read back and a non-finite gradient skips the whole step);
// otherwise the norm of the unscaled gradient and, above max_grad_norm, the clip
// coefficient max_grad_norm / norm; then the step t+1, the bias corrections
// 1 - beta^(t+1) by binary exponentiation and the nine FP32 coefficients of the
// fused update ("実験的なデバイス上の融合 AdamW / AMSGrad", section "低レベルの使用":
// coefficients formed on the host in FP64 and passed to the kernel in FP32).
// Every operation is an explicitly rounded intrinsic, so nothing is contracted
// into a fused multiply-add and the FP32 coefficients equal the host's bit for
// bit (the host code is compiled without contraction as well).
#include <cuda_runtime.h>

#include "internal.h"

namespace fa {
namespace {

__device__ double pow_uint(double base, uint64_t t) {
    double r = 1.0;
    while (t) {
        if (t & 1) r = __dmul_rn(r, base);
        base = __dmul_rn(base, base);
        t >>= 1;
    }
    return r;
}

__global__ void decide_kernel(fa_device_step *d, const DecideArgs a) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    const uint64_t t = d->t;
    uint32_t nonfinite = 0;
    double norm = 0.0, coef = 1.0;
    bool skip = false;
    if (a.report) {
        const fa_stats r = *a.report;
        nonfinite = r.nonfinite;
        skip = nonfinite > 0;
        const double sum = __dadd_rn(static_cast<double>(r.sum_sq), static_cast<double>(r.sum_sq_lo));
        norm = __ddiv_rn(__dsqrt_rn(sum), a.scale);
        if (!skip && a.max_grad_norm > 0 && norm > a.max_grad_norm)
            coef = __ddiv_rn(a.max_grad_norm, norm);
    }
    d->skipped = skip ? 1u : 0u;
    d->nonfinite = nonfinite;
    d->grad_norm = norm;
    d->clip_coef = coef;
    if (skip) return;  // t and the coefficients stay as they were

    const uint64_t t_new = t + 1;
    const double bc1 = __dsub_rn(1.0, pow_uint(a.beta1, t_new));
    const double bc2 = __dsub_rn(1.0, pow_uint(a.beta2, t_new));
    float *w = reinterpret_cast<float *>(d->reserved);
    w[0] = __double2float_rn(a.beta1);
    w[1] = __double2float_rn(__dsub_rn(1.0, a.beta1));
    w[2] = __double2float_rn(a.beta2);
    w[3] = __double2float_rn(__dsub_rn(1.0, a.beta2));
    w[4] = __double2float_rn(__ddiv_rn(a.lr, bc1));
    w[5] = __double2float_rn(__ddiv_rn(1.0, bc2));
    w[6] = __double2float_rn(a.eps);
    w[7] = __double2float_rn(__dsub_rn(1.0, __dmul_rn(a.lr, a.weight_decay)));
    w[8] = __double2float_rn(__ddiv_rn(__dmul_rn(a.sign, coef), a.scale));
    d->reserved[kStepFirstWord] = t == 0 ? 1u : 0u;
    d->t = t_new;
}

}  // namespace

cudaError_t launch_device_step_decide(fa_device_step *dstep, const DecideArgs &a,
                                      cudaStream_t stream) {
    decide_kernel<<<1, 32, 0, stream>>>(dstep, a);
    return cudaGetLastError();
}

}  // namespace fa
