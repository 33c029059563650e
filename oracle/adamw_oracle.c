/*
 * ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded FP64 restatement of the fused AdamW / AMSGrad
 * element update.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load this code; the product path never does.  It shares no source
 * with the CUDA library.
 *
 * Passages followed (RUDA documentation pages):
 *   - "実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw), section
 *     "この演算子を使用する理由": the per-element formula block, the AMSGrad max of
 *     the uncorrected second moment, epsilon outside the square root, decay never
 *     added to the gradient, host bias-correction coefficients from FP64 integer
 *     powers, and the defaults beta=(0.9,0.999), epsilon=1e-5, weight_decay=1e-4.
 *   - "实验性融合 AdamW / AMSGrad" (zh/docs/fused-adamw), section "增加的实际能力":
 *     FP32 parameters and moments, FP32/FP16/BF16 gradients, maximize, first
 *     update initialises the moments without reading them, empty tensor or
 *     skip_update changes nothing and does not advance the step count.
 *
 * Arithmetic is FP64 throughout.  The caller chooses whether state is kept in
 * FP64 between calls (for the closed-form pins) or rounded to FP32 after every
 * call (as the device stores it).  Build with -ffp-contract=off so that no
 * multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

/* ---- exact widening of the stored gradient --------------------------------- */

static double widen_f32(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* BF16 is the upper half of an FP32 pattern. */
static double widen_bf16(uint16_t bits)
{
    return widen_f32((uint32_t)bits << 16);
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t bits)
{
    int sign = bits >> 15;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac + 1024), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* Element i of a stored gradient widened exactly to FP64 ("实验性融合 AdamW /
 * AMSGrad", "增加的实际能力": gradients are FP32, FP16 or BF16). */
double oracle_widen(const void *g, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32) {
        uint32_t b;
        memcpy(&b, (const char *)g + 4 * i, 4);
        return widen_f32(b);
    }
    uint16_t h;
    memcpy(&h, (const char *)g + 2 * i, 2);
    return dtype == ORACLE_BF16 ? widen_bf16(h) : widen_f16(h);
}

/* ---- host coefficients ------------------------------------------------------ */

/* beta^t by repeated multiplication in FP64 ("実験的なデバイス上の融合 AdamW / AMSGrad",
 * "この演算子を使用する理由": the host forms the bias corrections from FP64 integer
 * powers). */
double oracle_int_pow(double beta, uint64_t t)
{
    double r = 1.0;
    for (uint64_t k = 0; k < t; ++k)
        r *= beta;
    return r;
}

/* max() that returns NaN when either operand is NaN. */
static double max_propagate_nan(double a, double b)
{
    if (isnan(a) || isnan(b))
        return NAN;
    return a > b ? a : b;
}

static double store(double x, int round_fp32)
{
    return round_fp32 ? (double)(float)x : x;
}

/*
 * One update call ("実験的なデバイス上の融合 AdamW / AMSGrad", "この演算子を使用する理由":
 * the per-element formula block; "实验性融合 AdamW / AMSGrad", "增加的实际能力":
 * maximize and the first update).  ``t`` is the 1-based step of this update (already
 * advanced by the caller).  ``have_state`` = 0 is the first update: the old
 * moments are taken as zero and the m/v/vmax arrays are only written.
 * ``clip_coef`` multiplies the unscaled gradient (1 = no clipping).
 */
void oracle_adamw_update(int64_t n, const void *g, int gdtype,
                         const oracle_options *o, double gradient_scale,
                         double clip_coef, uint64_t t, int have_state, int round_fp32,
                         double *p, double *m, double *v, double *vmax)
{
    const double bc1 = 1.0 - oracle_int_pow(o->beta1, t);
    const double bc2 = 1.0 - oracle_int_pow(o->beta2, t);

    for (int64_t i = 0; i < n; ++i) {
        double grad = oracle_widen(g, gdtype, i) / gradient_scale;
        if (o->maximize)
            grad = -grad;
        grad = grad * clip_coef;

        double m_old = have_state ? m[i] : 0.0;
        double v_old = have_state ? v[i] : 0.0;

        double m_new = o->beta1 * m_old + (1.0 - o->beta1) * grad;
        double v_new = o->beta2 * v_old + (1.0 - o->beta2) * grad * grad;

        double v_used = v_new;
        if (o->amsgrad) {
            double vmax_old = have_state ? vmax[i] : 0.0;
            double vmax_new = max_propagate_nan(vmax_old, v_new);
            vmax[i] = store(vmax_new, round_fp32);
            v_used = vmax_new;
        }

        double p_new = p[i] * (1.0 - o->lr * o->weight_decay)
                     - o->lr * (m_new / bc1) / (sqrt(v_used / bc2) + o->eps);

        p[i] = store(p_new, round_fp32);
        m[i] = store(m_new, round_fp32);
        v[i] = store(v_new, round_fp32);
    }
}

/* ---- low-precision model copy ------------------------------------------------
 *
 * "训练与状态保存" (zh/docs/training), section "FP32 主参数与混合参数存储": the FP32
 * master is updated in FP32 and the parameter is handed back in its storage
 * dtype; "实验性融合 AdamW / AMSGrad", section "增加的实际能力": the low-precision
 * write-back is the caller's job in the plain step.  The copy is the stored
 * FP32 master value rounded to nearest, ties to even, in the target format.
 *
 * Written from the format definitions: a finite non-zero x with binary
 * exponent e (2^e <= |x| < 2^(e+1)) has quantum 2^(e - (p - 1)) for p
 * significant bits in the normal range and the fixed subnormal quantum
 * below it; x / quantum is exact in FP64, rint() rounds it to the nearest
 * integer with ties to even, and a result at or above 2^(emax+1) overflows
 * to infinity.
 */
static double round_to_format(double x, int sig_bits, int emin, int emax)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e;
    frexp(x, &e);          /* |x| = f * 2^e, 0.5 <= f < 1 */
    e -= 1;                /* now 2^e <= |x| < 2^(e+1) */
    int qexp = (e < emin ? emin : e) - (sig_bits - 1);
    double q = ldexp(1.0, qexp);
    double y = rint(x / q) * q;
    if (fabs(y) >= ldexp(1.0, emax + 1))
        return x > 0 ? INFINITY : -INFINITY;
    return y;
}

/* BF16: 8 significant bits, exponents -126..127 (same range as FP32).  The model
 * copies follow "训练与状态保存", "FP32 主参数与混合参数存储" (parameters return in their
 * storage dtype); the pages name no rounding, and round-to-nearest-even, the IEEE
 * default, is the reading taken. */
uint16_t oracle_to_bf16(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    if (isnan(x))
        return (uint16_t)((b >> 16) | 0x40);            /* a quiet NaN */
    double y = round_to_format((double)x, 8, -126, 127);
    float yf = (float)y;                                 /* exact: y is a BF16 value */
    memcpy(&b, &yf, 4);
    return (uint16_t)(b >> 16);
}

/* IEEE binary16: 11 significant bits, exponents -14..15, subnormal quantum 2^-24. */
uint16_t oracle_to_f16(float x)
{
    if (isnan(x))
        return 0x7e00;
    double y = round_to_format((double)x, 11, -14, 15);
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    double a = fabs(y);
    if (isinf(a))
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14))                             /* subnormal or zero */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    int e;
    double f = frexp(a, &e);                             /* a = f * 2^e, 0.5 <= f < 1 */
    uint16_t expo = (uint16_t)(e - 1 + 15);
    uint16_t frac = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(expo << 10) | frac;
}

/* Model copies of n FP32 values: dtype ORACLE_BF16 or ORACLE_F16 ("训练与状态保存",
 * "FP32 主参数与混合参数存储"; rounding to nearest even). */
void oracle_model_copy(int64_t n, const float *p, int dtype, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == ORACLE_BF16 ? oracle_to_bf16(p[i]) : oracle_to_f16(p[i]);
}
