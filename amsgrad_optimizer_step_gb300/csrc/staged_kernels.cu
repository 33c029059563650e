// The staged AdamW / AMSGrad update: the benchmark-only comparison the pages
// describe ("実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw), section
// "割り当てとパフォーマンスのモデル"; "实验性融合 AdamW / AMSGrad", section "优化点与边界":
// an explicit staged baseline of 4 kernels, 5 with AMSGrad, with repeated
// gradient reads and a delta buffer, 48 and 60 bytes per parameter for FP32
// gradients in steady state, against 28 and 36 for the fused update).
//
// The split used here (the pages give only the totals):
//   1. m     = beta1*m + (1-beta1)*g          reads g, m      writes m
//   2. v     = beta2*v + (1-beta2)*g*g        reads g, v      writes v
//   3. vmax  = max(vmax, v)  (AMSGrad)        reads v, vmax   writes vmax
//   4. delta = step*m / (sqrt(v_used*rbc2)+eps)  reads m, v_used  writes delta
//   5. p     = p*decay - delta                reads p, delta  writes p
// FP32 gradients: 12 + 12 + (12) + 12 + 12 = 48 (60) bytes per parameter.  Each
// stage evaluates exactly the fused kernel's FP32 operations, so the two paths
// agree bit for bit.  Every stage is a grid-stride kernel over 4-element
// vectors (16-byte loads/stores) with a scalar tail.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace fa {
namespace {

FA_BOUNDS_COUNTER(g_staged_oob)

template <int GT>
__device__ __forceinline__ float grad1(const void *g, int64_t i) {
    if (GT == FA_F32) return __ldcs(static_cast<const float *>(g) + i);
    const unsigned short h = __ldcs(static_cast<const unsigned short *>(g) + i);
    if (GT == FA_BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
    return __half2float(__ushort_as_half(h));
}

template <int GT>
__device__ __forceinline__ float4 grad4(const void *g, int64_t i) {
    if (GT == FA_F32) return __ldcs(reinterpret_cast<const float4 *>(static_cast<const float *>(g) + i));
    const uint2 r = __ldcs(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(g) + i));
    if (GT == FA_BF16)
        return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                           __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Grid-stride loop: vector body over 4-element groups, then the scalar tail.
template <typename FV, typename FS>
__device__ __forceinline__ void grid_stride_vec4(int64_t n, FV body_vec, FS body_scalar) {
    const int64_t nv = n / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t q = first; q < nv; q += stride)
        if (fa_in_bounds(4 * q, 4, n)) body_vec(4 * q);
    for (int64_t i = 4 * nv + first; i < n; i += stride)
        if (fa_in_bounds(i, 1, n)) body_scalar(i);
}

// Stage 1: m = beta1*m + (1-beta1)*g   (first step: m = (1-beta1)*g, m not read)
template <int GT, bool FIRST>
__global__ void __launch_bounds__(kThreads) stage_m(const void *g, float *m, Coef c, int64_t n) {
    grid_stride_vec4(n, [&](int64_t i) {
        const float4 x = grad4<GT>(g, i);
        const float gg[4] = {x.x * c.gmul, x.y * c.gmul, x.z * c.gmul, x.w * c.gmul};
        float4 mo = FIRST ? make_float4(0.f, 0.f, 0.f, 0.f)
                          : __ldcs(reinterpret_cast<const float4 *>(m + i));
        float r[4] = {mo.x, mo.y, mo.z, mo.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = FIRST ? c.omb1 * gg[k] : fmaf(c.b1, r[k], c.omb1 * gg[k]);
        __stcs(reinterpret_cast<float4 *>(m + i), make_float4(r[0], r[1], r[2], r[3]));
    }, [&](int64_t i) {
        const float gg = grad1<GT>(g, i) * c.gmul;
        m[i] = FIRST ? c.omb1 * gg : fmaf(c.b1, m[i], c.omb1 * gg);
    });
}

// Stage 2: v = beta2*v + (1-beta2)*g*g
template <int GT, bool FIRST>
__global__ void __launch_bounds__(kThreads) stage_v(const void *g, float *v, Coef c, int64_t n) {
    grid_stride_vec4(n, [&](int64_t i) {
        const float4 x = grad4<GT>(g, i);
        const float gg[4] = {x.x * c.gmul, x.y * c.gmul, x.z * c.gmul, x.w * c.gmul};
        float4 vo = FIRST ? make_float4(0.f, 0.f, 0.f, 0.f)
                          : __ldcs(reinterpret_cast<const float4 *>(v + i));
        float r[4] = {vo.x, vo.y, vo.z, vo.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            r[k] = FIRST ? (c.omb2 * gg[k]) * gg[k] : fmaf(c.b2, r[k], (c.omb2 * gg[k]) * gg[k]);
        __stcs(reinterpret_cast<float4 *>(v + i), make_float4(r[0], r[1], r[2], r[3]));
    }, [&](int64_t i) {
        const float gg = grad1<GT>(g, i) * c.gmul;
        v[i] = FIRST ? (c.omb2 * gg) * gg : fmaf(c.b2, v[i], (c.omb2 * gg) * gg);
    });
}

__device__ __forceinline__ float max_keep_nan(float vmax_old, float v) {
    return (v > vmax_old || v != v) ? v : vmax_old;
}

// Stage 3 (AMSGrad): vmax = max(vmax, v)   (first step: vmax = max(0, v))
template <bool FIRST>
__global__ void __launch_bounds__(kThreads) stage_vmax(const float *v, float *vmax, int64_t n) {
    grid_stride_vec4(n, [&](int64_t i) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(v + i));
        const float4 b = FIRST ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : __ldcs(reinterpret_cast<const float4 *>(vmax + i));
        __stcs(reinterpret_cast<float4 *>(vmax + i),
               make_float4(max_keep_nan(b.x, a.x), max_keep_nan(b.y, a.y),
                           max_keep_nan(b.z, a.z), max_keep_nan(b.w, a.w)));
    }, [&](int64_t i) {
        vmax[i] = max_keep_nan(FIRST ? 0.f : vmax[i], v[i]);
    });
}

// Stage 4: delta = step_size*m / (sqrt(v_used*rbc2) + eps)
__global__ void __launch_bounds__(kThreads)
stage_delta(const float *m, const float *v_used, float *delta, Coef c, int64_t n) {
    grid_stride_vec4(n, [&](int64_t i) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(m + i));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(v_used + i));
        const float mm[4] = {a.x, a.y, a.z, a.w};
        const float vv[4] = {b.x, b.y, b.z, b.w};
        float d[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) d[k] = (c.step_size * mm[k]) / (sqrtf(vv[k] * c.rbc2) + c.eps);
        __stcs(reinterpret_cast<float4 *>(delta + i), make_float4(d[0], d[1], d[2], d[3]));
    }, [&](int64_t i) {
        delta[i] = (c.step_size * m[i]) / (sqrtf(v_used[i] * c.rbc2) + c.eps);
    });
}

// Stage 5: p = p*decay - delta
__global__ void __launch_bounds__(kThreads)
stage_p(float *p, const float *delta, Coef c, int64_t n) {
    grid_stride_vec4(n, [&](int64_t i) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p + i));
        const float4 d = __ldcs(reinterpret_cast<const float4 *>(delta + i));
        __stcs(reinterpret_cast<float4 *>(p + i),
               make_float4(fmaf(a.x, c.decay, -d.x), fmaf(a.y, c.decay, -d.y),
                           fmaf(a.z, c.decay, -d.z), fmaf(a.w, c.decay, -d.w)));
    }, [&](int64_t i) {
        p[i] = fmaf(p[i], c.decay, -delta[i]);
    });
}

template <typename K>
int grid_for(K kernel, int64_t n, int dev) {
    const int64_t need = (n / 4 + kThreads - 1) / kThreads;
    return persistent_grid(kernel, need > 0 ? need : 1, dev);
}

template <int GT, bool FIRST>
cudaError_t launch_staged_t(const StagedArgs &a, const Coef &c, bool ams, cudaStream_t s) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    auto km = stage_m<GT, FIRST>;
    km<<<grid_for(km, a.n, dev), kThreads, 0, s>>>(a.g, a.m, c, a.n);
    auto kv = stage_v<GT, FIRST>;
    kv<<<grid_for(kv, a.n, dev), kThreads, 0, s>>>(a.g, a.v, c, a.n);
    if (ams) {
        auto kx = stage_vmax<FIRST>;
        kx<<<grid_for(kx, a.n, dev), kThreads, 0, s>>>(a.v, a.vmax, a.n);
    }
    stage_delta<<<grid_for(stage_delta, a.n, dev), kThreads, 0, s>>>(a.m, ams ? a.vmax : a.v,
                                                                      a.delta, c, a.n);
    stage_p<<<grid_for(stage_p, a.n, dev), kThreads, 0, s>>>(a.p, a.delta, c, a.n);
    return cudaGetLastError();
}

template <int GT>
cudaError_t launch_staged_gt(const StagedArgs &a, const Coef &c, bool ams, bool first,
                             cudaStream_t s) {
    return first ? launch_staged_t<GT, true>(a, c, ams, s) : launch_staged_t<GT, false>(a, c, ams, s);
}

}  // namespace

cudaError_t staged_bounds_violations(unsigned long long *count, bool clear) {
#if FA_BOUNDS_CHECK
    cudaError_t err = cudaMemcpyFromSymbol(count, g_staged_oob, sizeof(*count));
    if (err != cudaSuccess || !clear) return err;
    const unsigned long long zero = 0;
    return cudaMemcpyToSymbol(g_staged_oob, &zero, sizeof(zero));
#else
    (void)clear;
    *count = 0;
    return cudaSuccess;
#endif
}

cudaError_t launch_staged(const StagedArgs &a, const Coef &c, fa_dtype gdt, bool amsgrad,
                          bool first, cudaStream_t stream) {
    switch (gdt) {
        case FA_F32: return launch_staged_gt<FA_F32>(a, c, amsgrad, first, stream);
        case FA_F16: return launch_staged_gt<FA_F16>(a, c, amsgrad, first, stream);
        case FA_BF16: return launch_staged_gt<FA_BF16>(a, c, amsgrad, first, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
