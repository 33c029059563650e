// Fused AdamW / AMSGrad element update for sm_103a.
//
// Follows RUDA "実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw), section
// "この演算子を使用する理由" (the per-element formula block: unscale, optional
// negation, first and second moments, optional AMSGrad max of the uncorrected
// second moment, decoupled decay, bias-corrected step with epsilon outside the
// square root; FP32 device arithmetic, fusion allowed) and "实验性融合 AdamW /
// AMSGrad" (zh/docs/fused-adamw), section "增加的实际能力" (FP32 parameters and
// moments, FP32/FP16/BF16 gradients, the first update initialises the moments
// inside the kernel without reading them).
//
// Design: one HBM pass per parameter.  The kernel is bandwidth bound (about
// 0.7 flop per byte), so it is built for bytes in flight: persistent CTAs,
// grid-stride over 8-element vectors, every stream moved with 16-byte
// evict-first loads and stores (p, m, v, vmax as two float4; a BF16/FP16
// gradient as one 16-byte word, an FP32 gradient as two float4), all loads of
// an iteration issued before any arithmetic.  Elements before the first
// 16-byte boundary and after the last full vector go through the same
// arithmetic one at a time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

// Tuning knobs (compile-time): vectors per thread per iteration, threads per
// CTA, and an L2 256-byte prefetch hint on the vector loads.
#ifndef FA_UPDATE_UNROLL
#define FA_UPDATE_UNROLL 2
#endif
#ifndef FA_UPDATE_THREADS
#define FA_UPDATE_THREADS 512
#endif
#ifndef FA_UPDATE_L2_PREFETCH
#define FA_UPDATE_L2_PREFETCH 0
#endif

namespace fa {
namespace {

constexpr int kVec = 8;  // elements per vector
constexpr int kUThreads = FA_UPDATE_THREADS;

// 16-byte evict-first loads of the vector body.
__device__ __forceinline__ float4 ld16(const float4 *q) {
#if FA_UPDATE_L2_PREFETCH
    float4 r;
    asm volatile("ld.global.cs.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(q));
    return r;
#else
    return __ldcs(q);
#endif
}

__device__ __forceinline__ uint4 ld16(const uint4 *q) {
#if FA_UPDATE_L2_PREFETCH
    uint4 r;
    asm volatile("ld.global.cs.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(q));
    return r;
#else
    return __ldcs(q);
#endif
}

// ---- stored-gradient widening ------------------------------------------------

template <int GT>
struct GradIO;

template <>
struct GradIO<FA_F32> {
    static __device__ __forceinline__ void load8(const void *g, int64_t i, float (&x)[kVec]) {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(g) + i);
        float4 a = ld16(q);
        float4 b = ld16(q + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        return __ldcs(static_cast<const float *>(g) + i);
    }
};

// BF16 is the upper half of an FP32 pattern: widening is a shift.
template <>
struct GradIO<FA_BF16> {
    static __device__ __forceinline__ void load8(const void *g, int64_t i, float (&x)[kVec]) {
        uint4 r = ld16(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + i));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        unsigned short h = __ldcs(static_cast<const unsigned short *>(g) + i);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
};

template <>
struct GradIO<FA_F16> {
    static __device__ __forceinline__ void load8(const void *g, int64_t i, float (&x)[kVec]) {
        uint4 r = ld16(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + i));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h2 = *reinterpret_cast<const __half2 *>(&w[k]);
            float2 f = __half22float2(h2);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        unsigned short h = __ldcs(static_cast<const unsigned short *>(g) + i);
        return __half2float(__ushort_as_half(h));
    }
};

// ---- the element update ------------------------------------------------------

// AMSGrad max that returns NaN when either operand is NaN.
__device__ __forceinline__ float max_keep_nan(float vmax_old, float v) {
    return (v > vmax_old || v != v) ? v : vmax_old;
}

template <bool AMS, bool FIRST>
__device__ __forceinline__ void adamw_element(const Coef &c, float x, float &p, float &m,
                                              float &v, float &vmax) {
    const float g = x * c.gmul;
    float m_new, v_new;
    if (FIRST) {  // state None: old moments are zero and are not read
        m_new = c.omb1 * g;
        v_new = (c.omb2 * g) * g;
    } else {
        m_new = fmaf(c.b1, m, c.omb1 * g);
        v_new = fmaf(c.b2, v, (c.omb2 * g) * g);
    }
    float v_used = v_new;
    if (AMS) {
        const float mx = FIRST ? max_keep_nan(0.0f, v_new) : max_keep_nan(vmax, v_new);
        vmax = mx;
        v_used = mx;
    }
    const float denom = sqrtf(v_used * c.rbc2) + c.eps;
    p = fmaf(p, c.decay, -(c.step_size * m_new) / denom);
    m = m_new;
    v = v_new;
}

__device__ __forceinline__ void load8f(const float *base, int64_t i, float (&x)[kVec]) {
    const float4 *q = reinterpret_cast<const float4 *>(base + i);
    float4 a = ld16(q);
    float4 b = ld16(q + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store8f(float *base, int64_t i, const float (&x)[kVec]) {
    float4 *q = reinterpret_cast<float4 *>(base + i);
    __stcs(q, make_float4(x[0], x[1], x[2], x[3]));
    __stcs(q + 1, make_float4(x[4], x[5], x[6], x[7]));
}

// Low-precision model copy of the updated FP32 parameter: round to nearest,
// ties to even ("训练与状态保存", section "FP32 主参数与混合参数存储": the FP32 master
// is updated and the parameter is returned in its storage dtype).
template <int MD>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if (MD == FA_BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int MD>
__device__ __forceinline__ void store8_model(void *base, int64_t i, const float (&x)[kVec]) {
    uint4 w;
    w.x = pack2<MD>(x[0], x[1]);
    w.y = pack2<MD>(x[2], x[3]);
    w.z = pack2<MD>(x[4], x[5]);
    w.w = pack2<MD>(x[6], x[7]);
    __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + i), w);
}

template <int MD>
__device__ __forceinline__ void store1_model(void *base, int64_t i, float x) {
    unsigned short h;
    if (MD == FA_BF16) h = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else h = __half_as_ushort(__float2half_rn(x));
    __stcs(static_cast<unsigned short *>(base) + i, h);
}

template <int GT, bool AMS, bool FIRST, int MD>
__device__ __forceinline__ void scalar_element(const UpdateArgs &a, const Coef &c, int64_t i) {
    float x = GradIO<GT>::load1(a.g, i);
    float p = __ldcs(a.p_in + i);
    float m = 0.f, v = 0.f, vm = 0.f;
    if (!FIRST) {
        m = __ldcs(a.m_in + i);
        v = __ldcs(a.v_in + i);
        if (AMS) vm = __ldcs(a.vmax_in + i);
    }
    adamw_element<AMS, FIRST>(c, x, p, m, v, vm);
    __stcs(a.p_out + i, p);
    __stcs(a.m_out + i, m);
    __stcs(a.v_out + i, v);
    if (AMS) __stcs(a.vmax_out + i, vm);
    if (MD != kNoModel) store1_model<MD>(a.p_model, i, p);
}

// Vector body + scalar head/tail.  Each thread owns UNROLL vectors per
// grid-stride iteration, spaced kThreads vectors apart so that a warp's
// accesses to each stream are contiguous.
template <int GT, bool AMS, bool FIRST, int UNROLL, int MD>
__global__ void __launch_bounds__(kUThreads)
update_vec_kernel(const UpdateArgs a, const Coef c) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kUThreads + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kUThreads * UNROLL;

    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kUThreads * UNROLL + threadIdx.x;
         base < a.nvec; base += stride) {
        float x[UNROLL][kVec], p[UNROLL][kVec], m[UNROLL][kVec], v[UNROLL][kVec],
            vm[UNROLL][kVec];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t vi = base + static_cast<int64_t>(u) * kUThreads;
            if (vi < a.nvec) {
                const int64_t e = a.head + vi * kVec;
                GradIO<GT>::load8(a.g, e, x[u]);
                load8f(a.p_in, e, p[u]);
                if (!FIRST) {
                    load8f(a.m_in, e, m[u]);
                    load8f(a.v_in, e, v[u]);
                    if (AMS) load8f(a.vmax_in, e, vm[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t vi = base + static_cast<int64_t>(u) * kUThreads;
            if (vi < a.nvec) {
                const int64_t e = a.head + vi * kVec;
#pragma unroll
                for (int k = 0; k < kVec; ++k)
                    adamw_element<AMS, FIRST>(c, x[u][k], p[u][k], m[u][k], v[u][k], vm[u][k]);
                store8f(a.p_out, e, p[u]);
                store8f(a.m_out, e, m[u]);
                store8f(a.v_out, e, v[u]);
                if (AMS) store8f(a.vmax_out, e, vm[u]);
                if (MD != kNoModel) store8_model<MD>(a.p_model, e, p[u]);
            }
        }
    }

    // Scalar head [0, head) and tail [head + 8*nvec, n).
    if (tid < a.head) scalar_element<GT, AMS, FIRST, MD>(a, c, tid);
    const int64_t tail0 = a.head + a.nvec * kVec;
    if (tid < a.n - tail0) scalar_element<GT, AMS, FIRST, MD>(a, c, tail0 + tid);
}

// Every element one at a time (pointers not co-aligned to 16 bytes).
template <int GT, bool AMS, bool FIRST, int MD>
__global__ void __launch_bounds__(kThreads)
update_scalar_kernel(const UpdateArgs a, const Coef c) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < a.n;
         i += stride)
        scalar_element<GT, AMS, FIRST, MD>(a, c, i);
}

constexpr int kUnroll = FA_UPDATE_UNROLL;

template <int GT, bool AMS, bool FIRST, int MD>
cudaError_t launch_typed(const UpdateArgs &a, const Coef &c, bool vector_ok,
                         cudaStream_t stream) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (sm_count(dev) <= 0) return cudaErrorInvalidDevice;

    if (vector_ok) {
        auto kern = update_vec_kernel<GT, AMS, FIRST, kUnroll, MD>;
        const int64_t per_cta = static_cast<int64_t>(kUThreads) * kUnroll;
        int64_t need = (a.nvec + per_cta - 1) / per_cta;
        if (need == 0 && a.n > 0) need = 1;  // head/tail elements only
        const int grid = persistent_grid(kern, need, dev, kUThreads);
        if (grid == 0) return cudaSuccess;
        kern<<<grid, kUThreads, 0, stream>>>(a, c);
    } else {
        auto kern = update_scalar_kernel<GT, AMS, FIRST, MD>;
        const int grid = persistent_grid(kern, (a.n + kThreads - 1) / kThreads, dev);
        if (grid == 0) return cudaSuccess;
        kern<<<grid, kThreads, 0, stream>>>(a, c);
    }
    return cudaGetLastError();
}

template <int GT, int MD>
cudaError_t launch_md(const UpdateArgs &a, const Coef &c, bool ams, bool first, bool vec,
                      cudaStream_t s) {
    if (ams)
        return first ? launch_typed<GT, true, true, MD>(a, c, vec, s)
                     : launch_typed<GT, true, false, MD>(a, c, vec, s);
    return first ? launch_typed<GT, false, true, MD>(a, c, vec, s)
                 : launch_typed<GT, false, false, MD>(a, c, vec, s);
}

template <int GT>
cudaError_t launch_gt(const UpdateArgs &a, const Coef &c, bool ams, bool first, bool vec,
                      int model_dtype, cudaStream_t s) {
    switch (model_dtype) {
        case kNoModel: return launch_md<GT, kNoModel>(a, c, ams, first, vec, s);
        case FA_F16: return launch_md<GT, FA_F16>(a, c, ams, first, vec, s);
        case FA_BF16: return launch_md<GT, FA_BF16>(a, c, ams, first, vec, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_update(const UpdateArgs &a, const Coef &c, fa_dtype gdt, bool amsgrad,
                          bool first, bool vector_ok, int model_dtype, cudaStream_t stream) {
    switch (gdt) {
        case FA_F32:
            return launch_gt<FA_F32>(a, c, amsgrad, first, vector_ok, model_dtype, stream);
        case FA_F16:
            return launch_gt<FA_F16>(a, c, amsgrad, first, vector_ok, model_dtype, stream);
        case FA_BF16:
            return launch_gt<FA_BF16>(a, c, amsgrad, first, vector_ok, model_dtype, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
