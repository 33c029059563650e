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
// Design: one HBM pass per parameter.  The update is bandwidth bound (about
// 0.7 flop per byte), so it is built for bytes in flight.  Three kernels share the
// element arithmetic:
//   - update_vec_kernel: 8-element vectors, every stream moved with 16-byte
//     evict-first loads and stores (p, m, v, vmax as two float4; a BF16/FP16
//     gradient as one 16-byte word, an FP32 gradient as two float4), all loads of
//     an iteration issued before any arithmetic.  A launch with its multiplier
//     from the host runs a full grid of 64-thread CTAs, each covering one stretch
//     of 1024 elements;
//   - update_vec_cta_gate_kernel: the same full grid for a gated launch whose
//     gradient scale is a power of two, thread 0 of each CTA taking the decision
//     (with multiplications by the exact inverse scale) while the loads fly;
//   - gated launches with any other scale: update_tma_kernel for steady steps of
//     large tensors (one CTA per SM staging tiles of every stream through shared
//     memory with 1-D TMA bulk copies and mbarriers, several stages in flight,
//     bounded waits; further below), persistent 512-thread update_vec_kernel CTAs
//     otherwise: few CTAs, each taking the FP64 decision once;
//   - views not co-aligned to 16 bytes: update_scalar_kernel.
// The per-segment update (one multiplier per segment) runs update_seg_grid_kernel on
// the full grid with multipliers from the host; decided on the device, it runs
// update_tma_kernel<SEG> for steady steps of large buckets and the persistent
// update_segscaled_kernel otherwise.
// Elements before the first 16-byte boundary and after the last full vector or
// tile go through the same arithmetic one at a time.  A gated launch takes the
// skip / clip decision itself, from the 12-byte statistics report (or one report
// per segment) that the merge before it wrote, and is launched as that merge's
// programmatic dependent.
#include <atomic>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

// Tuning knobs (compile-time): vectors per thread per iteration, threads per
// CTA of the full-grid and of the persistent (gated) vector launches, and an L2
// 256-byte prefetch hint on the vector loads.
#ifndef FA_UPDATE_UNROLL
#define FA_UPDATE_UNROLL 2
#endif
#ifndef FA_UPDATE_THREADS
#define FA_UPDATE_THREADS 64
#endif
#ifndef FA_UPDATE_GATED_THREADS
#define FA_UPDATE_GATED_THREADS 512
#endif
#ifndef FA_UPDATE_L2_PREFETCH
#define FA_UPDATE_L2_PREFETCH 0
#endif
// Stores: 0 = evict-first (st.global.cs), 1 = default write-back policy.
#ifndef FA_UPDATE_ST_WB
#define FA_UPDATE_ST_WB 0
#endif
// 1 = large tensors stage tiles through shared memory with 1-D TMA bulk copies
// (see below); 0 = every size uses the register-staged vector kernel.
#ifndef FA_UPDATE_TMA
#define FA_UPDATE_TMA 1
#endif

namespace fa {
namespace {

constexpr int kVec = 8;  // elements per vector
constexpr int kUThreads = FA_UPDATE_THREADS;
constexpr int kUThreadsGated = FA_UPDATE_GATED_THREADS;
constexpr int kUnroll = FA_UPDATE_UNROLL;

// CTAs of a full grid over nvec vectors: one per kUThreads * kUnroll vectors, and one
// for a launch of scalar head and tail elements only (nvec == 0 < n).
inline int64_t full_grid_ctas(int64_t nvec, int64_t n) {
    const int64_t per_cta = static_cast<int64_t>(kUThreads) * kUnroll;
    const int64_t need = (nvec + per_cta - 1) / per_cta;
    return need == 0 && n > 0 ? 1 : need;
}

FA_BOUNDS_COUNTER(g_update_oob)

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

// x / a.gate_scale.  For a power-of-two scale it is the multiplication by the exact
// inverse, which gives the same bits; GB300's FP64 divisions are slow enough that two
// of them per CTA of a full grid cost 5 % of a steady step (4.16 against 3.95 ms at
// 1.07e9 parameters).
__device__ __forceinline__ double gate_unscale(const UpdateArgs &a, double x) {
    return a.gate_inv_scale != 0.0 ? x * a.gate_inv_scale : x / a.gate_scale;
}

// The gradient multiplier of a report without non-finite values: the host's clip
// decision with the same FP64 operations in the same order (norm = sqrt(sum) /
// scale; coef = max_norm / norm above max_norm; sign * coef / scale), so it is
// bit-identical to the host-decided multiplier.
__device__ __forceinline__ float decided_multiplier(const UpdateArgs &a, const fa_stats &r) {
    const double sum = record_sum_sq(r);
    const double norm = gate_unscale(a, sqrt(sum));
    double coef = 1.0;
    if (a.gate_max_norm > 0 && norm > a.gate_max_norm) coef = a.gate_max_norm / norm;
    return static_cast<float>(gate_unscale(a, a.gate_sign * coef));
}

// The host's skip / clip decision, taken on the device from the same report:
// false = skip the update.
__device__ __forceinline__ bool gate_decision(const UpdateArgs &a, float *gmul) {
    const fa_stats r = *a.gate;
    if (r.nonfinite > 0) return false;
    *gmul = decided_multiplier(a, r);
    return true;
}

__device__ __forceinline__ void load8f(const float *base, int64_t i, float (&x)[kVec]) {
    const float4 *q = reinterpret_cast<const float4 *>(base + i);
    float4 a = ld16(q);
    float4 b = ld16(q + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void st16(float4 *q, float4 v) {
#if FA_UPDATE_ST_WB
    *q = v;
#else
    __stcs(q, v);
#endif
}

__device__ __forceinline__ void store8f(float *base, int64_t i, const float (&x)[kVec]) {
    float4 *q = reinterpret_cast<float4 *>(base + i);
    st16(q, make_float4(x[0], x[1], x[2], x[3]));
    st16(q + 1, make_float4(x[4], x[5], x[6], x[7]));
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
    if (!fa_in_bounds(i, 1, a.n)) return;
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
// grid-stride iteration, spaced THREADS vectors apart so that a warp's
// accesses to each stream are contiguous.
template <int GT, bool AMS, bool FIRST, int UNROLL, int MD, int THREADS>
__global__ void __launch_bounds__(THREADS)
update_vec_kernel(const UpdateArgs a, const Coef c0) {
    fa_grid_dependency_wait();  // (a gated launch may start before the merge ends)
    Coef c = c0;
    if (a.gate && !gate_decision(a, &c.gmul)) return;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * THREADS * UNROLL;

    for (int64_t base = static_cast<int64_t>(blockIdx.x) * THREADS * UNROLL + threadIdx.x;
         base < a.nvec; base += stride) {
        float x[UNROLL][kVec], p[UNROLL][kVec], m[UNROLL][kVec], v[UNROLL][kVec],
            vm[UNROLL][kVec];
        bool ok[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t vi = base + static_cast<int64_t>(u) * THREADS;
            ok[u] = vi < a.nvec && fa_in_bounds(a.head + vi * kVec, kVec, a.n);
            if (ok[u]) {
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
            const int64_t vi = base + static_cast<int64_t>(u) * THREADS;
            if (ok[u]) {
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

// The full-grid form of a gated launch: update_vec_kernel's body for one stretch
// of THREADS * UNROLL vectors per CTA, with the decision taken once per CTA.  Every
// thread first issues its loads; thread 0 then takes the decision and shares it
// through shared memory, so that its latency hides behind the loads in flight.  The
// barrier is reached by every thread of the CTA exactly once, before any exit.
template <int GT, bool AMS, bool FIRST, int UNROLL, int MD, int THREADS>
__global__ void __launch_bounds__(THREADS)
update_vec_cta_gate_kernel(const UpdateArgs a, const Coef c0) {
    fa_grid_dependency_wait();  // (launched while the merge before it may still run)
    __shared__ float s_gmul;
    __shared__ int s_go;
    Coef c = c0;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * THREADS * UNROLL;
    int64_t base = static_cast<int64_t>(blockIdx.x) * THREADS * UNROLL + threadIdx.x;

    float x[UNROLL][kVec], p[UNROLL][kVec], m[UNROLL][kVec], v[UNROLL][kVec], vm[UNROLL][kVec];
    bool ok[UNROLL];
    auto load_group = [&]() {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t vi = base + static_cast<int64_t>(u) * THREADS;
            ok[u] = vi < a.nvec && fa_in_bounds(a.head + vi * kVec, kVec, a.n);
            if (ok[u]) {
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
    };
    load_group();
    if (threadIdx.x == 0) {
        float gm = 0.f;
        s_go = gate_decision(a, &gm) ? 1 : 0;
        s_gmul = gm;
    }
    __syncthreads();
    if (!s_go) return;  // the whole CTA: nothing is stored
    c.gmul = s_gmul;
    // One stretch per CTA unless the grid was capped at the launch limit.
    for (;;) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t vi = base + static_cast<int64_t>(u) * THREADS;
            if (ok[u]) {
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
        base += stride;
        if (base >= a.nvec) break;
        load_group();
    }

    // Scalar head [0, head) and tail [head + 8*nvec, n).
    if (tid < a.head) scalar_element<GT, AMS, FIRST, MD>(a, c, tid);
    const int64_t tail0 = a.head + a.nvec * kVec;
    if (tid < a.n - tail0) scalar_element<GT, AMS, FIRST, MD>(a, c, tail0 + tid);
}

// Every element one at a time (pointers not co-aligned to 16 bytes).
template <int GT, bool AMS, bool FIRST, int MD>
__global__ void __launch_bounds__(kThreads)
update_scalar_kernel(const UpdateArgs a, const Coef c0) {
    fa_grid_dependency_wait();
    Coef c = c0;
    if (a.gate && !gate_decision(a, &c.gmul)) return;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < a.n;
         i += stride)
        scalar_element<GT, AMS, FIRST, MD>(a, c, i);
}

// ---- one gradient multiplier per segment -----------------------------------------
//
// Per-parameter clipping ("训练与状态保存", section "FP32 主参数与混合参数存储": clipping
// follows a per-parameter rule, not a whole-model norm): the bucket update with
// the gradient multiplier of the segment each element belongs to, from a
// segment table in kernel parameters.  Register-staged 8-element vectors; a
// thread's vectors only move forward, so its segment index follows by a forward
// scan; a vector that straddles a boundary looks up each element.
__device__ __forceinline__ int find_seg_in(const SegScaleArgs &s, int64_t e, int lo, int hi) {
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.seg_start[mid] <= e) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The same search over a copy of the segment starts in shared memory.
__device__ __forceinline__ int find_seg_smem(const int64_t *seg_start, int64_t e, int lo, int hi) {
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_start[mid] <= e) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int find_seg(const SegScaleArgs &s, int64_t e) {
    int lo = 0, hi = s.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.seg_start[mid] <= e) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int GT, bool AMS, bool FIRST>
__device__ __forceinline__ void scalar_element_seg(const SegScaleArgs &s, const float *gm,
                                                   const Coef &c, int64_t i) {
    Coef cc = c;
    cc.gmul = gm[find_seg(s, i)];
    scalar_element<GT, AMS, FIRST, kNoModel>(s.a, cc, i);
}

// This launch's per-segment multipliers into gm[0, s.nseg), from the kernel
// parameters or, with s.reports, decided on the device: false (skip the launch) when
// any segment of the bucket counts a non-finite value, else each segment's clip
// multiplier with the host's FP64 operations in the host's order (norm =
// sqrt(sum) / scale; coef = max_norm / norm above max_norm; sign * coef / scale), so
// every multiplier is bit-identical to the host-decided step's.  Every thread of the
// CTA calls it (the skip is a CTA-wide vote); gm is read after the next barrier.
__device__ __forceinline__ bool segment_multipliers(const SegScaleArgs &s, float *gm) {
    if (!s.reports) {
        for (int j = threadIdx.x; j < s.nseg; j += blockDim.x) gm[j] = s.gmul[j];
        return true;
    }
    bool bad = false;
    for (int64_t j = threadIdx.x; j < s.nreports; j += blockDim.x)
        bad |= s.reports[j].nonfinite != 0;
    if (__syncthreads_or(bad)) return false;
    for (int j = threadIdx.x; j < s.nseg; j += blockDim.x)
        gm[j] = decided_multiplier(s.a, s.reports[s.k0 + j]);
    return true;
}

// Every segment's decision, once for the whole bucket (see launch_segment_decide).
// The bucket's record from the FP64 total of its segments' sums of squares and their
// non-finite count (saturating): a (hi, lo) pair of floats, scaled by 2^-192 and
// negated once the total leaves the range where FP32 holds it safely, the two forms
// that record_sum_sq decodes.
__device__ __forceinline__ fa_stats bucket_record(double sum, unsigned long long count) {
    fa_stats r;
    r.nonfinite = count > 0xffffffffull ? 0xffffffffu : static_cast<uint32_t>(count);
    const bool scaled = !(sum < 0x1p126);
    const double s = scaled ? sum * 0x1p-192 : sum;
    const float hi = static_cast<float>(s);
    const float lo = static_cast<float>(s - static_cast<double>(hi));
    r.sum_sq = scaled ? -hi : hi;
    r.sum_sq_lo = scaled ? -lo : lo;
    return r;
}

constexpr int kDecideThreads = 256;
__global__ void __launch_bounds__(kDecideThreads)
segment_decide_kernel(const UpdateArgs a, const fa_stats *reports, int32_t nseg,
                      float *decided, fa_report_mailbox *post, uint32_t seq) {
    fa_grid_dependency_wait();  // the merge that writes the records may still run
    bool bad = false;
    double sum = 0.0;
    unsigned long long count = 0;
    for (int j = threadIdx.x; j < nseg; j += kDecideThreads) {
        const fa_stats r = reports[j];
        bad |= r.nonfinite != 0;
        count += r.nonfinite;
        sum += record_sum_sq(r);
        if (decided) decided[1 + j] = decided_multiplier(a, r);
    }
    const int skip = __syncthreads_or(bad);
    if (decided && threadIdx.x == 0) decided[0] = skip ? 1.0f : 0.0f;
    if (!post) return;
    // the bucket's totals, in a fixed order: each warp by a shuffle tree, then the
    // warps in turn
    __shared__ double s_sum[kDecideThreads / 32];
    __shared__ unsigned long long s_count[kDecideThreads / 32];
    for (int d = 16; d > 0; d >>= 1) {
        sum += __shfl_down_sync(0xffffffffu, sum, d);
        count += __shfl_down_sync(0xffffffffu, count, d);
    }
    if ((threadIdx.x & 31) == 0) {
        s_sum[threadIdx.x >> 5] = sum;
        s_count[threadIdx.x >> 5] = count;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    double total = 0.0;
    unsigned long long total_count = 0;
    for (int w = 0; w < kDecideThreads / 32; ++w) {
        total += s_sum[w];
        total_count += s_count[w];
    }
    const fa_stats rec = bucket_record(total, total_count);
    volatile uint32_t *out = reinterpret_cast<volatile uint32_t *>(&post->report);
    out[0] = __float_as_uint(rec.sum_sq);
    out[1] = rec.nonfinite;
    out[2] = __float_as_uint(rec.sum_sq_lo);
    __threadfence_system();  // a host that sees seq reads the whole record
    *reinterpret_cast<volatile uint32_t *>(&post->seq) = seq;
}

// The per-segment update on the full grid, with multipliers from the host or
// decided once for the bucket on the device (s.decided): one stretch of THREADS *
// UNROLL vectors per CTA (the launcher guarantees that the grid covers every
// stretch), the body of update_vec_kernel.  A CTA copies the multipliers of only the
// segments its elements fall in, [k_lo, k_hi] (usually one), from the kernel
// parameters or the decided table into shared memory; a decided skip ends every
// CTA before it stores anything.  CTA 0 also takes the scalar head and the last CTA
// the scalar tail, so their ranges include those elements.  A vector finds its
// segment by a forward scan from k_lo; one that straddles a boundary looks up each
// element.  (Deciding in every CTA from the reports measured slower than the
// pipeline: 6.35-6.63 against 6.11 ms for the 1.2e9-parameter, 199-segment FP16
// AMSGrad bucket.)
template <int GT, bool AMS, bool FIRST, int UNROLL, int THREADS>
__global__ void __launch_bounds__(THREADS)
update_seg_grid_kernel(const __grid_constant__ SegScaleArgs s, const Coef c) {
    __shared__ float gm[kMaxSegPerLaunch];
    fa_grid_dependency_wait();
    const UpdateArgs &a = s.a;
    const int64_t vb = static_cast<int64_t>(blockIdx.x) * THREADS * UNROLL;
    float x[UNROLL][kVec], p[UNROLL][kVec], m[UNROLL][kVec], v[UNROLL][kVec], vm[UNROLL][kVec];
    bool ok[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t vi = vb + threadIdx.x + static_cast<int64_t>(u) * THREADS;
        ok[u] = vi < a.nvec && fa_in_bounds(a.head + vi * kVec, kVec, a.n);
        if (ok[u]) {
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

    // elements [e_lo, e_hi) of this CTA, and their segments [k_lo, k_hi]
    const int64_t body_end = a.head + a.nvec * kVec;
    const int64_t e_lo = blockIdx.x == 0 ? 0 : a.head + vb * kVec;
    int64_t e_hi = a.head + (vb + static_cast<int64_t>(THREADS) * UNROLL) * kVec;
    if (e_hi > body_end) e_hi = body_end;
    if (blockIdx.x == gridDim.x - 1) e_hi = a.n;
    const int k_lo = find_seg(s, e_lo);
    const int k_hi = e_hi > e_lo ? find_seg(s, e_hi - 1) : k_lo;
    __shared__ int s_skip;
    const float *decided = s.decided;
    for (int k = k_lo + threadIdx.x; k <= k_hi; k += THREADS)
        gm[k] = decided ? decided[1 + s.k0 + k] : s.gmul[k];
    if (threadIdx.x == 0) s_skip = decided != nullptr && decided[0] != 0.0f;
    __syncthreads();
    if (s_skip) return;  // the whole CTA: nothing is stored

    int k = k_lo;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        if (!ok[u]) continue;
        const int64_t e = a.head + (vb + threadIdx.x + static_cast<int64_t>(u) * THREADS) * kVec;
        while (k < k_hi && s.seg_start[k + 1] <= e) ++k;
        Coef cc = c;
        if (e + kVec <= s.seg_start[k + 1]) {
            cc.gmul = gm[k];
#pragma unroll
            for (int q = 0; q < kVec; ++q)
                adamw_element<AMS, FIRST>(cc, x[u][q], p[u][q], m[u][q], v[u][q], vm[u][q]);
        } else {
#pragma unroll
            for (int q = 0; q < kVec; ++q) {
                cc.gmul = gm[find_seg_in(s, e + q, k, k_hi)];
                adamw_element<AMS, FIRST>(cc, x[u][q], p[u][q], m[u][q], v[u][q], vm[u][q]);
            }
        }
        store8f(a.p_out, e, p[u]);
        store8f(a.m_out, e, m[u]);
        store8f(a.v_out, e, v[u]);
        if (AMS) store8f(a.vmax_out, e, vm[u]);
    }
    if (blockIdx.x == 0 && threadIdx.x < a.head)
        scalar_element_seg<GT, AMS, FIRST>(s, gm, c, threadIdx.x);
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x < a.n - body_end)
        scalar_element_seg<GT, AMS, FIRST>(s, gm, c, body_end + threadIdx.x);
}

#if FA_UPDATE_TMA
// ---- shared-memory staging with 1-D TMA bulk copies ---------------------------
//
// One CTA per SM.  Tiles of TmaLayout::kTile elements move between HBM and shared
// memory as one cp.async.bulk per stream (p, g, m, v[, vmax] in; p, m,
// v[, vmax][, model copy] out), completion tracked by one mbarrier per
// stage.  S stages are in flight; thread 0 issues all copies.  Each thread
// updates two 4-element chunks of a tile in shared memory (chunks strided by
// 4*kTmaThreads so that a warp's 16-byte accesses are contiguous).  Waits are
// bounded: a wait that gives up sets g_update_tma_error, drains this CTA's
// own copies (bounded again) and returns.
#ifndef FA_TMA_THREADS
#define FA_TMA_THREADS 256
#endif
constexpr int kTmaThreads = FA_TMA_THREADS;
constexpr int kTmaSmemBudget = 226 * 1024;  // dynamic shared memory per CTA
constexpr int kSmemPerCtaMax = 227 * 1024;  // the architectural limit, tables included
// The per-segment table staged in shared memory: starts and multipliers.
constexpr int kSegTableBytes = (kMaxSegPerLaunch + 1) * 8 + kMaxSegPerLaunch * 4;
constexpr uint32_t kTmaSpinLimit = 1u << 20;   // tries per wait (x kTmaSuspendNs: ~1 s)
constexpr uint32_t kTmaSuspendNs = 1000;

__device__ int g_update_tma_error;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    // each try suspends at most kTmaSuspendNs before reporting "not yet"
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
                 " selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(kTmaSuspendNs) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(smem_addr(src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Per-instantiation tile size and stage count, by bytes per element (all
// streams in and out).  Measured on GB300 (1.07e9 elements; tile x stages):
//   14 B (BF16/FP16 AdamW)           3072 x 4   6.89 TB/s
//   16 B (FP32 AdamW; BF16 + copy)   4096 x 3   6.93 / 6.73 TB/s
//   18-22 B (AMSGrad, copies)        3072 x 3   6.75-6.87 TB/s
// Two stages, and some power-of-two tile/stage pairs, fell to 3.1-6.4 TB/s.
template <int GT, bool AMS, int MD>
struct TmaLayout {
    static constexpr int kGB = GT == FA_F32 ? 4 : 2;
    static constexpr int kElemBytes = 12 + (AMS ? 4 : 0) + kGB + (MD != kNoModel ? 2 : 0);
    static constexpr int kQuantum = 4 * kTmaThreads;
#ifdef FA_TMA_TILE_OVERRIDE
    static constexpr int kTile = FA_TMA_TILE_OVERRIDE;
#else
    static constexpr int kTile = kElemBytes == 16 ? 4096 : 3072;
#endif
#ifdef FA_TMA_STAGES_OVERRIDE
    static constexpr int kWantStages = FA_TMA_STAGES_OVERRIDE;
#else
    static constexpr int kWantStages = kElemBytes <= 14 ? 4 : 3;
#endif
    static_assert(kTile % kQuantum == 0, "tile must be a whole number of 4-element chunks");
    static constexpr int kChunks = kTile / kQuantum;  // 4-element chunks per thread
    static constexpr int kP = 0;
    static constexpr int kM = kTile * 4;
    static constexpr int kV = kTile * 8;
    static constexpr int kVM = kTile * 12;
    static constexpr int kG = kTile * (AMS ? 16 : 12);
    static constexpr int kModel = kG + kTile * kGB;
    static constexpr int kStage = kModel + (MD != kNoModel ? kTile * 2 : 0);
    static constexpr int kStagesRaw = (kTmaSmemBudget - 64) / kStage;
    static constexpr int kStages = kWantStages <= kStagesRaw ? kWantStages : kStagesRaw;
    static constexpr int kSmem = kStages * kStage + kStages * 8;
    static_assert(kStages >= 2, "at least two stages");
};

// Dynamic shared memory of one launch: the stages, their barriers and, with SEG,
// the segment table (read at every segment crossing: in shared memory it costs a
// few tens of cycles, where an indexed kernel-parameter read that misses the
// constant cache stalled the tile loop for hundreds).
template <int GT, bool AMS, int MD, bool SEG>
constexpr int tma_smem_bytes() {
    return TmaLayout<GT, AMS, MD>::kSmem + (SEG ? kSegTableBytes : 0);
}

// SEG: one gradient multiplier per segment from s's table (MD must be kNoModel);
// otherwise s.nseg is 0 and c.gmul applies to every element.
template <int GT, bool AMS, bool FIRST, int MD, bool SEG>
__global__ void __launch_bounds__(kTmaThreads, 1)
update_tma_kernel(const __grid_constant__ SegScaleArgs sa, const Coef c0, int64_t ntiles) {
    const UpdateArgs &a = sa.a;
    Coef c = c0;
    fa_grid_dependency_wait();  // (a gated launch may start before the merge ends)
    // a skipped step returns before any copy is issued (every thread decides alike)
    if (a.gate && !gate_decision(a, &c.gmul)) return;
    using L = TmaLayout<GT, AMS, MD>;
    constexpr int S = L::kStages;
    constexpr uint32_t kLoadBytes =
        L::kTile * (4 + L::kGB + (FIRST ? 0 : (AMS ? 12 : 8)));
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * L::kStage);
    int64_t *s_seg = reinterpret_cast<int64_t *>(smem + S * L::kStage + S * 8);  // SEG only
    float *s_gmul = reinterpret_cast<float *>(s_seg + kMaxSegPerLaunch + 1);
    const int tid = threadIdx.x;

    // thread 0's view of each stage: loads issued and consumed
    uint32_t issued[S], consumed[S];
#pragma unroll
    for (int s = 0; s < S; ++s) issued[s] = consumed[s] = 0;

    auto issue_loads = [&](int s, int64_t tile) {
        unsigned char *b = smem + s * L::kStage;
        const int64_t e = a.head + tile * L::kTile;
        // (a tile out of range is skipped; its wait then runs out and the
        // pipeline's error flag is raised as well)
        if (!fa_in_bounds(e, L::kTile, a.n)) return;
        mbar_expect_tx(&bars[s], kLoadBytes + a.extra_tx);
        bulk_load(b + L::kP, a.p_in + e, L::kTile * 4, &bars[s]);
        bulk_load(b + L::kG, static_cast<const char *>(a.g) + e * L::kGB, L::kTile * L::kGB,
                  &bars[s]);
        if (!FIRST) {
            bulk_load(b + L::kM, a.m_in + e, L::kTile * 4, &bars[s]);
            bulk_load(b + L::kV, a.v_in + e, L::kTile * 4, &bars[s]);
            if (AMS) bulk_load(b + L::kVM, a.vmax_in + e, L::kTile * 4, &bars[s]);
        }
        ++issued[s];
    };

    if (SEG) {
        // a launch skipped by the device-side decision returns before any copy
        if (!segment_multipliers(sa, s_gmul)) return;
        for (int j = tid; j <= sa.nseg; j += kTmaThreads) s_seg[j] = sa.seg_start[j];
    }
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bars[s]);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t tile = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (tile < ntiles) issue_loads(s, tile);
        }
    }

    bool failed = false;
    int64_t k = 0;
    // segment of the current tile's first element: a CTA's tiles only move forward,
    // so the index advances by a scan whose total length over the launch is at most
    // the number of segments; the next segment's start and the current multiplier
    // stay in registers, so a tile inside one segment reads no table entry
    int k_lo = 0;
    int64_t next_start = INT64_MAX;
    float seg_gmul = 0.f;
    if (SEG) {
        if (sa.nseg > 1) next_start = sa.seg_start[1];
        seg_gmul = s_gmul[0];
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
        const int s = static_cast<int>(k % S);
        const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
        // segments of this tile's first and last element (warp-uniform scans), found
        // before the wait so that they cost nothing between the tile's arrival and
        // the refill that follows its update
        int k_hi = 0;
        if (SEG) {
            const int64_t t0 = a.head + tile * L::kTile;
            if (t0 >= next_start) {
                do {
                    ++k_lo;
                    next_start = k_lo + 1 < sa.nseg ? s_seg[k_lo + 1] : INT64_MAX;
                } while (t0 >= next_start);
                seg_gmul = s_gmul[k_lo];
            }
            k_hi = k_lo;
            if (t0 + L::kTile > next_start) {  // the tile reaches into later segments
                k_hi = k_lo + 1;
                while (k_hi + 1 < sa.nseg && s_seg[k_hi + 1] < t0 + L::kTile) ++k_hi;
            }
        }
        uint32_t it = 0;
        while (!mbar_try_wait(&bars[s], parity)) {
            if (++it == kTmaSpinLimit) { failed = true; break; }
        }
        if (__syncthreads_or(failed)) { failed = true; break; }
        if (tid == 0) consumed[s] = issued[s];

        unsigned char *b = smem + s * L::kStage;
        Coef ct = c;
        if (SEG) ct.gmul = seg_gmul;
        // One 4-element chunk per call; PER_ELEM looks up each element's segment (a tile
        // that straddles a boundary).  The branch between the two forms is taken once
        // per tile, so a tile inside one segment runs the same straight-line code over
        // all its chunks as the kernel without a segment table (a branch per chunk cost
        // the per-segment update 1 % of its time).
        auto chunk = [&](int h, auto per_elem) {
            const int j = h * 4 * kTmaThreads + 4 * tid;  // first element of this chunk
            float x[4], p[4], m[4], v[4], vm[4];
            if (GT == FA_F32) {
                const float4 t4 = *reinterpret_cast<const float4 *>(b + L::kG + 4 * j);
                x[0] = t4.x; x[1] = t4.y; x[2] = t4.z; x[3] = t4.w;
            } else {
                const uint2 r = *reinterpret_cast<const uint2 *>(b + L::kG + 2 * j);
                if (GT == FA_BF16) {
                    x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xffff0000u);
                    x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xffff0000u);
                } else {
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
                    x[0] = f0.x; x[1] = f0.y; x[2] = f1.x; x[3] = f1.y;
                }
            }
            float4 *pp = reinterpret_cast<float4 *>(b + L::kP + 4 * j);
            float4 *mp = reinterpret_cast<float4 *>(b + L::kM + 4 * j);
            float4 *vp = reinterpret_cast<float4 *>(b + L::kV + 4 * j);
            float4 *vmp = reinterpret_cast<float4 *>(b + L::kVM + 4 * j);
            const float4 p4 = *pp;
            p[0] = p4.x; p[1] = p4.y; p[2] = p4.z; p[3] = p4.w;
            if (!FIRST) {
                const float4 m4 = *mp, v4 = *vp;
                m[0] = m4.x; m[1] = m4.y; m[2] = m4.z; m[3] = m4.w;
                v[0] = v4.x; v[1] = v4.y; v[2] = v4.z; v[3] = v4.w;
                if (AMS) {
                    const float4 w4 = *vmp;
                    vm[0] = w4.x; vm[1] = w4.y; vm[2] = w4.z; vm[3] = w4.w;
                }
            }
            if constexpr (decltype(per_elem)::value) {
                const int64_t e = a.head + tile * L::kTile + j;
                Coef cc = ct;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    cc.gmul = s_gmul[find_seg_smem(s_seg, e + q, k_lo, k_hi)];
                    adamw_element<AMS, FIRST>(cc, x[q], p[q], m[q], v[q], vm[q]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    adamw_element<AMS, FIRST>(ct, x[q], p[q], m[q], v[q], vm[q]);
            }
            *pp = make_float4(p[0], p[1], p[2], p[3]);
            *mp = make_float4(m[0], m[1], m[2], m[3]);
            *vp = make_float4(v[0], v[1], v[2], v[3]);
            if (AMS) *vmp = make_float4(vm[0], vm[1], vm[2], vm[3]);
            if (MD != kNoModel) {
                uint2 w;
                w.x = pack2<MD>(p[0], p[1]);
                w.y = pack2<MD>(p[2], p[3]);
                *reinterpret_cast<uint2 *>(b + L::kModel + 2 * j) = w;
            }
        };
        if (!SEG || k_lo == k_hi) {
#pragma unroll
            for (int h = 0; h < L::kChunks; ++h) chunk(h, std::false_type{});
        } else {
#pragma unroll 1
            for (int h = 0; h < L::kChunks; ++h) chunk(h, std::true_type{});
        }
        fence_async_shared();
        __syncthreads();
        if (tid == 0) {
            const int64_t e = a.head + tile * L::kTile;
            if (fa_in_bounds(e, L::kTile, a.n)) {
                bulk_store(a.p_out + e, b + L::kP, L::kTile * 4);
                bulk_store(a.m_out + e, b + L::kM, L::kTile * 4);
                bulk_store(a.v_out + e, b + L::kV, L::kTile * 4);
                if (AMS) bulk_store(a.vmax_out + e, b + L::kVM, L::kTile * 4);
                if (MD != kNoModel)
                    bulk_store(static_cast<uint16_t *>(a.p_model) + e, b + L::kModel,
                               L::kTile * 2);
            }
            bulk_commit();
            // refill the stage used one iteration ago: its stores had a whole
            // iteration to finish reading shared memory
            if (k >= 1) {
                const int sp = static_cast<int>((k - 1) % S);
                const int64_t next = tile + static_cast<int64_t>(S - 1) * gridDim.x;
                if (next < ntiles) {
                    bulk_wait_read1();
                    issue_loads(sp, next);
                }
            }
        }
    }

    if (tid == 0) {
        if (failed) {
            atomicExch(&g_update_tma_error, 1);
            // drain this CTA's own loads still in flight, bounded again
#pragma unroll
            for (int s = 0; s < S; ++s) {
                if (issued[s] > consumed[s]) {
                    const uint32_t par = (issued[s] - 1) & 1;
                    for (uint32_t it = 0; it < kTmaSpinLimit && !mbar_try_wait(&bars[s], par); ++it) {
                    }
                }
            }
        }
        bulk_wait_all();
    }
    __syncthreads();
    if (failed) return;

    // scalar head [0, head) and tail after the last full tile
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kTmaThreads + tid;
    const int64_t gsz = static_cast<int64_t>(gridDim.x) * kTmaThreads;
    const int64_t tail0 = a.head + ntiles * L::kTile;
    if (SEG) {
        for (int64_t i = gtid; i < a.head; i += gsz)
            scalar_element_seg<GT, AMS, FIRST>(sa, s_gmul, c, i);
        for (int64_t i = tail0 + gtid; i < a.n; i += gsz)
            scalar_element_seg<GT, AMS, FIRST>(sa, s_gmul, c, i);
    } else {
        for (int64_t i = gtid; i < a.head; i += gsz) scalar_element<GT, AMS, FIRST, MD>(a, c, i);
        for (int64_t i = tail0 + gtid; i < a.n; i += gsz) scalar_element<GT, AMS, FIRST, MD>(a, c, i);
    }
}
#endif  // FA_UPDATE_TMA

#if FA_UPDATE_TMA
// Steady steps of at least two tiles per SM that are gated with a scale that is not a
// power of two, or decided per segment on the device, take the TMA pipeline, whose
// 152 CTAs take the decisions once each; the
// first step (moments only written: 6 B in, 12 B out) measured faster through
// the register kernel (3.0 vs 3.7 ms at 1.07e9), and so did small tensors.
template <int GT, bool AMS, bool FIRST, int MD, bool SEG>
cudaError_t launch_tma_if_large(const SegScaleArgs &s, const Coef &c, bool vector_ok, int dev,
                                cudaStream_t stream, bool *launched) {
    using L = TmaLayout<GT, AMS, MD>;
    constexpr int kSmem = tma_smem_bytes<GT, AMS, MD, SEG>();
    static_assert(kSmem <= kSmemPerCtaMax, "shared memory per CTA");
    *launched = false;
    const int64_t ntiles = (s.a.n - s.a.head) / L::kTile;
    const int64_t sms = sm_count(dev);
    if (FIRST || !vector_ok || ntiles < 2 * sms) return cudaSuccess;
    auto kern = update_tma_kernel<GT, AMS, FIRST, MD, SEG>;
    // the attribute is per device; setting it twice from racing threads is harmless
    static std::atomic<bool> configured[64] = {};
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        const cudaError_t err =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(true, std::memory_order_release);
    }
    const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
    *launched = true;
    // gated (one report, or one per segment): scheduled while the merge before it
    // runs; the kernel waits for it
    if (s.a.gate || s.reports)
        return launch_dependent(kern, dim3(grid), dim3(kTmaThreads), kSmem, stream, s, c,
                                ntiles);
    kern<<<grid, kTmaThreads, kSmem, stream>>>(s, c, ntiles);
    return cudaGetLastError();
}
#endif

template <int GT, bool AMS, bool FIRST>
__global__ void __launch_bounds__(kThreads)
update_segscaled_kernel(const __grid_constant__ SegScaleArgs s, const Coef c) {
    __shared__ float gm[kMaxSegPerLaunch];
    fa_grid_dependency_wait();
    if (!segment_multipliers(s, gm)) return;
    __syncthreads();
    const UpdateArgs &a = s.a;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int k = 0;  // segment of e; e only grows, so a forward scan finds it
    for (int64_t vi = tid; vi < a.nvec; vi += stride) {
        const int64_t e = a.head + vi * kVec;
        if (!fa_in_bounds(e, kVec, a.n)) continue;
        float x[kVec], p[kVec], m[kVec], v[kVec], vm[kVec];
        GradIO<GT>::load8(a.g, e, x);
        load8f(a.p_in, e, p);
        if (!FIRST) {
            load8f(a.m_in, e, m);
            load8f(a.v_in, e, v);
            if (AMS) load8f(a.vmax_in, e, vm);
        }
        while (k + 1 < s.nseg && s.seg_start[k + 1] <= e) ++k;
        Coef cc = c;
        if (e + kVec <= s.seg_start[k + 1]) {
            cc.gmul = gm[k];
#pragma unroll
            for (int q = 0; q < kVec; ++q) adamw_element<AMS, FIRST>(cc, x[q], p[q], m[q], v[q], vm[q]);
        } else {
#pragma unroll
            for (int q = 0; q < kVec; ++q) {
                cc.gmul = gm[find_seg_in(s, e + q, k, s.nseg - 1)];
                adamw_element<AMS, FIRST>(cc, x[q], p[q], m[q], v[q], vm[q]);
            }
        }
        store8f(a.p_out, e, p);
        store8f(a.m_out, e, m);
        store8f(a.v_out, e, v);
        if (AMS) store8f(a.vmax_out, e, vm);
    }
    if (tid < a.head) scalar_element_seg<GT, AMS, FIRST>(s, gm, c, tid);
    const int64_t tail0 = a.head + a.nvec * kVec;
    if (tid < a.n - tail0) scalar_element_seg<GT, AMS, FIRST>(s, gm, c, tail0 + tid);
}

template <int GT, bool AMS, bool FIRST>
__global__ void __launch_bounds__(kThreads)
update_segscaled_scalar_kernel(const __grid_constant__ SegScaleArgs s, const Coef c) {
    __shared__ float gm[kMaxSegPerLaunch];
    fa_grid_dependency_wait();
    if (!segment_multipliers(s, gm)) return;
    __syncthreads();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < s.a.n;
         i += stride)
        scalar_element_seg<GT, AMS, FIRST>(s, gm, c, i);
}

template <int GT, bool AMS, bool FIRST>
cudaError_t launch_seg_typed(const SegScaleArgs &s, const Coef &c, bool vec, cudaStream_t st) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // Multipliers from the host, or decided once for the bucket: the full grid.
    // Decided by each launch from the reports: few CTAs (the pipeline, or persistent
    // CTAs), each taking every segment's decision once.
    if (vec && (!s.reports || s.decided)) {
        auto kern = update_seg_grid_kernel<GT, AMS, FIRST, kUnroll, kUThreads>;
        const int64_t need = full_grid_ctas(s.a.nvec, s.a.n);
        if (need <= kMaxGridX) {  // the kernel has no loop: every stretch its own CTA
            const int grid = static_cast<int>(need);
            if (grid == 0) return cudaSuccess;
            if (s.decided)  // scheduled while the decision kernel before it runs
                return launch_dependent(kern, dim3(grid), dim3(kUThreads), 0, st, s, c);
            kern<<<grid, kUThreads, 0, st>>>(s, c);
            return cudaGetLastError();
        }
    }
    // decided on the device: scheduled while the merge before it runs
    const bool dependent = s.reports != nullptr;
#if FA_UPDATE_TMA
    bool launched = false;
    err = launch_tma_if_large<GT, AMS, FIRST, kNoModel, true>(s, c, vec, dev, st, &launched);
    if (err != cudaSuccess || launched) return err;
#endif
    if (vec) {
        auto kern = update_segscaled_kernel<GT, AMS, FIRST>;
        int64_t need = (s.a.nvec + kThreads - 1) / kThreads;
        if (need == 0 && s.a.n > 0) need = 1;
        const int grid = persistent_grid(kern, need, dev);
        if (grid == 0) return cudaSuccess;
        if (dependent) return launch_dependent(kern, dim3(grid), dim3(kThreads), 0, st, s, c);
        kern<<<grid, kThreads, 0, st>>>(s, c);
    } else {
        auto kern = update_segscaled_scalar_kernel<GT, AMS, FIRST>;
        const int grid = persistent_grid(kern, (s.a.n + kThreads - 1) / kThreads, dev);
        if (grid == 0) return cudaSuccess;
        if (dependent) return launch_dependent(kern, dim3(grid), dim3(kThreads), 0, st, s, c);
        kern<<<grid, kThreads, 0, st>>>(s, c);
    }
    return cudaGetLastError();
}

template <int GT>
cudaError_t launch_seg_gt(const SegScaleArgs &s, const Coef &c, bool ams, bool first, bool vec,
                          cudaStream_t st) {
    if (ams)
        return first ? launch_seg_typed<GT, true, true>(s, c, vec, st)
                     : launch_seg_typed<GT, true, false>(s, c, vec, st);
    return first ? launch_seg_typed<GT, false, true>(s, c, vec, st)
                 : launch_seg_typed<GT, false, false>(s, c, vec, st);
}


template <int GT, bool AMS, bool FIRST, int MD>
cudaError_t launch_typed(const UpdateArgs &a, const Coef &c, bool vector_ok,
                         cudaStream_t stream) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (sm_count(dev) <= 0) return cudaErrorInvalidDevice;

    // A gated launch whose scale has an exact inverse: the full grid, deciding once
    // per CTA (with multiplications instead of the FP64 divisions).
    if (vector_ok && a.gate && a.gate_inv_scale != 0.0) {
        auto kern = update_vec_cta_gate_kernel<GT, AMS, FIRST, kUnroll, MD, kUThreads>;
        const int64_t need = full_grid_ctas(a.nvec, a.n);  // beyond the cap: the loop
        const int grid = static_cast<int>(need < kMaxGridX ? need : kMaxGridX);
        if (grid == 0) return cudaSuccess;
        return launch_dependent(kern, dim3(grid), dim3(kUThreads), 0, stream, a, c);
    }
#if FA_UPDATE_TMA
    if (a.gate) {
        SegScaleArgs s;
        s.a = a;
        s.nseg = 0;
        s.reports = nullptr;
        s.nreports = 0;
        s.k0 = 0;
        s.decided = nullptr;
        bool launched = false;
        err = launch_tma_if_large<GT, AMS, FIRST, MD, false>(s, c, vector_ok, dev, stream, &launched);
        if (err != cudaSuccess || launched) return err;
    }
#endif
    if (vector_ok && a.gate) {
        // Other scales: persistent CTAs, each taking the decision (with its FP64
        // divisions) once; GB300's FP64 rate makes those divisions in every small CTA
        // of a full grid cost more than the grid gains (4.16 against 4.07 ms for the
        // TMA pipeline at 1.07e9 parameters).
        auto kern = update_vec_kernel<GT, AMS, FIRST, kUnroll, MD, kUThreadsGated>;
        const int64_t per_cta = static_cast<int64_t>(kUThreadsGated) * kUnroll;
        int64_t need = (a.nvec + per_cta - 1) / per_cta;
        if (need == 0 && a.n > 0) need = 1;  // head/tail elements only
        const int grid = persistent_grid(kern, need, dev, kUThreadsGated);
        if (grid == 0) return cudaSuccess;
        return launch_dependent(kern, dim3(grid), dim3(kUThreadsGated), 0, stream, a, c);
    } else if (vector_ok) {
        // A full grid: one small CTA per kUThreads * kUnroll vectors, each CTA normally
        // one iteration (the loop matters only for a grid capped at the launch limit).
        // Measured on GB300 (1.07e9 parameters, CUDA events) against persistent grids
        // of the same kernel and against the shared-memory (TMA) pipeline, it moves
        // every byte mix fastest.
        auto kern = update_vec_kernel<GT, AMS, FIRST, kUnroll, MD, kUThreads>;
        const int64_t need = full_grid_ctas(a.nvec, a.n);  // beyond the cap: the loop
        const int grid = static_cast<int>(need < kMaxGridX ? need : kMaxGridX);
        if (grid == 0) return cudaSuccess;
        kern<<<grid, kUThreads, 0, stream>>>(a, c);
    } else {
        auto kern = update_scalar_kernel<GT, AMS, FIRST, MD>;
        const int grid = persistent_grid(kern, (a.n + kThreads - 1) / kThreads, dev);
        if (grid == 0) return cudaSuccess;
        if (a.gate) return launch_dependent(kern, dim3(grid), dim3(kThreads), 0, stream, a, c);
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

cudaError_t launch_segment_decide(const UpdateArgs &a, const fa_stats *reports, int32_t nseg,
                                  float *decided, fa_report_mailbox *post, uint32_t seq,
                                  cudaStream_t stream) {
    return launch_dependent(segment_decide_kernel, dim3(1), dim3(kDecideThreads), 0, stream, a,
                            reports, nseg, decided, post, seq);
}

cudaError_t launch_update_segment_scaled(const SegScaleArgs &s, const Coef &c, fa_dtype gdt,
                                         bool amsgrad, bool first, bool vector_ok,
                                         cudaStream_t stream) {
    switch (gdt) {
        case FA_F32: return launch_seg_gt<FA_F32>(s, c, amsgrad, first, vector_ok, stream);
        case FA_F16: return launch_seg_gt<FA_F16>(s, c, amsgrad, first, vector_ok, stream);
        case FA_BF16: return launch_seg_gt<FA_BF16>(s, c, amsgrad, first, vector_ok, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_pipeline_selftest(const UpdateArgs &a, const Coef &c, fa_dtype gdt,
                                     bool *launched, cudaStream_t stream) {
    *launched = false;
#if FA_UPDATE_TMA
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    SegScaleArgs s;
    s.a = a;
    s.nseg = 0;
    s.reports = nullptr;
    s.nreports = 0;
    s.k0 = 0;
    s.decided = nullptr;
    switch (gdt) {
        case FA_F32:
            return launch_tma_if_large<FA_F32, false, false, kNoModel, false>(s, c, true, dev,
                                                                             stream, launched);
        case FA_F16:
            return launch_tma_if_large<FA_F16, false, false, kNoModel, false>(s, c, true, dev,
                                                                             stream, launched);
        case FA_BF16:
            return launch_tma_if_large<FA_BF16, false, false, kNoModel, false>(s, c, true, dev,
                                                                              stream, launched);
    }
    return cudaErrorInvalidValue;
#else
    (void)a; (void)c; (void)gdt; (void)stream;
    return cudaSuccess;
#endif
}

cudaError_t update_bounds_violations(unsigned long long *count, bool clear) {
#if FA_BOUNDS_CHECK
    cudaError_t err = cudaMemcpyFromSymbol(count, g_update_oob, sizeof(*count));
    if (err != cudaSuccess || !clear) return err;
    const unsigned long long zero = 0;
    return cudaMemcpyToSymbol(g_update_oob, &zero, sizeof(zero));
#else
    (void)clear;
    *count = 0;
    return cudaSuccess;
#endif
}

cudaError_t update_pipeline_error(int *flag, bool clear) {
#if FA_UPDATE_TMA
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_update_tma_error, sizeof(int));
    if (err != cudaSuccess || !clear) return err;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_update_tma_error, &zero, sizeof(int));
#else
    (void)clear;
    *flag = 0;
    return cudaSuccess;
#endif
}

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
