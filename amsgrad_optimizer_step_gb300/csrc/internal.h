// Internal interface between the C-ABI host layer (abi.cpp) and the kernels.
#pragma once

#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "fused_adamw.h"

// Bounds-checked build (-DFA_BOUNDS_CHECK=1, a test variant of the library): every
// kernel checks the element range it is about to touch against the length of its
// array; an access outside it is counted in the translation unit's device counter
// and skipped, never performed.  The normal build compiles the checks out.
#ifndef FA_BOUNDS_CHECK
#define FA_BOUNDS_CHECK 0
#endif

#if defined(__CUDACC__)
#if FA_BOUNDS_CHECK
#define FA_BOUNDS_COUNTER(counter)                                                     \
    static __device__ unsigned long long counter;                                     \
    __device__ __forceinline__ bool fa_in_bounds(int64_t first, int64_t count,          \
                                                 int64_t n) {                          \
        if (first >= 0 && count >= 0 && first + count <= n) return true;              \
        atomicAdd(&counter, 1ull);                                                     \
        return false;                                                                  \
    }
#else
#define FA_BOUNDS_COUNTER(counter)                                                     \
    __device__ __forceinline__ constexpr bool fa_in_bounds(int64_t, int64_t, int64_t) { \
        return true;                                                                   \
    }
#endif
#endif

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization allowed (launch_dependent below) may be scheduled while the kernel
// before it in the stream is still running, once every CTA of that kernel has
// called fa_allow_dependents() or exited.  fa_grid_dependency_wait() then blocks
// until the earlier kernel has completed and its writes are visible; in a kernel
// launched the ordinary way it returns at once.  Every kernel launched through
// launch_dependent calls it before its first global-memory access, so starting
// early never reads anything stale: what overlaps is launch latency, CTA
// scheduling and shared-memory setup.
#if defined(__CUDACC__)
__device__ __forceinline__ void fa_grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void fa_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

namespace fa {

#if defined(__CUDACC__)
// Launches ``kernel`` with programmatic stream serialization allowed.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block,
                                    size_t smem, cudaStream_t stream, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

constexpr int kThreads = 256;            // threads per CTA for every kernel here
constexpr int kFanIn = 1024;             // merge fan-in
constexpr int64_t kMaxRows = 4194304;    // largest statistics plan
constexpr int kMaxSegPerLaunch = 240;    // segment table entries carried in kernel parameters

// The sum of squares a statistics record stands for.  A row whose FP32 sum of
// squares overflows while it holds no NaN or +-Inf (a finite value above about
// 1.8e19 squares past FP32's range) is summed again with every value multiplied
// by 2^-96 first, so its record carries the sum times 2^-192; such a record, and
// every merge that takes one in, is stored negated, its sign marking the form:
//   sum_sq >= 0:  sum = sum_sq + sum_sq_lo
//   sum_sq <  0:  sum = -(sum_sq + sum_sq_lo) * 2^192
// (an exact power-of-two scaling, so the decoded FP64 value has the precision of
// the stored one).  The host decision and the device-side gates decode with this
// one function: the same FP64 operations in the same order.
// 1 / s when s is a power of two whose inverse is a normal double, else 0.  For such
// an s, x / s and x * (1 / s) are the rounding of one and the same real number, so
// IEEE arithmetic gives them the same bits for every x (subnormal, infinite and NaN
// results included).
inline double power_of_two_inverse(double s) {
    int e = 0;
    if (!(s > 0.0) || std::frexp(s, &e) != 0.5) return 0.0;  // s = 2^(e-1)
    const int k = e - 1;
    return (k < -1022 || k > 1022) ? 0.0 : std::ldexp(1.0, -k);
}

constexpr int64_t kMaxGridX = 0x7fffffff;  // the launch limit on gridDim.x

constexpr int kRescueValueExp = 96;  // values of a rescued row are multiplied by 2^-96
__host__ __device__ inline double record_sum_sq(const fa_stats &r) {
    const double s = static_cast<double>(r.sum_sq) + static_cast<double>(r.sum_sq_lo);
    return r.sum_sq < 0.0f ? -s * 0x1p192 : s;
}

// FP32 coefficients of one update, computed on the host in FP64.
struct Coef {
    float b1, omb1, b2, omb2;
    float step_size;  // lr / (1 - beta1^t)
    float rbc2;       // 1 / (1 - beta2^t)
    float eps;
    float decay;      // 1 - lr * weight_decay
    float gmul;       // (maximize ? -1 : 1) * grad_mult / gradient_scale
};

// Pointers of one update launch.  In place: *_out == *_in.
struct UpdateArgs {
    const float *p_in, *m_in, *v_in, *vmax_in;
    const void *g;
    float *p_out, *m_out, *v_out, *vmax_out;
    void *p_model;  // low-precision copy of the updated p (nullptr: none)
    uint32_t extra_tx;  // self-test only: bytes a pipeline barrier waits for but never gets
    // Device-side decision (nullptr: none): skip when the report counts a
    // non-finite value, else gmul = sign * coef / scale with the host's formula.
    // gate_inv_scale: power_of_two_inverse(gate_scale), so that the divisions by the
    // scale can be multiplications with the same result.
    const fa_stats *gate;
    double gate_scale, gate_max_norm, gate_sign, gate_inv_scale;
    int64_t n;     // elements
    int64_t head;  // scalar elements before the 16-byte aligned vector body
    int64_t nvec;  // 8-element vectors in the body
};

// Enqueues one update kernel over a.n elements.  vector_ok: every pointer is
// 16-byte aligned at element a.head.  Returns the CUDA launch status.
// Self-test of the pipeline's bounded waits: one steady update launched with
// a.extra_tx > 0 on the TMA path, so every wait runs out; *launched is false
// when the tensor is too small for that path.
cudaError_t launch_pipeline_selftest(const UpdateArgs &a, const Coef &c, fa_dtype gdt,
                                     bool *launched, cudaStream_t stream);

// Reads (and optionally clears) the flag an update kernel sets when a bounded
// wait in its shared-memory pipeline gives up.  Waits for the device.
cudaError_t update_pipeline_error(int *flag, bool clear);

// Out-of-range accesses counted (and skipped) by each file's kernels in the
// bounds-checked build since the last clear; always 0 in the normal build.
// Wait for the device.
cudaError_t update_bounds_violations(unsigned long long *count, bool clear);
cudaError_t stats_bounds_violations(unsigned long long *count, bool clear);
cudaError_t staged_bounds_violations(unsigned long long *count, bool clear);

// model_dtype: FA_F16 or FA_BF16 when a.p_model is set, else kNoModel.
constexpr int kNoModel = -1;
cudaError_t launch_update(const UpdateArgs &a, const Coef &c, fa_dtype gdt, bool amsgrad,
                          bool first, bool vector_ok, int model_dtype, cudaStream_t stream);

// The staged comparison: 4 kernels (5 with AMSGrad) through an FP32 delta buffer.
struct StagedArgs {
    float *p, *m, *v, *vmax, *delta;
    const void *g;
    int64_t n;
};
cudaError_t launch_staged(const StagedArgs &a, const Coef &c, fa_dtype gdt, bool amsgrad,
                          bool first, cudaStream_t stream);

// Row-statistics launch over up to kMaxSegPerLaunch segments.
struct AnalyzeArgs {
    const void *g;
    int64_t n;            // elements of g (bounds-checked build)
    fa_stats *out;        // first row record of this launch
    int64_t row_len;
    int64_t rows;         // rows in this launch
    int32_t nseg;         // segments in this launch
    int64_t seg_start[kMaxSegPerLaunch + 1];  // element offsets; [nseg] = end of the last
    int64_t row_start[kMaxSegPerLaunch + 1];  // first row of each segment; [nseg] = rows
};

cudaError_t launch_analyze(const AnalyzeArgs &a, fa_dtype gdt, bool vector_ok,
                           cudaStream_t stream);

// Per-chunk merge of up to kMaxSegPerLaunch chunks: level A reduces groups of
// at most kFanIn rows within a chunk into ``partial``, level B one chunk's
// groups into out[k].
struct ChunkMergeArgs {
    const fa_stats *in;   // row records; chunk k holds [row_start[k], row_start[k+1])
    fa_stats *partial;    // group_start[nchunks] level-A records
    fa_stats *out;        // nchunks records
    int32_t nchunks;
    int64_t row_start[kMaxSegPerLaunch + 1];
    int64_t group_start[kMaxSegPerLaunch + 1];
};
cudaError_t launch_merge_chunks(const ChunkMergeArgs &a, cudaStream_t stream);

// The update with one gradient multiplier per segment (per-parameter clipping).
struct SegScaleArgs {
    UpdateArgs a;        // pointers of this launch's first element; a.n elements
    int32_t nseg;
    int64_t seg_start[kMaxSegPerLaunch + 1];  // relative to the launch's first element
    float gmul[kMaxSegPerLaunch];             // (maximize ? -1 : 1) * multiplier / scale
    // Device-side decision (reports == nullptr: gmul above is used).  reports holds
    // one 12-byte record per segment of the whole bucket: any non-finite count skips
    // the launch, and segment j of this launch takes the clip multiplier of record
    // k0 + j, computed like the host's from a.gate_scale, a.gate_max_norm, a.gate_sign.
    const fa_stats *reports;
    int64_t nreports;
    int32_t k0;
    // With reports: the decisions already taken once for the whole bucket by
    // launch_segment_decide (nullptr: each launch decides itself): decided[0] is the
    // skip flag (non-zero: skip), decided[1 + k0 + j] segment j's multiplier.
    const float *decided;
};
cudaError_t launch_update_segment_scaled(const SegScaleArgs &s, const Coef &c, fa_dtype gdt,
                                         bool amsgrad, bool first, bool vector_ok,
                                         cudaStream_t stream);

// One CTA takes every segment's decision from its record (the host formula's FP64
// operations with a.gate_scale, a.gate_inv_scale, a.gate_max_norm, a.gate_sign) into
// decided[1 + k] for k < nseg, and the skip flag (any non-finite count) into
// decided[0] (decided == nullptr: no table).  With ``post`` (device address of a
// pinned host mailbox) it also posts the bucket's record there: the exact non-finite
// count and the FP64 total of the segments' sums of squares, then ``seq``.  Launched as
// the programmatic dependent of the merge that wrote the records.
cudaError_t launch_segment_decide(const UpdateArgs &a, const fa_stats *reports, int32_t nseg,
                                  float *decided, fa_report_mailbox *post, uint32_t seq,
                                  cudaStream_t stream);

// One merge level: ceil(count / kFanIn) output records from count input records.
// ``post`` (device address of a pinned host mailbox, final level only) also receives
// the single output record, followed by ``seq``.
cudaError_t launch_merge(const fa_stats *in, int64_t count, fa_stats *out, cudaStream_t stream,
                         fa_report_mailbox *post = nullptr, uint32_t seq = 0);

// Device address and size of the library's fixed merge scratch on ``device``
// (which must be the current device).  Looked up once per device; with
// ``lookup_allowed`` false (the caller's stream is being captured) an address
// not looked up yet is not looked up now: cudaErrorStreamCaptureUnsupported.
constexpr int64_t kStaticMergeScratchFloats = 12300;  // 3 * (4096 + 4): the largest plan
cudaError_t static_merge_scratch(int device, bool lookup_allowed, float **ptr,
                                 int64_t *capacity_floats);

// SM count of the current device (cached per device).
int sm_count(int device);

// Resident CTAs per SM of ``kernel`` at ``threads`` threads (cached per device and
// kernel; >= 1), and the persistent grid for ``need`` CTAs of work.
int resident_ctas(const void *kernel, int device, int threads = kThreads);

template <typename Kernel>
inline int persistent_grid(Kernel kernel, int64_t need, int device, int threads = kThreads) {
    const int64_t cap = static_cast<int64_t>(sm_count(device)) *
                        resident_ctas(reinterpret_cast<const void *>(kernel), device, threads);
    return static_cast<int>(need < cap ? need : cap);
}

}  // namespace fa
