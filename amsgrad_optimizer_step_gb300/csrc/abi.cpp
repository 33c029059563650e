// C-ABI host layer: validation, FP64 host coefficients, the statistics plan,
// the skip / clip decision, and kernel launches.  Everything that touches the
// device goes through the kernels in update_kernels.cu, stats_kernels.cu and
// staged_kernels.cu (the staged comparison).
//
// Contract sources (RUDA documentation pages):
//   "実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw): "この演算子を使用する
//     理由" (formula, host FP64 coefficients, defaults), "サポートされている契約"
//     (flattened buckets share options and step; no host pointers), "低レベルの使用"
//     (AdamWOptions, StepControl, validation leaves inputs untouched, success =
//     enqueued), "ネイティブ PyTorch ストレージと階層統計" (storage kernels, StatsPlan).
//   "实验性融合 AdamW / AMSGrad" (zh/docs/fused-adamw): "增加的实际能力" (dtypes; empty
//     tensor or skip_update launches nothing and does not advance the step).
//   "训练与状态保存" (zh/docs/training): "在 ruda:0 上进行原生 PyTorch 训练" (12-byte
//     report read back first, non-finite skip, global clip after unscale).
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <utility>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "fused_adamw.h"
#include "internal.h"

namespace fa {

int sm_count(int device) {
    static std::atomic<int> cache[64] = {};  // immutable device property; any thread may fill it
    if (device >= 0 && device < 64) {
        const int c = cache[device].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return 0;
    if (device >= 0 && device < 64) cache[device].store(n, std::memory_order_relaxed);
    return n;
}

int resident_ctas(const void *kernel, int device, int threads) {
    // Immutable per (device, kernel, threads): computed once, then looked up.
    static std::mutex mu;
    static std::map<std::pair<std::pair<int, int>, const void *>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(std::make_pair(device, threads), kernel);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, 0) != cudaSuccess) {
        cudaGetLastError();
        occ = 0;
    }
    if (occ < 1) occ = 1;
    cache[key] = occ;
    return occ;
}

}  // namespace fa

namespace {

using fa::Coef;

bool is_finite(double x) { return std::isfinite(x); }

// beta^t as an FP64 integer power (binary exponentiation).
double int_pow(double beta, uint64_t t) {
    double r = 1.0, b = beta;
    while (t) {
        if (t & 1) r *= b;
        b *= b;
        t >>= 1;
    }
    return r;
}

fa_status check_options(const fa_options *o) {
    if (!o) return FA_ERR_NULL;
    if (!is_finite(o->lr) || o->lr < 0) return FA_ERR_OPTION;
    if (!is_finite(o->beta1) || o->beta1 < 0 || o->beta1 >= 1) return FA_ERR_OPTION;
    if (!is_finite(o->beta2) || o->beta2 < 0 || o->beta2 >= 1) return FA_ERR_OPTION;
    if (!is_finite(o->eps) || o->eps < 0) return FA_ERR_OPTION;
    if (!is_finite(o->weight_decay) || o->weight_decay < 0) return FA_ERR_OPTION;
    if ((o->amsgrad != 0 && o->amsgrad != 1) || (o->maximize != 0 && o->maximize != 1))
        return FA_ERR_OPTION;
    return FA_OK;
}

fa_status check_control(const fa_step_control &c) {
    if (!is_finite(c.gradient_scale) || c.gradient_scale <= 0) return FA_ERR_OPTION;
    if (c.skip_update != 0 && c.skip_update != 1) return FA_ERR_OPTION;
    return FA_OK;
}

bool valid_dtype(fa_dtype d) { return d == FA_F32 || d == FA_F16 || d == FA_BF16; }
size_t dtype_bytes(fa_dtype d) { return d == FA_F32 ? 4 : 2; }

// Host-side trace ranges (NVTX): a profiler attached to the process shows each
// entry point's span around the kernels it enqueues; without one they cost nothing.
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

// The current device, checked against the stream's device (the legacy default
// stream belongs to the current device).
fa_status stream_device(void *stream, int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (stream) {
        // A stream that is being captured into a graph cannot report its device
        // (the query fails and ends the capture); its work is recorded for the
        // device the capture belongs to, so the check is left out then.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_POINTER;
        }
        if (cs == cudaStreamCaptureStatusActive) return FA_OK;
        int sdev = -1;
        if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_POINTER;
        }
        if (sdev != *dev) return FA_ERR_POINTER;
    }
    return FA_OK;
}

// Device (or managed) memory of device ``dev``, aligned to ``align`` bytes.
fa_status check_device_ptr(const void *p, int dev, size_t align) {
    if (!p) return FA_ERR_NULL;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_POINTER;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return FA_ERR_POINTER;
    if (at.device != dev) return FA_ERR_POINTER;
    if (reinterpret_cast<uintptr_t>(p) % align) return FA_ERR_ALIGN;
    return FA_OK;
}

struct Range {
    const void *p;
    size_t bytes;
};

bool overlap(Range a, Range b) {
    if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool any_overlap(const Range *r, int count) {
    for (int i = 0; i < count; ++i)
        for (int j = i + 1; j < count; ++j)
            if (overlap(r[i], r[j])) return true;
    return false;
}

fa_status make_coef(const fa_options *o, uint64_t t, double scale, double grad_mult, Coef *c) {
    if (t == 0) return FA_ERR_OPTION;
    if (!is_finite(grad_mult) || grad_mult < 0) return FA_ERR_OPTION;
    const double bc1 = 1.0 - int_pow(o->beta1, t);
    const double bc2 = 1.0 - int_pow(o->beta2, t);
    if (!(bc1 > 0) || !(bc2 > 0)) return FA_ERR_OPTION;  // beta == 0 is fine; bc = 1
    c->b1 = static_cast<float>(o->beta1);
    c->omb1 = static_cast<float>(1.0 - o->beta1);
    c->b2 = static_cast<float>(o->beta2);
    c->omb2 = static_cast<float>(1.0 - o->beta2);
    c->step_size = static_cast<float>(o->lr / bc1);
    c->rbc2 = static_cast<float>(1.0 / bc2);
    c->eps = static_cast<float>(o->eps);
    c->decay = static_cast<float>(1.0 - o->lr * o->weight_decay);
    c->gmul = static_cast<float>((o->maximize ? -1.0 : 1.0) * grad_mult / scale);
    return FA_OK;
}

// First element index at which every pointer is 16-byte aligned (-1: none).
int64_t vector_head(const void *const *ptrs, const size_t *esize, int count, int64_t n) {
    for (int64_t h = 0; h < 8; ++h) {
        bool ok = true;
        for (int i = 0; i < count && ok; ++i)
            if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) + h * esize[i]) % 16) ok = false;
        if (ok) return h < n ? h : n;
    }
    return -1;
}

// Shared by the out-of-place, in-place and bucket entry points: all pointers
// already validated.
fa_status enqueue_update(int64_t n, const float *p, const void *g, fa_dtype gdt, const float *m,
                         const float *v, const float *vmax, float *p_out, float *m_out,
                         float *v_out, float *vmax_out, const fa_options *o, uint64_t t_new,
                         double scale, double grad_mult, void *stream,
                         void *p_model = nullptr, int model_dtype = fa::kNoModel,
                         const fa_stats *gate = nullptr, double gate_max_norm = 0.0) {
    Coef c;
    fa_status st = make_coef(o, t_new, scale, grad_mult, &c);
    if (st != FA_OK) return st;
    const bool first = t_new == 1;
    fa::UpdateArgs a;
    a.p_in = p;
    a.m_in = first ? nullptr : m;
    a.v_in = first ? nullptr : v;
    a.vmax_in = (first || !o->amsgrad) ? nullptr : vmax;
    a.g = g;
    a.p_out = p_out;
    a.m_out = m_out;
    a.v_out = v_out;
    a.vmax_out = o->amsgrad ? vmax_out : nullptr;
    a.p_model = model_dtype == fa::kNoModel ? nullptr : p_model;
    a.extra_tx = 0;
    a.gate = gate;
    a.gate_scale = scale;
    a.gate_max_norm = gate_max_norm;
    a.gate_sign = o->maximize ? -1.0 : 1.0;
    a.gate_inv_scale = fa::power_of_two_inverse(scale);
    a.n = n;
    const void *ptrs[] = {a.p_in, a.m_in, a.v_in, a.vmax_in, a.g,
                          a.p_out, a.m_out, a.v_out, a.vmax_out, a.p_model};
    const size_t es[] = {4, 4, 4, 4, dtype_bytes(gdt), 4, 4, 4, 4, 2};
    const int64_t head = vector_head(ptrs, es, 10, n);
    const bool vec = head >= 0;
    a.head = vec ? head : 0;
    a.nvec = vec ? (n - a.head) / 8 : 0;
    cudaError_t err = fa::launch_update(a, c, gdt, o->amsgrad != 0, first, vec,
                                        a.p_model ? model_dtype : fa::kNoModel,
                                        static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Validates the in-place argument set: device pointers, alignment, and no overlap.
fa_status check_inplace(int64_t n, float *p, const void *g, fa_dtype gdt, float *m, float *v,
                        float *vmax, const fa_options *o, int dev) {
    fa_status st;
    if ((st = check_device_ptr(p, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(g, dev, dtype_bytes(gdt))) != FA_OK) return st;
    if ((st = check_device_ptr(m, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(v, dev, 4)) != FA_OK) return st;
    if (o->amsgrad && (st = check_device_ptr(vmax, dev, 4)) != FA_OK) return st;
    if (!o->amsgrad && vmax) return FA_ERR_NULL;
    const size_t b = static_cast<size_t>(n) * 4;
    const Range r[] = {{p, b}, {g, static_cast<size_t>(n) * dtype_bytes(gdt)}, {m, b}, {v, b},
                       {o->amsgrad ? vmax : nullptr, b}};
    if (any_overlap(r, 5)) return FA_ERR_ALIAS;
    return FA_OK;
}

// The first checks of every step entry point, in this order: options, control,
// gradient dtype, element count.
fa_status check_step_args(const fa_options *o, fa_step_control ctl, fa_dtype gdt, int64_t n) {
    fa_status st;
    if ((st = check_options(o)) != FA_OK) return st;
    if ((st = check_control(ctl)) != FA_OK) return st;
    if (!valid_dtype(gdt)) return FA_ERR_DTYPE;
    return n < 0 ? FA_ERR_SIZE : FA_OK;
}

fa_status check_segments(const int64_t *seg, int32_t nseg, int64_t n) {
    if (nseg < 0) return FA_ERR_SEGMENTS;
    if (nseg == 0) return FA_OK;
    if (!seg) return FA_ERR_NULL;
    if (seg[0] != 0 || seg[nseg] != n) return FA_ERR_SEGMENTS;
    for (int32_t k = 0; k < nseg; ++k)
        if (seg[k + 1] < seg[k]) return FA_ERR_SEGMENTS;
    return FA_OK;
}

// The per-segment update, one launch per kMaxSegPerLaunch segments (arguments
// validated).  Each segment's multiplier comes from seg_grad_mult (decided on the
// host) or, with ``reports`` (device, one record per segment), is decided on the
// device from the records: any non-finite count skips every launch, and segment
// k's clip coefficient is the host formula's with max_grad_norm.  ``decided``
// (device, nseg + 1 floats, or nullptr): where the decisions are first taken once
// for the whole bucket (launch_segment_decide), for the update kernels to read.
// ``post`` (device address of a pinned mailbox, or nullptr): where that kernel also
// posts the bucket's record, then ``seq``.
fa_status enqueue_segment_update(const int64_t *seg_offsets, int32_t nseg, float *p,
                                 const void *g, fa_dtype gdt, float *m, float *v, float *vmax,
                                 uint64_t t_new, const fa_options *options, fa_step_control ctl,
                                 const double *seg_grad_mult, const fa_stats *reports,
                                 double max_grad_norm, void *stream,
                                 float *decided = nullptr, fa_report_mailbox *post = nullptr,
                                 uint32_t seq = 0) {
    Coef c;
    fa_status st = make_coef(options, t_new, ctl.gradient_scale, 1.0, &c);
    if (st != FA_OK) return st;
    const bool first = t_new == 1;
    const bool ams = options->amsgrad != 0;
    const double sign = options->maximize ? -1.0 : 1.0;
    const size_t gb = dtype_bytes(gdt);
    if (decided || post) {
        fa::UpdateArgs gate{};
        gate.gate_scale = ctl.gradient_scale;
        gate.gate_max_norm = max_grad_norm;
        gate.gate_sign = sign;
        gate.gate_inv_scale = fa::power_of_two_inverse(ctl.gradient_scale);
        if (fa::launch_segment_decide(gate, reports, nseg, decided, post, seq,
                                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    for (int32_t k0 = 0; k0 < nseg; k0 += fa::kMaxSegPerLaunch) {
        const int32_t cnt = nseg - k0 < fa::kMaxSegPerLaunch ? nseg - k0 : fa::kMaxSegPerLaunch;
        const int64_t e0 = seg_offsets[k0], e1 = seg_offsets[k0 + cnt];
        if (e1 == e0) continue;
        fa::SegScaleArgs sa;
        fa::UpdateArgs &a = sa.a;
        a.p_in = p + e0;
        a.m_in = first ? nullptr : m + e0;
        a.v_in = first ? nullptr : v + e0;
        a.vmax_in = (first || !ams) ? nullptr : vmax + e0;
        a.g = static_cast<const char *>(g) + e0 * gb;
        a.p_out = p + e0;
        a.m_out = m + e0;
        a.v_out = v + e0;
        a.vmax_out = ams ? vmax + e0 : nullptr;
        a.p_model = nullptr;
        a.extra_tx = 0;
        a.gate = nullptr;
        a.gate_scale = ctl.gradient_scale;
        a.gate_max_norm = max_grad_norm;
        a.gate_sign = sign;
        a.gate_inv_scale = fa::power_of_two_inverse(ctl.gradient_scale);
        a.n = e1 - e0;
        const void *ptrs[] = {a.p_in, a.m_in, a.v_in, a.vmax_in, a.g};
        const size_t es[] = {4, 4, 4, 4, gb};
        const int64_t head = vector_head(ptrs, es, 5, a.n);
        const bool vec = head >= 0;
        a.head = vec ? head : 0;
        a.nvec = vec ? (a.n - a.head) / 8 : 0;
        sa.nseg = cnt;
        for (int32_t j = 0; j <= cnt; ++j) sa.seg_start[j] = seg_offsets[k0 + j] - e0;
        for (int32_t j = 0; j < cnt; ++j)
            sa.gmul[j] = seg_grad_mult
                             ? static_cast<float>(sign * seg_grad_mult[k0 + j] / ctl.gradient_scale)
                             : 0.0f;
        sa.reports = reports;
        sa.nreports = reports ? nseg : 0;
        sa.k0 = k0;
        sa.decided = decided;
        if (fa::launch_update_segment_scaled(sa, c, gdt, ams, first, vec,
                                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Enqueues the merge levels of ``rows`` records (``kernels`` of them, from the plan)
// into ``report``; intermediate records go to ``scratch``.  The level that writes the
// report also posts it to ``post`` (device address of a host mailbox) when given.
fa_status enqueue_merge_levels(const fa_stats *rows_in, int64_t rows, int32_t kernels,
                               float *scratch, fa_stats *report, fa_report_mailbox *post,
                               uint32_t seq, cudaStream_t stream) {
    const fa_stats *in = rows_in;
    int64_t count = rows;
    fa_stats *next = reinterpret_cast<fa_stats *>(scratch);
    for (int32_t level = 0; level < kernels; ++level) {
        const int64_t out_count = (count + fa::kFanIn - 1) / fa::kFanIn;
        const bool last = out_count == 1;
        fa_stats *out = last ? report : next;
        if (fa::launch_merge(in, count, out, stream, last ? post : nullptr, seq) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_CUDA;
        }
        in = out;
        count = out_count;
        next = out + out_count;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int32_t fa_abi_version(void) { return FA_ABI_VERSION; }

fa_status fa_stats_sum_sq(const fa_stats *record, double *sum_sq) {
    if (!record || !sum_sq) return FA_ERR_NULL;
    *sum_sq = fa::record_sum_sq(*record);
    return FA_OK;
}

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "null pointer, or state pointers inconsistent with the step count";
        case FA_ERR_DTYPE: return "unsupported gradient dtype";
        case FA_ERR_SIZE: return "negative size or buffer too small";
        case FA_ERR_OPTION: return "option or control value out of range";
        case FA_ERR_ALIAS: return "buffers overlap";
        case FA_ERR_POINTER: return "not device memory of the current device";
        case FA_ERR_ALIGN: return "pointer not aligned to its element size";
        case FA_ERR_PLAN: return "statistics rows outside 1..4194304";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_SEGMENTS: return "malformed segment table";
    }
    return "unknown status";
}

fa_status fa_device_error(int32_t *flag, int32_t clear) {
    if (!flag) return FA_ERR_NULL;
    int v = 0;
    if (fa::update_pipeline_error(&v, clear != 0) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    *flag = v;
    return FA_OK;
}

fa_status fa_bounds_check_report(int32_t *enabled, uint64_t *violations, int32_t clear) {
    if (!enabled) return FA_ERR_NULL;
    *enabled = FA_BOUNDS_CHECK;
    if (!violations) return FA_OK;
#if FA_BOUNDS_CHECK
    unsigned long long a = 0, b = 0, c = 0;
    if (fa::update_bounds_violations(&a, clear != 0) != cudaSuccess ||
        fa::stats_bounds_violations(&b, clear != 0) != cudaSuccess ||
        fa::staged_bounds_violations(&c, clear != 0) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    *violations = a + b + c;
#else
    (void)clear;
    *violations = 0;
#endif
    return FA_OK;
}

fa_status fa_pipeline_selftest(int64_t n, float *p, const void *g, fa_dtype gdt, float *m,
                               float *v, int32_t *flag, void *stream) {
    if (!flag) return FA_ERR_NULL;
    if (!valid_dtype(gdt)) return FA_ERR_DTYPE;
    if (n < 1) return FA_ERR_SIZE;
    fa_options o = fa_options_default();
    int dev = 0;
    fa_status st;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n, p, g, gdt, m, v, nullptr, &o, dev)) != FA_OK) return st;
    Coef c;
    if ((st = make_coef(&o, 2, 1.0, 1.0, &c)) != FA_OK) return st;
    fa::UpdateArgs a;
    a.p_in = p;
    a.m_in = m;
    a.v_in = v;
    a.vmax_in = nullptr;
    a.g = g;
    a.p_out = p;
    a.m_out = m;
    a.v_out = v;
    a.vmax_out = nullptr;
    a.p_model = nullptr;
    a.extra_tx = 16;  // a barrier that waits for 16 bytes nobody sends
    a.gate = nullptr;
    a.gate_scale = a.gate_max_norm = a.gate_sign = a.gate_inv_scale = 0.0;
    a.n = n;
    const void *ptrs[] = {p, m, v, g};
    const size_t es[] = {4, 4, 4, dtype_bytes(gdt)};
    const int64_t head = vector_head(ptrs, es, 4, n);
    if (head < 0) return FA_ERR_ALIGN;
    a.head = head;
    a.nvec = (n - head) / 8;
    int prior = 0;
    if (fa::update_pipeline_error(&prior, true) != cudaSuccess) return FA_ERR_CUDA;
    bool launched = false;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fa::launch_pipeline_selftest(a, c, gdt, &launched, s) != cudaSuccess) return FA_ERR_CUDA;
    if (!launched) return FA_ERR_SIZE;
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    int v_flag = 0;
    if (fa::update_pipeline_error(&v_flag, true) != cudaSuccess) return FA_ERR_CUDA;
    *flag = v_flag;
    return FA_OK;
}

fa_options fa_options_default(void) {
    fa_options o;
    o.lr = 1e-3;
    o.beta1 = 0.9;
    o.beta2 = 0.999;
    o.eps = 1e-5;
    o.weight_decay = 1e-4;
    o.amsgrad = 0;
    o.maximize = 0;
    return o;
}

fa_status fa_step_coefficients(const fa_options *options, uint64_t t, double gradient_scale,
                               double grad_mult, float coef_out[9]) {
    fa_status st = check_options(options);
    if (st != FA_OK) return st;
    if (!coef_out) return FA_ERR_NULL;
    fa_step_control ctl{gradient_scale, 0};
    if ((st = check_control(ctl)) != FA_OK) return st;
    Coef c;
    if ((st = make_coef(options, t, gradient_scale, grad_mult, &c)) != FA_OK) return st;
    const float v[9] = {c.b1, c.omb1, c.b2, c.omb2, c.step_size, c.rbc2, c.eps, c.decay, c.gmul};
    std::memcpy(coef_out, v, sizeof v);
    return FA_OK;
}

fa_status fa_adamw_step(int64_t n, const float *p, const void *g, fa_dtype gdt, const float *m,
                        const float *v, const float *vmax, uint64_t t_in,
                        const fa_options *options, fa_step_control ctl, float *p_out,
                        float *m_out, float *v_out, float *vmax_out, uint64_t *t_out,
                        int32_t *updated, void *stream) {
    TraceRange trace("fa_adamw_step");
    fa_status st;
    if (!t_out || !updated) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n)) != FA_OK) return st;
    if (n == 0 || ctl.skip_update) {  // nothing launched, no buffer touched or checked
        *t_out = t_in;
        *updated = 0;
        return FA_OK;
    }
    const bool ams = options->amsgrad != 0;
    // State is None before the first update: all moment pointers NULL.
    if (t_in == 0) {
        if (m || v || vmax) return FA_ERR_NULL;
    } else {
        if (!m || !v || (ams != (vmax != nullptr))) return FA_ERR_NULL;
    }
    if (t_in == UINT64_MAX) return FA_ERR_OPTION;
    {
        int dev = 0;
        if ((st = stream_device(stream, &dev)) != FA_OK) return st;
        const size_t gb = dtype_bytes(gdt);
        if ((st = check_device_ptr(p, dev, 4)) != FA_OK) return st;
        if ((st = check_device_ptr(g, dev, gb)) != FA_OK) return st;
        if (t_in > 0) {
            if ((st = check_device_ptr(m, dev, 4)) != FA_OK) return st;
            if ((st = check_device_ptr(v, dev, 4)) != FA_OK) return st;
            if (ams && (st = check_device_ptr(vmax, dev, 4)) != FA_OK) return st;
        }
        if ((st = check_device_ptr(p_out, dev, 4)) != FA_OK) return st;
        if ((st = check_device_ptr(m_out, dev, 4)) != FA_OK) return st;
        if ((st = check_device_ptr(v_out, dev, 4)) != FA_OK) return st;
        if (ams && (st = check_device_ptr(vmax_out, dev, 4)) != FA_OK) return st;
        if (!ams && vmax_out) return FA_ERR_NULL;
        const size_t b = static_cast<size_t>(n) * 4;
        const Range outs[] = {{p_out, b}, {m_out, b}, {v_out, b}, {ams ? vmax_out : nullptr, b}};
        const Range ins[] = {{p, b}, {g, static_cast<size_t>(n) * gb}, {m, b}, {v, b},
                             {ams ? vmax : nullptr, b}};
        if (any_overlap(outs, 4)) return FA_ERR_ALIAS;
        for (const Range &o : outs)
            for (const Range &i : ins)
                if (overlap(o, i)) return FA_ERR_ALIAS;
    }
    st = enqueue_update(n, p, g, gdt, m, v, vmax, p_out, m_out, v_out, vmax_out, options,
                        t_in + 1, ctl.gradient_scale, 1.0, stream);
    if (st != FA_OK) return st;
    *t_out = t_in + 1;
    *updated = 1;
    return FA_OK;
}

fa_status fa_adamw_step_inplace(int64_t n, float *p, const void *g, fa_dtype gdt, float *m,
                                float *v, float *vmax, uint64_t *t,
                                const fa_options *options, fa_step_control ctl,
                                double grad_mult, int32_t *updated, void *stream) {
    TraceRange trace("fa_adamw_step_inplace");
    fa_status st;
    if (!t || !updated) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n)) != FA_OK) return st;
    if (!is_finite(grad_mult) || grad_mult < 0) return FA_ERR_OPTION;
    if (n == 0 || ctl.skip_update) {  // nothing launched, no buffer touched or checked
        *updated = 0;
        return FA_OK;
    }
    if (*t == UINT64_MAX) return FA_ERR_OPTION;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    st = enqueue_update(n, p, g, gdt, m, v, vmax, p, m, v, vmax, options, *t + 1,
                        ctl.gradient_scale, grad_mult, stream);
    if (st != FA_OK) return st;
    *t += 1;
    *updated = 1;
    return FA_OK;
}

fa_status fa_bucket_step(const int64_t *seg_offsets, int32_t nseg, int64_t n_total, float *p,
                         const void *g, fa_dtype gdt, float *m, float *v, float *vmax,
                         uint64_t *t, const fa_options *options, fa_step_control ctl,
                         double grad_mult, int32_t *updated, void *stream) {
    TraceRange trace("fa_bucket_step");
    if (n_total < 0) return FA_ERR_SIZE;
    fa_status st = check_segments(seg_offsets, nseg, n_total);
    if (st != FA_OK) return st;
    return fa_adamw_step_inplace(n_total, p, g, gdt, m, v, vmax, t, options, ctl, grad_mult,
                                 updated, stream);
}

fa_status fa_bucket_update(const fa_bucket_update_args *u, const fa_options *options,
                           fa_step_control ctl, int32_t *enqueued, void *stream) {
    TraceRange trace("fa_bucket_update");
    fa_status st;
    if (!u || !enqueued) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, u->gdt, u->n_total)) != FA_OK) return st;
    const bool per_segment = u->seg_grad_mult || u->seg_reports;
    const bool on_device = u->report || u->seg_reports;
    const int sources = (u->seg_grad_mult != nullptr) + (u->report != nullptr) +
                        (u->seg_reports != nullptr);
    if (sources > 1) return FA_ERR_OPTION;
    if (!is_finite(u->grad_mult) || u->grad_mult < 0) return FA_ERR_OPTION;
    if (sources == 1 && u->grad_mult != 1.0) return FA_ERR_OPTION;
    if (on_device && std::isnan(u->max_grad_norm)) return FA_ERR_OPTION;
    if (u->p_model) {
        if (u->model_dtype != FA_F16 && u->model_dtype != FA_BF16) return FA_ERR_DTYPE;
        if (per_segment) return FA_ERR_OPTION;  // no per-segment kernel writes a model copy
    }
    if (u->seg_decided && !u->seg_reports) return FA_ERR_OPTION;
    if (per_segment && u->nseg < 1) return FA_ERR_SEGMENTS;
    if ((st = check_segments(u->seg_offsets, u->nseg, u->n_total)) != FA_OK) return st;
    if (u->seg_decided && u->seg_decided_elements < static_cast<int64_t>(u->nseg) + 1)
        return FA_ERR_SIZE;
    if (u->seg_grad_mult)
        for (int32_t k = 0; k < u->nseg; ++k)
            if (!is_finite(u->seg_grad_mult[k]) || u->seg_grad_mult[k] < 0) return FA_ERR_OPTION;
    if (u->n_total == 0 || ctl.skip_update) {  // nothing launched, no buffer touched or checked
        *enqueued = 0;
        return FA_OK;
    }
    if (u->t == UINT64_MAX) return FA_ERR_OPTION;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(u->n_total, u->p, u->g, u->gdt, u->m, u->v, u->vmax, options, dev)) !=
        FA_OK)
        return st;
    if (u->p_model && (st = check_device_ptr(u->p_model, dev, 2)) != FA_OK) return st;
    const fa_stats *reports = u->report ? u->report : u->seg_reports;
    if (reports && (st = check_device_ptr(reports, dev, 4)) != FA_OK) return st;
    // the model copy and the reports must stay clear of every buffer the update touches
    const size_t b = static_cast<size_t>(u->n_total) * 4;
    const Range model{u->p_model, static_cast<size_t>(u->n_total) * 2};
    const Range rep{reports, static_cast<size_t>(u->report ? 1 : u->nseg) * 12};
    const Range state[] = {{u->p, b},
                           {u->g, static_cast<size_t>(u->n_total) * dtype_bytes(u->gdt)},
                           {u->m, b},
                           {u->v, b},
                           {options->amsgrad ? u->vmax : nullptr, b}};
    for (const Range &r : state)
        if (overlap(model, r) || overlap(rep, r)) return FA_ERR_ALIAS;
    if (overlap(model, rep)) return FA_ERR_ALIAS;
    if (u->seg_decided) {
        if ((st = check_device_ptr(u->seg_decided, dev, 4)) != FA_OK) return st;
        const Range dec{u->seg_decided, (static_cast<size_t>(u->nseg) + 1) * 4};
        for (const Range &r : state)
            if (overlap(dec, r)) return FA_ERR_ALIAS;
        if (overlap(dec, rep)) return FA_ERR_ALIAS;
    }
    if (per_segment)
        st = enqueue_segment_update(u->seg_offsets, u->nseg, u->p, u->g, u->gdt, u->m, u->v,
                                    u->vmax, u->t + 1, options, ctl, u->seg_grad_mult,
                                    u->seg_reports, u->max_grad_norm, stream, u->seg_decided);
    else
        st = enqueue_update(u->n_total, u->p, u->g, u->gdt, u->m, u->v, u->vmax, u->p, u->m, u->v,
                            u->vmax, options, u->t + 1, ctl.gradient_scale, u->grad_mult, stream,
                            u->p_model, u->p_model ? u->model_dtype : fa::kNoModel, u->report,
                            u->max_grad_norm);
    if (st != FA_OK) return st;
    *enqueued = 1;
    return FA_OK;
}

fa_status fa_adamw_step_staged(int64_t n, float *p, const void *g, fa_dtype gdt, float *m,
                               float *v, float *vmax, uint64_t *t, const fa_options *options,
                               fa_step_control ctl, double grad_mult, float *delta,
                               int32_t *updated, void *stream) {
    TraceRange trace("fa_adamw_step_staged");
    fa_status st;
    if (!t || !updated) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n)) != FA_OK) return st;
    if (!is_finite(grad_mult) || grad_mult < 0) return FA_ERR_OPTION;
    if (n == 0 || ctl.skip_update) {  // nothing launched, no buffer touched or checked
        *updated = 0;
        return FA_OK;
    }
    if (*t == UINT64_MAX) return FA_ERR_OPTION;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    if ((st = check_device_ptr(delta, dev, 4)) != FA_OK) return st;
    const size_t b = static_cast<size_t>(n) * 4;
    const Range others[] = {{p, b}, {g, static_cast<size_t>(n) * dtype_bytes(gdt)}, {m, b},
                            {v, b}, {options->amsgrad ? vmax : nullptr, b}};
    for (const Range &r : others)
        if (overlap({delta, b}, r)) return FA_ERR_ALIAS;
    // the stages move 16-byte vectors from the first element: every stream aligned
    const void *ptrs[] = {p, m, v, options->amsgrad ? vmax : nullptr, delta};
    for (const void *q : ptrs)
        if (q && reinterpret_cast<uintptr_t>(q) % 16) return FA_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(g) % (gdt == FA_F32 ? 16 : 8)) return FA_ERR_ALIGN;
    Coef c;
    if ((st = make_coef(options, *t + 1, ctl.gradient_scale, grad_mult, &c)) != FA_OK) return st;
    fa::StagedArgs a{p, m, v, options->amsgrad ? vmax : nullptr, delta, g, n};
    if (fa::launch_staged(a, c, gdt, options->amsgrad != 0, *t == 0,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    *t += 1;
    *updated = 1;
    return FA_OK;
}

namespace {

// The device address of a caller's report mailbox: pinned host memory that the
// device can write (cudaHostAlloc, or registered and mapped, with unified
// addressing).  Pageable or device memory: FA_ERR_POINTER.
fa_status mailbox_device_ptr(fa_report_mailbox *mailbox, fa_report_mailbox **dev_ptr) {
    if (!mailbox) return FA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(mailbox) % 4) return FA_ERR_ALIGN;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, mailbox) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_POINTER;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return FA_ERR_POINTER;
    *dev_ptr = static_cast<fa_report_mailbox *>(attr.devicePointer);
    return FA_OK;
}

// Waits until the device has posted report ``seq`` to the mailbox, then copies the
// report out.  The wait ends early with FA_ERR_CUDA when the stream reports an
// error, or when the stream has finished without the report having been posted;
// and in any case after five minutes.
fa_status wait_for_post(const fa_report_mailbox *mailbox, uint32_t seq, cudaStream_t stream,
                        fa_stats *out) {
    const uint32_t *seq_word = &mailbox->seq;
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::minutes(5);
    for (uint64_t it = 0;; ++it) {
        if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) == seq) break;
        if (it % 4096 == 4095) {  // now and then: is the stream still able to post it?
            const cudaError_t q = cudaStreamQuery(stream);
            if (q != cudaSuccess && q != cudaErrorNotReady) {
                cudaGetLastError();
                return FA_ERR_CUDA;
            }
            if (q == cudaSuccess && __atomic_load_n(seq_word, __ATOMIC_ACQUIRE) != seq)
                return FA_ERR_CUDA;  // all work done and nothing posted
            if (std::chrono::steady_clock::now() > deadline) return FA_ERR_CUDA;
        }
        if (it > 256) std::this_thread::yield();
    }
    const volatile uint32_t *w = reinterpret_cast<const volatile uint32_t *>(&mailbox->report);
    const uint32_t words[3] = {w[0], w[1], w[2]};
    std::memcpy(&out->sum_sq, &words[0], 4);
    out->nonfinite = words[1];
    std::memcpy(&out->sum_sq_lo, &words[2], 4);
    return FA_OK;
}

}  // namespace

fa_status fa_bucket_step_clipped_gated(const int64_t *seg_offsets, int32_t nseg, int64_t n_total,
                                       float *p, const void *g, fa_dtype gdt, float *m, float *v,
                                       float *vmax, uint64_t *t, const fa_options *options,
                                       fa_step_control ctl, double max_grad_norm,
                                       int32_t row_len, fa_stats *rows_buf,
                                       int64_t rows_capacity, float *scratch,
                                       int64_t scratch_elements, fa_stats *report_dev,
                                       fa_report_mailbox *mailbox, fa_step_report *out,
                                       void *stream) {
    TraceRange trace("fa_bucket_step_clipped_gated");
    fa_status st;
    if (!t || !out) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n_total)) != FA_OK) return st;
    if (std::isnan(max_grad_norm)) return FA_ERR_OPTION;
    if ((st = check_segments(seg_offsets, nseg, n_total)) != FA_OK) return st;
    if (*t == UINT64_MAX) return FA_ERR_OPTION;
    fa_step_report rep{0, 0, 0, 0.0, 1.0};
    if (n_total == 0 || ctl.skip_update) {
        *out = rep;
        return FA_OK;
    }
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n_total, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    int64_t rows = 0;
    if ((st = fa_stats_rows(n_total, row_len, seg_offsets, nseg, &rows)) != FA_OK) return st;
    int32_t kernels = 0;
    int64_t need = 0;
    if ((st = fa_stats_plan(rows, &kernels, &need)) != FA_OK) return st;
    if (rows_capacity < rows || scratch_elements < need) return FA_ERR_SIZE;
    const size_t b = static_cast<size_t>(n_total) * 4;
    const Range r[] = {{p, b}, {g, static_cast<size_t>(n_total) * dtype_bytes(gdt)}, {m, b},
                       {v, b}, {options->amsgrad ? vmax : nullptr, b},
                       {rows_buf, static_cast<size_t>(rows) * 12},
                       {scratch, static_cast<size_t>(need) * 4}, {report_dev, 12}};
    if (any_overlap(r, 8)) return FA_ERR_ALIAS;
    if (need > 0 && (st = check_device_ptr(scratch, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(report_dev, dev, 4)) != FA_OK) return st;
    fa_report_mailbox *post = nullptr;
    if ((st = mailbox_device_ptr(mailbox, &post)) != FA_OK) return st;
    const uint32_t seq = __atomic_load_n(&mailbox->seq, __ATOMIC_ACQUIRE) + 1;

    if ((st = fa_analyze_gradient(g, gdt, n_total, row_len, seg_offsets, nseg, rows_buf,
                                  rows_capacity, stream)) != FA_OK)
        return st;
    // the merge that writes the report also posts it to the mailbox; no stream
    // operation sits between it and the update, which starts as its dependent
    if ((st = enqueue_merge_levels(rows_buf, rows, kernels, scratch, report_dev, post, seq,
                                   static_cast<cudaStream_t>(stream))) != FA_OK)
        return st;
    if ((st = enqueue_update(n_total, p, g, gdt, m, v, vmax, p, m, v, vmax, options, *t + 1,
                             ctl.gradient_scale, 1.0, stream, nullptr, fa::kNoModel, report_dev,
                             max_grad_norm)) != FA_OK)
        return st;
    // meanwhile the host reads the same report and takes the same decision
    fa_stats h{};
    if ((st = wait_for_post(mailbox, seq, static_cast<cudaStream_t>(stream), &h)) != FA_OK)
        return st;
    int32_t skip = 0;
    double norm = 0, coef = 1;
    const double sum = fa::record_sum_sq(h);
    if ((st = fa_clip_decision(sum, h.nonfinite, ctl.gradient_scale, max_grad_norm, &skip, &norm,
                               &coef)) != FA_OK)
        return st;
    rep.nonfinite = h.nonfinite;
    rep.grad_norm = norm;
    rep.clip_coef = coef;
    if (skip) {
        rep.skipped_nonfinite = 1;
    } else {
        *t += 1;
        rep.updated = 1;
    }
    *out = rep;
    return FA_OK;
}

// ---- statistics ---------------------------------------------------------------

fa_status fa_stats_plan(int64_t rows, int32_t *merge_kernels, int64_t *scratch_elements) {
    if (!merge_kernels || !scratch_elements) return FA_ERR_NULL;
    if (rows < 1 || rows > fa::kMaxRows) return FA_ERR_PLAN;
    int32_t k = 0;
    int64_t scratch_records = 0;
    for (int64_t c = rows;;) {
        c = (c + fa::kFanIn - 1) / fa::kFanIn;
        ++k;
        if (c == 1) break;
        scratch_records += c;
    }
    *merge_kernels = k;
    *scratch_elements = 3 * scratch_records;  // 12-byte records = 3 FP32 words
    return FA_OK;
}

fa_status fa_stats_rows(int64_t n, int32_t row_len, const int64_t *seg_offsets, int32_t nseg,
                        int64_t *rows) {
    if (!rows) return FA_ERR_NULL;
    if (n < 0 || row_len <= 0) return FA_ERR_SIZE;
    fa_status st = check_segments(seg_offsets, nseg, n);
    if (st != FA_OK) return st;
    int64_t r = 0;
    if (nseg == 0) {
        r = (n + row_len - 1) / row_len;
    } else {
        for (int32_t k = 0; k < nseg; ++k)
            r += (seg_offsets[k + 1] - seg_offsets[k] + row_len - 1) / row_len;
    }
    *rows = r;
    return FA_OK;
}

fa_status fa_analyze_gradient(const void *g, fa_dtype gdt, int64_t n, int32_t row_len,
                              const int64_t *seg_offsets, int32_t nseg, fa_stats *rows_out,
                              int64_t rows_capacity, void *stream) {
    TraceRange trace("fa_analyze_gradient");
    if (!valid_dtype(gdt)) return FA_ERR_DTYPE;
    int64_t rows = 0;
    fa_status st = fa_stats_rows(n, row_len, seg_offsets, nseg, &rows);
    if (st != FA_OK) return st;
    if (rows < 1 || rows > fa::kMaxRows) return FA_ERR_PLAN;
    if (rows_capacity < rows) return FA_ERR_SIZE;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    const size_t gb = dtype_bytes(gdt);
    if ((st = check_device_ptr(g, dev, gb)) != FA_OK) return st;
    if ((st = check_device_ptr(rows_out, dev, 4)) != FA_OK) return st;
    if (overlap({g, static_cast<size_t>(n) * gb}, {rows_out, static_cast<size_t>(rows) * 12}))
        return FA_ERR_ALIAS;

    const int64_t one[2] = {0, n};
    const int64_t *seg = nseg == 0 ? one : seg_offsets;
    const int32_t ns = nseg == 0 ? 1 : nseg;
    // 16-byte loads need every row start aligned: aligned base, segment starts
    // and row length all multiples of 16 bytes.
    bool vec = reinterpret_cast<uintptr_t>(g) % 16 == 0 && (row_len * gb) % 16 == 0;
    for (int32_t k = 0; k < ns && vec; ++k) vec = (seg[k] * gb) % 16 == 0;

    int64_t row_base = 0;
    for (int32_t k0 = 0; k0 < ns; k0 += fa::kMaxSegPerLaunch) {
        const int32_t cnt = ns - k0 < fa::kMaxSegPerLaunch ? ns - k0 : fa::kMaxSegPerLaunch;
        fa::AnalyzeArgs a;
        a.g = g;
        a.n = n;
        a.out = rows_out + row_base;
        a.row_len = row_len;
        a.nseg = cnt;
        int64_t r = 0;
        for (int32_t j = 0; j <= cnt; ++j) {
            a.seg_start[j] = seg[k0 + j];
            a.row_start[j] = r;
            if (j < cnt) r += (seg[k0 + j + 1] - seg[k0 + j] + row_len - 1) / row_len;
        }
        a.rows = r;
        if (r > 0) {
            cudaError_t err = fa::launch_analyze(a, gdt, vec, static_cast<cudaStream_t>(stream));
            if (err != cudaSuccess) return FA_ERR_CUDA;
        }
        row_base += r;
    }
    return FA_OK;
}

fa_status fa_merge_gradient_stats(const fa_stats *rows_in, int64_t rows, float *scratch,
                                  int64_t scratch_elements, fa_stats *report, void *stream) {
    TraceRange trace("fa_merge_gradient_stats");
    int32_t kernels = 0;
    int64_t need = 0;
    fa_status st = fa_stats_plan(rows, &kernels, &need);
    if (st != FA_OK) return st;
    if (scratch_elements < need || (need > 0 && !scratch)) return FA_ERR_SIZE;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_device_ptr(rows_in, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(report, dev, 4)) != FA_OK) return st;
    if (need > 0 && (st = check_device_ptr(scratch, dev, 4)) != FA_OK) return st;
    const Range r[] = {{rows_in, static_cast<size_t>(rows) * 12},
                       {scratch, static_cast<size_t>(need) * 4},
                       {report, 12}};
    if (any_overlap(r, 3)) return FA_ERR_ALIAS;
    return enqueue_merge_levels(rows_in, rows, kernels, scratch, report, nullptr, 0,
                                static_cast<cudaStream_t>(stream));
}

fa_status fa_merge_gradient_stats_static(const fa_stats *rows_in, int64_t rows,
                                         fa_stats *report, void *stream) {
    TraceRange trace("fa_merge_gradient_stats_static");
    int32_t kernels = 0;
    int64_t need = 0;
    fa_status st = fa_stats_plan(rows, &kernels, &need);
    if (st != FA_OK) return st;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_device_ptr(rows_in, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(report, dev, 4)) != FA_OK) return st;
    if (overlap({rows_in, static_cast<size_t>(rows) * 12}, {report, 12})) return FA_ERR_ALIAS;
    // While the stream is being captured, stream_device could not check the
    // stream's device, and a first address lookup must not run inside the
    // capture: only an address an earlier call looked up for the current device
    // is used then; without one the call fails with nothing enqueued.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (stream && cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_POINTER;
    }
    float *scratch = nullptr;
    int64_t capacity = 0;
    if (fa::static_merge_scratch(dev, cs == cudaStreamCaptureStatusNone, &scratch, &capacity) !=
        cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (need > capacity) return FA_ERR_SIZE;
    return enqueue_merge_levels(rows_in, rows, kernels, scratch, report, nullptr, 0,
                                static_cast<cudaStream_t>(stream));
}

// ---- per-chunk (per-parameter) statistics and clipping ------------------------

fa_status fa_stats_chunk_scratch(const int64_t *chunk_rows, int32_t nchunks,
                                 int64_t *scratch_elements) {
    if (!scratch_elements) return FA_ERR_NULL;
    if (nchunks < 1) return FA_ERR_SEGMENTS;
    if (!chunk_rows) return FA_ERR_NULL;
    if (chunk_rows[0] != 0) return FA_ERR_SEGMENTS;
    int64_t groups = 0;
    for (int32_t k = 0; k < nchunks; ++k) {
        const int64_t r = chunk_rows[k + 1] - chunk_rows[k];
        if (r < 0) return FA_ERR_SEGMENTS;
        groups += (r + fa::kFanIn - 1) / fa::kFanIn;
    }
    if (chunk_rows[nchunks] < 1 || chunk_rows[nchunks] > fa::kMaxRows) return FA_ERR_PLAN;
    *scratch_elements = 3 * groups;
    return FA_OK;
}

fa_status fa_merge_gradient_stats_chunks(const fa_stats *rows_in, const int64_t *chunk_rows,
                                         int32_t nchunks, float *scratch,
                                         int64_t scratch_elements, fa_stats *chunk_reports,
                                         void *stream) {
    TraceRange trace("fa_merge_gradient_stats_chunks");
    int64_t need = 0;
    fa_status st = fa_stats_chunk_scratch(chunk_rows, nchunks, &need);
    if (st != FA_OK) return st;
    if (scratch_elements < need || !scratch) return FA_ERR_SIZE;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_device_ptr(rows_in, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(chunk_reports, dev, 4)) != FA_OK) return st;
    if ((st = check_device_ptr(scratch, dev, 4)) != FA_OK) return st;
    const int64_t rows = chunk_rows[nchunks];
    const Range r[] = {{rows_in, static_cast<size_t>(rows) * 12},
                       {scratch, static_cast<size_t>(need) * 4},
                       {chunk_reports, static_cast<size_t>(nchunks) * 12}};
    if (any_overlap(r, 3)) return FA_ERR_ALIAS;
    fa_stats *partial = reinterpret_cast<fa_stats *>(scratch);
    for (int32_t k0 = 0; k0 < nchunks; k0 += fa::kMaxSegPerLaunch) {
        const int32_t cnt =
            nchunks - k0 < fa::kMaxSegPerLaunch ? nchunks - k0 : fa::kMaxSegPerLaunch;
        fa::ChunkMergeArgs a;
        a.in = rows_in + chunk_rows[k0];
        a.partial = partial;
        a.out = chunk_reports + k0;
        a.nchunks = cnt;
        int64_t groups = 0;
        for (int32_t j = 0; j <= cnt; ++j) {
            a.row_start[j] = chunk_rows[k0 + j] - chunk_rows[k0];
            a.group_start[j] = groups;
            if (j < cnt)
                groups += (chunk_rows[k0 + j + 1] - chunk_rows[k0 + j] + fa::kFanIn - 1) / fa::kFanIn;
        }
        if (fa::launch_merge_chunks(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FA_ERR_CUDA;
        partial += groups;
    }
    return FA_OK;
}

fa_status fa_bucket_step_clipped_per_segment(
    const int64_t *seg_offsets, int32_t nseg, int64_t n_total, float *p, const void *g,
    fa_dtype gdt, float *m, float *v, float *vmax, uint64_t *t, const fa_options *options,
    fa_step_control ctl, double max_grad_norm, int32_t row_len, fa_stats *rows_buf,
    int64_t rows_capacity, float *scratch, int64_t scratch_elements, fa_stats *seg_reports,
    double *seg_norms, double *seg_coefs, fa_step_report *out, void *stream) {
    TraceRange trace("fa_bucket_step_clipped_per_segment");
    fa_status st;
    if (!t || !out) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n_total)) != FA_OK) return st;
    if (row_len <= 0) return FA_ERR_SIZE;
    if (nseg < 1) return FA_ERR_SEGMENTS;
    if ((st = check_segments(seg_offsets, nseg, n_total)) != FA_OK) return st;
    if (std::isnan(max_grad_norm)) return FA_ERR_OPTION;
    if (*t == UINT64_MAX) return FA_ERR_OPTION;
    fa_step_report rep{0, 0, 0, 0.0, 1.0};
    if (n_total == 0 || ctl.skip_update) {
        *out = rep;
        return FA_OK;
    }
    std::vector<int64_t> chunk_rows(static_cast<size_t>(nseg) + 1, 0);
    for (int32_t k = 0; k < nseg; ++k)
        chunk_rows[k + 1] = chunk_rows[k] + (seg_offsets[k + 1] - seg_offsets[k] + row_len - 1) / row_len;
    int64_t need = 0;
    if ((st = fa_stats_chunk_scratch(chunk_rows.data(), nseg, &need)) != FA_OK) return st;
    if (scratch_elements < need || rows_capacity < chunk_rows[nseg]) return FA_ERR_SIZE;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n_total, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    if ((st = fa_analyze_gradient(g, gdt, n_total, row_len, seg_offsets, nseg, rows_buf,
                                  rows_capacity, stream)) != FA_OK)
        return st;
    if ((st = fa_merge_gradient_stats_chunks(rows_buf, chunk_rows.data(), nseg, scratch,
                                             scratch_elements, seg_reports, stream)) != FA_OK)
        return st;
    std::vector<fa_stats> host(static_cast<size_t>(nseg));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host.data(), seg_reports, host.size() * sizeof(fa_stats),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    std::vector<double> coef(static_cast<size_t>(nseg), 1.0);
    double total = 0.0, min_coef = 1.0;
    uint64_t bad = 0;
    for (int32_t k = 0; k < nseg; ++k) {
        const double sum = fa::record_sum_sq(host[k]);
        int32_t skip = 0;
        double norm = 0.0;
        if ((st = fa_clip_decision(sum, host[k].nonfinite, ctl.gradient_scale, max_grad_norm, &skip,
                                   &norm, &coef[k])) != FA_OK)
            return st;
        bad += host[k].nonfinite;
        if (!skip) total += sum;
        if (coef[k] < min_coef) min_coef = coef[k];
        if (seg_norms) seg_norms[k] = norm;
        if (seg_coefs) seg_coefs[k] = coef[k];
    }
    rep.nonfinite = bad;
    rep.grad_norm = std::sqrt(total) / ctl.gradient_scale;
    rep.clip_coef = min_coef;
    if (bad > 0) {  // any non-finite value skips the whole step
        rep.skipped_nonfinite = 1;
        *out = rep;
        return FA_OK;
    }
    if ((st = enqueue_segment_update(seg_offsets, nseg, p, g, gdt, m, v, vmax, *t + 1, options,
                                     ctl, coef.data(), nullptr, 0.0, stream)) != FA_OK)
        return st;
    *t += 1;
    rep.updated = 1;
    *out = rep;
    return FA_OK;
}

fa_status fa_bucket_step_clipped_per_segment_gated(
    const int64_t *seg_offsets, int32_t nseg, int64_t n_total, float *p, const void *g,
    fa_dtype gdt, float *m, float *v, float *vmax, uint64_t t, const fa_options *options,
    fa_step_control ctl, double max_grad_norm, int32_t row_len, fa_stats *rows_buf,
    int64_t rows_capacity, float *scratch, int64_t scratch_elements, fa_stats *seg_reports,
    fa_report_mailbox *mailbox, void *stream) {
    TraceRange trace("fa_bucket_step_clipped_per_segment_gated");
    fa_status st;
    if ((st = check_step_args(options, ctl, gdt, n_total)) != FA_OK) return st;
    if (row_len <= 0) return FA_ERR_SIZE;
    if (nseg < 1) return FA_ERR_SEGMENTS;
    if ((st = check_segments(seg_offsets, nseg, n_total)) != FA_OK) return st;
    if (std::isnan(max_grad_norm)) return FA_ERR_OPTION;
    if (t == UINT64_MAX) return FA_ERR_OPTION;
    if (n_total == 0 || ctl.skip_update) return FA_OK;
    std::vector<int64_t> chunk_rows(static_cast<size_t>(nseg) + 1, 0);
    for (int32_t k = 0; k < nseg; ++k)
        chunk_rows[k + 1] = chunk_rows[k] + (seg_offsets[k + 1] - seg_offsets[k] + row_len - 1) / row_len;
    int64_t need = 0;
    if ((st = fa_stats_chunk_scratch(chunk_rows.data(), nseg, &need)) != FA_OK) return st;
    if (scratch_elements < need || rows_capacity < chunk_rows[nseg]) return FA_ERR_SIZE;
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n_total, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    if ((st = check_device_ptr(seg_reports, dev, 4)) != FA_OK) return st;
    const size_t b = static_cast<size_t>(n_total) * 4;
    const Range rep{seg_reports, static_cast<size_t>(nseg) * 12};
    const Range others[] = {{p, b}, {m, b}, {v, b}, {options->amsgrad ? vmax : nullptr, b}};
    for (const Range &r : others)
        if (overlap(rep, r)) return FA_ERR_ALIAS;
    fa_report_mailbox *post = nullptr;
    uint32_t seq = 0;
    if (mailbox) {
        if ((st = mailbox_device_ptr(mailbox, &post)) != FA_OK) return st;
        seq = __atomic_load_n(&mailbox->seq, __ATOMIC_ACQUIRE) + 1;
    }
    if ((st = fa_analyze_gradient(g, gdt, n_total, row_len, seg_offsets, nseg, rows_buf,
                                  rows_capacity, stream)) != FA_OK)
        return st;
    if ((st = fa_merge_gradient_stats_chunks(rows_buf, chunk_rows.data(), nseg, scratch,
                                             scratch_elements, seg_reports, stream)) != FA_OK)
        return st;
    // The merges are done with the scratch once the reports are written: when it holds
    // nseg + 1 floats, every segment's decision is taken there once, and the update
    // runs on the full grid reading it.
    float *decided = scratch_elements >= static_cast<int64_t>(nseg) + 1 ? scratch : nullptr;
    if ((st = enqueue_segment_update(seg_offsets, nseg, p, g, gdt, m, v, vmax, t + 1, options,
                                     ctl, nullptr, seg_reports, max_grad_norm, stream, decided,
                                     post, seq)) != FA_OK)
        return st;
    if (!mailbox) return FA_OK;
    // the decision kernel posted the bucket's record before the update ran: wait for it
    // only, so that the caller can advance its count while the update runs
    fa_stats h{};
    return wait_for_post(mailbox, seq, static_cast<cudaStream_t>(stream), &h);
}

fa_status fa_read_report(const fa_stats *report_dev, fa_stats *report_host, void *stream) {
    TraceRange trace("fa_read_report");
    if (!report_host) return FA_ERR_NULL;
    int dev = 0;
    fa_status st = stream_device(stream, &dev);
    if (st != FA_OK) return st;
    if ((st = check_device_ptr(report_dev, dev, 4)) != FA_OK) return st;
    fa_stats tmp;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&tmp, report_dev, sizeof tmp, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    *report_host = tmp;
    return FA_OK;
}

fa_status fa_clip_decision(double sum_sq_stored, uint64_t nonfinite, double gradient_scale,
                           double max_grad_norm, int32_t *skip, double *grad_norm,
                           double *clip_coef) {
    if (!skip || !grad_norm || !clip_coef) return FA_ERR_NULL;
    if (!is_finite(gradient_scale) || gradient_scale <= 0) return FA_ERR_OPTION;
    if (std::isnan(max_grad_norm)) return FA_ERR_OPTION;
    const int32_t s = nonfinite > 0;
    const double norm = std::sqrt(sum_sq_stored) / gradient_scale;
    double coef = 1.0;
    if (!s && max_grad_norm > 0 && norm > max_grad_norm) coef = max_grad_norm / norm;
    *skip = s;
    *grad_norm = norm;
    *clip_coef = coef;
    return FA_OK;
}

fa_status fa_clip_decide(const fa_stats *report_dev, double gradient_scale, double max_grad_norm,
                         int32_t *skip, double *grad_norm, double *clip_coef, void *stream) {
    if (!skip || !grad_norm || !clip_coef) return FA_ERR_NULL;
    fa_stats h;
    fa_status st = fa_read_report(report_dev, &h, stream);
    if (st != FA_OK) return st;
    const double sum = fa::record_sum_sq(h);
    return fa_clip_decision(sum, h.nonfinite, gradient_scale, max_grad_norm, skip, grad_norm,
                            clip_coef);
}

fa_status fa_bucket_step_clipped(const int64_t *seg_offsets, int32_t nseg, int64_t n_total,
                                 float *p, const void *g, fa_dtype gdt, float *m, float *v,
                                 float *vmax, uint64_t *t, const fa_options *options,
                                 fa_step_control ctl, double max_grad_norm, int32_t row_len,
                                 fa_stats *rows_buf, int64_t rows_capacity, float *scratch,
                                 int64_t scratch_elements, fa_stats *report_dev,
                                 fa_step_report *out, void *stream) {
    TraceRange trace("fa_bucket_step_clipped");
    fa_status st;
    if (!t || !out) return FA_ERR_NULL;
    if ((st = check_step_args(options, ctl, gdt, n_total)) != FA_OK) return st;
    if (std::isnan(max_grad_norm)) return FA_ERR_OPTION;
    if ((st = check_segments(seg_offsets, nseg, n_total)) != FA_OK) return st;
    if (*t == UINT64_MAX) return FA_ERR_OPTION;
    fa_step_report rep{0, 0, 0, 0.0, 1.0};
    if (n_total == 0 || ctl.skip_update) {
        *out = rep;
        return FA_OK;
    }
    int dev = 0;
    if ((st = stream_device(stream, &dev)) != FA_OK) return st;
    if ((st = check_inplace(n_total, p, g, gdt, m, v, vmax, options, dev)) != FA_OK) return st;
    int64_t rows = 0;
    if ((st = fa_stats_rows(n_total, row_len, seg_offsets, nseg, &rows)) != FA_OK) return st;
    int32_t kernels = 0;
    int64_t need = 0;
    if ((st = fa_stats_plan(rows, &kernels, &need)) != FA_OK) return st;
    if (rows_capacity < rows || scratch_elements < need) return FA_ERR_SIZE;
    const size_t b = static_cast<size_t>(n_total) * 4;
    const Range r[] = {{p, b}, {g, static_cast<size_t>(n_total) * dtype_bytes(gdt)}, {m, b},
                       {v, b}, {options->amsgrad ? vmax : nullptr, b},
                       {rows_buf, static_cast<size_t>(rows) * 12},
                       {scratch, static_cast<size_t>(need) * 4}, {report_dev, 12}};
    if (any_overlap(r, 8)) return FA_ERR_ALIAS;

    if ((st = fa_analyze_gradient(g, gdt, n_total, row_len, seg_offsets, nseg, rows_buf,
                                  rows_capacity, stream)) != FA_OK)
        return st;
    if ((st = fa_merge_gradient_stats(rows_buf, rows, scratch, scratch_elements, report_dev,
                                      stream)) != FA_OK)
        return st;
    fa_stats h;
    if ((st = fa_read_report(report_dev, &h, stream)) != FA_OK) return st;
    int32_t skip = 0;
    double norm = 0, coef = 1;
    const double sum = fa::record_sum_sq(h);
    if ((st = fa_clip_decision(sum, h.nonfinite, ctl.gradient_scale, max_grad_norm, &skip, &norm,
                               &coef)) != FA_OK)
        return st;
    rep.nonfinite = h.nonfinite;
    rep.grad_norm = norm;
    rep.clip_coef = coef;
    if (skip) {
        rep.skipped_nonfinite = 1;
        *out = rep;
        return FA_OK;
    }
    st = enqueue_update(n_total, p, g, gdt, m, v, vmax, p, m, v, vmax, options, *t + 1,
                        ctl.gradient_scale, coef, stream);
    if (st != FA_OK) return st;
    *t += 1;
    rep.updated = 1;
    *out = rep;
    return FA_OK;
}

}  // extern "C"
