// Gradient statistics for sm_103a: per-row analysis and the fan-in-1024 merge.
//
// Follows RUDA "训练与状态保存" (zh/docs/training), section "在 ruda:0 上进行原生
// PyTorch 训练" (read-only gradient analysis; a 12-byte report read back before
// the update; any non-finite gradient skips the step; hierarchical statistics
// at fan-in 1024 change the reduction order only) and "実験的なデバイス上の融合
// AdamW / AMSGrad" (ja/docs/fused-adamw), section "ネイティブ PyTorch ストレージと
// 階層統計" (analyze_gradient, merge_gradient_stats, up to 4,194,304 rows).
//
// Record layout (12 bytes): {sum_sq: f32, nonfinite: u32, sum_sq_lo: f32}.
// A row's sum of squares is accumulated in FP32 (8 values per lane, then a
// warp shuffle tree) -- at 256 elements per row its relative error stays
// below 1e-6.  Merges add (hi, lo) pairs as double-float values with
// error-free FP32 transformations and hand each total to the next level as a
// (hi, lo) pair of floats, so later levels lose nothing.
//
// Finite values whose squares leave FP32's range: a row whose FP32 sum comes
// out non-finite while it holds no NaN or +-Inf is summed again with every
// value multiplied by 2^-96 (squares by 2^-192: a square of any FP32 value is
// then at most 2^64), and its record stores that sum negated.  A merge works in
// the scaled domain as soon as one of its inputs is scaled or a partial sum
// reaches 2^126 (below that two partial sums cannot overflow), and then
// multiplies unscaled inputs by 2^-192 as it takes them in; its output is
// negated in turn.  record_sum_sq (internal.h) decodes both forms.
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace fa {
namespace {

constexpr int kVec = 8;
constexpr int kRowsPerWarp = 4;  // rows a warp analyses concurrently

FA_BOUNDS_COUNTER(g_stats_oob)

// Widened value and whether the stored pattern is NaN or +-Inf (exponent all ones).
template <int GT>
struct StatIO;

template <>
struct StatIO<FA_F32> {
    static __device__ __forceinline__ void acc1(uint32_t b, float &s, uint32_t &c) {
        const bool bad = (b & 0x7f800000u) == 0x7f800000u;
        const float x = __uint_as_float(b);
        c += bad;
        s = bad ? s : fmaf(x, x, s);
    }
    static __device__ __forceinline__ void acc8(const void *g, int64_t i, float &s, uint32_t &c) {
        const uint4 *q = reinterpret_cast<const uint4 *>(static_cast<const float *>(g) + i);
        uint4 a = __ldcs(q);
        uint4 b = __ldcs(q + 1);
        acc1(a.x, s, c); acc1(a.y, s, c); acc1(a.z, s, c); acc1(a.w, s, c);
        acc1(b.x, s, c); acc1(b.y, s, c); acc1(b.z, s, c); acc1(b.w, s, c);
    }
    static __device__ __forceinline__ void accs(const void *g, int64_t i, float &s, uint32_t &c) {
        acc1(__ldcs(reinterpret_cast<const unsigned int *>(g) + i), s, c);
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        return __uint_as_float(__ldcs(reinterpret_cast<const unsigned int *>(g) + i));
    }
    static __device__ __forceinline__ void acc16(const uint4 &r, float &s, uint32_t &c) {
        acc1(r.x, s, c); acc1(r.y, s, c); acc1(r.z, s, c); acc1(r.w, s, c);
    }
};

template <>
struct StatIO<FA_BF16> {
    static __device__ __forceinline__ void acc1(uint32_t h, float &s, uint32_t &c) {
        const bool bad = (h & 0x7f80u) == 0x7f80u;
        const float x = __uint_as_float(h << 16);
        c += bad;
        s = bad ? s : fmaf(x, x, s);
    }
    static __device__ __forceinline__ void acc8(const void *g, int64_t i, float &s, uint32_t &c) {
        uint4 r = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + i));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc1(w[k] & 0xffffu, s, c);
            acc1(w[k] >> 16, s, c);
        }
    }
    static __device__ __forceinline__ void accs(const void *g, int64_t i, float &s, uint32_t &c) {
        acc1(__ldcs(static_cast<const unsigned short *>(g) + i), s, c);
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        return __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short *>(g) + i))
                               << 16);
    }
    static __device__ __forceinline__ void acc16(const uint4 &r, float &s, uint32_t &c) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc1(w[k] & 0xffffu, s, c);
            acc1(w[k] >> 16, s, c);
        }
    }
};

template <>
struct StatIO<FA_F16> {
    static __device__ __forceinline__ void acc1(uint32_t h, float &s, uint32_t &c) {
        const bool bad = (h & 0x7c00u) == 0x7c00u;
        const float x = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
        c += bad;
        s = bad ? s : fmaf(x, x, s);
    }
    static __device__ __forceinline__ void acc8(const void *g, int64_t i, float &s, uint32_t &c) {
        uint4 r = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + i));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc1(w[k] & 0xffffu, s, c);
            acc1(w[k] >> 16, s, c);
        }
    }
    static __device__ __forceinline__ void accs(const void *g, int64_t i, float &s, uint32_t &c) {
        acc1(__ldcs(static_cast<const unsigned short *>(g) + i), s, c);
    }
    static __device__ __forceinline__ float load1(const void *g, int64_t i) {
        return __half2float(__ushort_as_half(__ldcs(static_cast<const unsigned short *>(g) + i)));
    }
    static __device__ __forceinline__ void acc16(const uint4 &r, float &s, uint32_t &c) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc1(w[k] & 0xffffu, s, c);
            acc1(w[k] >> 16, s, c);
        }
    }
};

// Values of a rescued row are multiplied by 2^-96 before they are squared.
constexpr float kRescueScale = 0x1p-96f;
static_assert(kRescueValueExp == 96, "kRescueScale and record_sum_sq must agree");

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Segment holding launch-relative row r (binary search; warp-uniform).
__device__ __forceinline__ int find_segment(const AnalyzeArgs &a, int64_t r) {
    int lo = 0, hi = a.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.row_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Scaled sum of squares of elements [start, end) of one row, lane-strided and
// summed over the warp: values multiplied by 2^-96 before squaring (the
// rescue of a row whose FP32 sum overflowed without any NaN or +-Inf).  Every
// lane of the warp calls it; rare, so it simply reads the row again.
template <int GT>
__device__ __noinline__ float rescued_row_sum(const void *g, int64_t start, int64_t end, int64_t n,
                                              int lane) {
    float s = 0.f;
    for (int64_t i = start + lane; i < end; i += 32) {
        if (fa_in_bounds(i, 1, n)) {
            const float x = StatIO<GT>::load1(g, i) * kRescueScale;
            s = fmaf(x, x, s);
        }
    }
    return warp_sum(s);
}

// One warp per row, kRowsPerWarp rows in flight per warp.  Lane l reads
// elements [l*8, l*8+8) of each 256-element stretch of its rows.
template <int GT, bool VEC>
__global__ void __launch_bounds__(kThreads)
analyze_kernel(const __grid_constant__ AnalyzeArgs a) {
    fa_allow_dependents();  // the merge that follows waits for this grid to finish
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

    for (int64_t r0 = warp * kRowsPerWarp; r0 < a.rows; r0 += nwarps * kRowsPerWarp) {
        float s[kRowsPerWarp];
        uint32_t c[kRowsPerWarp];
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            s[j] = 0.f;
            c[j] = 0;
            const int64_t r = r0 + j;
            if (r < a.rows) {
                const int k = a.nseg == 1 ? 0 : find_segment(a, r);
                const int64_t start = a.seg_start[k] + (r - a.row_start[k]) * a.row_len;
                const int64_t seg_end = a.seg_start[k + 1];
                const int64_t end = start + a.row_len < seg_end ? start + a.row_len : seg_end;
                for (int64_t i = start + lane * kVec; i < end; i += 32 * kVec) {
                    if (VEC && i + kVec <= end) {
                        if (fa_in_bounds(i, kVec, a.n)) StatIO<GT>::acc8(a.g, i, s[j], c[j]);
                    } else {
                        const int64_t e = i + kVec < end ? i + kVec : end;
                        for (int64_t q = i; q < e; ++q)
                            if (fa_in_bounds(q, 1, a.n)) StatIO<GT>::accs(a.g, q, s[j], c[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            float tot = warp_sum(s[j]);
            const uint32_t cnt = __reduce_add_sync(0xffffffffu, c[j]);
            const int64_t r = r0 + j;
            if (!isfinite(tot) && cnt == 0 && r < a.rows) {  // (warp-uniform)
                const int k = a.nseg == 1 ? 0 : find_segment(a, r);
                const int64_t start = a.seg_start[k] + (r - a.row_start[k]) * a.row_len;
                const int64_t seg_end = a.seg_start[k + 1];
                const int64_t end = start + a.row_len < seg_end ? start + a.row_len : seg_end;
                tot = -rescued_row_sum<GT>(a.g, start, end, a.n, lane);
            }
            if (lane == j && r < a.rows && fa_in_bounds(r, 1, a.rows)) {
                fa_stats rec;
                rec.sum_sq = tot;
                rec.nonfinite = cnt;
                rec.sum_sq_lo = 0.f;
                a.out[r] = rec;
            }
        }
    }
}

// Squares of one 16-byte word, added unconditionally (no finiteness test);
// RESCUE: each value multiplied by 2^-96 first.
template <int GT, bool RESCUE = false>
__device__ __forceinline__ void sq16(const uint4 &r, float &s) {
    const float k = RESCUE ? kRescueScale : 1.0f;
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (GT == FA_F32) {
            const float x = RESCUE ? __uint_as_float(w[q]) * k : __uint_as_float(w[q]);
            s = fmaf(x, x, s);
        } else if (GT == FA_BF16) {
            float lo = __uint_as_float(w[q] << 16);
            float hi = __uint_as_float(w[q] & 0xffff0000u);
            if (RESCUE) {
                lo *= k;
                hi *= k;
            }
            s = fmaf(lo, lo, s);
            s = fmaf(hi, hi, s);
        } else {
            float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[q]));
            if (RESCUE) {
                f.x *= k;
                f.y *= k;
            }
            s = fmaf(f.x, f.x, s);
            s = fmaf(f.y, f.y, s);
        }
    }
}

// Exact count of NaN / +-Inf patterns in one 16-byte word.
template <int GT>
__device__ __forceinline__ uint32_t count_nonfinite16(const uint4 &r) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (GT == FA_F32) {
            c += (w[k] & 0x7f800000u) == 0x7f800000u;
        } else {
            const uint32_t e = GT == FA_BF16 ? 0x7f80u : 0x7c00u;
            c += (w[k] & e) == e;
            c += ((w[k] >> 16) & e) == e;
        }
    }
    return c;
}

// Sums R rows' per-lane partials across the warp in one transposed butterfly:
// at each of the first log2(R) levels a lane keeps half of its rows and
// trades the other half with its partner, so R rows cost R-1 shuffles plus
// the 5-log2(R) of a single butterfly.  Returns the total of row
// (lane >> (5 - log2 R)) & (R - 1), which every lane of that group holds.
template <int R>
__device__ __forceinline__ float transpose_reduce(const float (&s)[R], int lane) {
    float cur[R];
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i] = s[i];
    int off = 16;
#pragma unroll
    for (int h = R / 2; h >= 1; h >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? cur[i] : cur[i + h];
            const float keep = upper ? cur[i + h] : cur[i];
            cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        off >>= 1;
    }
#pragma unroll
    for (; off >= 1; off >>= 1) cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], off);
    return cur[0];
}

// Fast path: every row start 16-byte aligned and a full row exactly CH
// 512-byte warp chunks (so the row length is a compile-time constant).  A
// warp takes R = 8/CH consecutive rows per iteration and issues all their
// 16-byte loads (8 per lane, 4 KB per warp) before any arithmetic; in a
// single-segment buffer the rows of an iteration share one base address.
// Squares are summed without a finiteness test: a row's FP32 sum of
// non-negative terms is finite exactly when none of its values is NaN or
// +-Inf (unless a finite value's square overflows FP32), so the exact
// bit-pattern count runs only for rows whose sum came out non-finite, from
// the words still held in registers.  Short rows at a segment's end take a
// checked scalar loop.
template <int GT, int CH, bool MULTI, int THREADS>
__global__ void __launch_bounds__(THREADS)
analyze_fast_kernel(const __grid_constant__ AnalyzeArgs a) {
    fa_allow_dependents();  // the merge that follows waits for this grid to finish
    constexpr int R = 8 / CH;
    constexpr int kLog2R = R == 8 ? 3 : R == 4 ? 2 : R == 2 ? 1 : 0;
    constexpr int64_t kElemBytes = GT == FA_F32 ? 4 : 2;
    constexpr int64_t kRowElems = 512 * CH / kElemBytes;
    const int lane = threadIdx.x & 31;
    const int my_row = (lane >> (5 - kLog2R)) & (R - 1);
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
    const char *gb = static_cast<const char *>(a.g);
    const int64_t single_full_rows = MULTI ? 0 : (a.seg_start[1] - a.seg_start[0]) / kRowElems;

    for (int64_t r0 = warp * R; r0 < a.rows; r0 += nwarps * R) {
        uint32_t full = 0, valid = 0;
        uint4 buf[R][CH];
        if (!MULTI && r0 + R <= single_full_rows &&
            fa_in_bounds(a.seg_start[0] + r0 * kRowElems, R * kRowElems, a.n)) {
            const uint4 *q = reinterpret_cast<const uint4 *>(
                                 gb + (a.seg_start[0] + r0 * kRowElems) * kElemBytes) + lane;
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) buf[j][ch] = __ldcs(q + (j * CH + ch) * 32);
            full = valid = (1u << R) - 1;
        } else {
            int k = MULTI ? find_segment(a, r0) : 0;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int64_t r = r0 + j;
                if (r < a.rows) {
                    valid |= 1u << j;
                    if (MULTI)
                        while (k + 1 < a.nseg && a.row_start[k + 1] <= r) ++k;
                    const int64_t start = a.seg_start[k] + (r - a.row_start[k]) * kRowElems;
                    if (start + kRowElems <= a.seg_start[k + 1] &&
                        fa_in_bounds(start, kRowElems, a.n)) {
                        full |= 1u << j;
                        const uint4 *q =
                            reinterpret_cast<const uint4 *>(gb + start * kElemBytes) + lane;
#pragma unroll
                        for (int ch = 0; ch < CH; ++ch) buf[j][ch] = __ldcs(q + ch * 32);
                    }
                }
            }
        }
        float s[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            s[j] = 0.f;
            if (full & (1u << j)) {
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) sq16<GT>(buf[j][ch], s[j]);
            }
        }
        float tot = transpose_reduce<R>(s, lane);
        uint32_t cnt = 0;

        // rows whose FP32 sum is non-finite: exact count from the registers
        const unsigned bad = __ballot_sync(0xffffffffu, ((full >> my_row) & 1u) && !isfinite(tot));
        if (bad) {
#pragma unroll
            for (int j = 0; j < R; ++j) {
                if (bad & (1u << (j << (5 - kLog2R)))) {
                    uint32_t c = 0;
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) c += count_nonfinite16<GT>(buf[j][ch]);
                    c = __reduce_add_sync(0xffffffffu, c);
                    if (my_row == j) cnt = c;
                    if (c == 0) {  // finite values whose squares overflowed: rescue
                        float sr = 0.f;
#pragma unroll
                        for (int ch = 0; ch < CH; ++ch) sq16<GT, true>(buf[j][ch], sr);
                        sr = warp_sum(sr);
                        if (my_row == j) tot = -sr;
                    }
                }
            }
        }
        // short rows at a segment's end: checked scalar loop
        const uint32_t partial = valid & ~full;
        if (partial) {
            for (int j = 0; j < R; ++j) {
                if (!(partial & (1u << j))) continue;
                const int64_t r = r0 + j;
                const int ks = MULTI ? find_segment(a, r) : 0;
                const int64_t start = a.seg_start[ks] + (r - a.row_start[ks]) * kRowElems;
                const int64_t end = a.seg_start[ks + 1];
                float sj = 0.f;
                uint32_t c = 0;
                for (int64_t i = start + lane; i < end; i += 32)
                    if (fa_in_bounds(i, 1, a.n)) StatIO<GT>::accs(a.g, i, sj, c);
                sj = warp_sum(sj);
                c = __reduce_add_sync(0xffffffffu, c);
                if (!isfinite(sj) && c == 0)  // (warp-uniform) rescue
                    sj = -rescued_row_sum<GT>(a.g, start, end, a.n, lane);
                if (my_row == j) {
                    tot = sj;
                    cnt = c;
                }
            }
        }
        if ((lane & ((32 >> kLog2R) - 1)) == 0 && ((valid >> my_row) & 1u) &&
            fa_in_bounds(r0 + my_row, 1, a.rows)) {
            fa_stats rec;
            rec.sum_sq = tot;
            rec.nonfinite = cnt;
            rec.sum_sq_lo = 0.f;
            a.out[r0 + my_row] = rec;
        }
    }
}

// Error-free addition (Knuth's TwoSum): s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Adds (bh, bl) into the double-float (h, l).
__device__ __forceinline__ void df_add(float &h, float &l, float bh, float bl) {
    float s, e;
    two_sum(h, bh, s, e);
    e += l + bl;
    two_sum(s, e, h, l);
}

// Partial sums at or above this switch a merge to the scaled domain: two
// unscaled partial sums below it add up to less than 2^127, which cannot overflow.
constexpr float kScaleSwitch = 0x1p126f;

// Multiplies a double-float by 2^-192 (two exact power-of-two steps; only values
// that fall below FP32's normal range lose bits, and those are negligible next
// to the sum that caused the switch, which is at least 2^-66 after scaling).
__device__ __forceinline__ void df_scale_down(float &h, float &l) {
    h = h * kRescueScale * kRescueScale;
    l = l * kRescueScale * kRescueScale;
}

// Adds (bh, bl) -- scaled when bs -- into the double-float (h, l) -- scaled when
// *hs -- moving the accumulator to the scaled domain first when either side is
// scaled or either partial sum has reached kScaleSwitch.
__device__ __forceinline__ void df_add_domain(float &h, float &l, bool &hs, float bh, float bl,
                                              bool bs) {
    const bool scaled = hs || bs || h >= kScaleSwitch || bh >= kScaleSwitch;
    if (scaled && !hs) df_scale_down(h, l);
    if (scaled && !bs) df_scale_down(bh, bl);
    hs = scaled;
    df_add(h, l, bh, bl);
}

// Lane sums below this let a warp's 32-lane shuffle tree stay below kScaleSwitch.
constexpr float kWarpTreeLimit = 0x1p121f;

// Adds records [lo + lane, hi) with stride 32 into (sh, sl): plain records with plain
// double-float additions, marking in *special any record that is scaled, at or above
// kScaleSwitch, or NaN; or (DOMAIN) with the domain-aware addition, tracking *ss.
template <bool DOMAIN>
__device__ __forceinline__ void lane_merge(const fa_stats *__restrict__ in, int64_t lo, int64_t hi,
                                           int lane, float &sh, float &sl, bool &ss,
                                           bool &special, unsigned long long &c) {
    constexpr int kBatch = DOMAIN ? 4 : 16;  // (the rare path: fewer registers)
    for (int64_t base = lo + lane; base < hi; base += 32 * kBatch) {
        fa_stats r[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * 32;
            if (i < hi) r[u] = in[i];
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * 32;
            if (i < hi) {
                if (DOMAIN) {
                    const bool rs = r[u].sum_sq < 0.f;
                    df_add_domain(sh, sl, ss, rs ? -r[u].sum_sq : r[u].sum_sq,
                                  rs ? -r[u].sum_sq_lo : r[u].sum_sq_lo, rs);
                } else {
                    special |= !(r[u].sum_sq >= 0.f && r[u].sum_sq < kScaleSwitch);
                    df_add(sh, sl, r[u].sum_sq, r[u].sum_sq_lo);
                    c += r[u].nonfinite;
                }
            }
        }
    }
}

// One warp reduces records [lo, hi) into *out.  Lane l adds records l, l + 32, ...
// as double-float values (an FP32 value and its FP32 residual, combined with
// error-free TwoSum, so every operation stays on the FP32 units: GB300's FP64
// rate made an FP64 first level compute-bound), 16 records' loads issued
// together; then the warp's shuffle tree, and lane 0 writes the total as an FP32
// (hi, lo) pair.  When a lane met a scaled record, a record at or above
// kScaleSwitch or a NaN, or holds a sum that could overflow the tree, the warp
// adds its records again with the domain-aware addition (rare: it needs a finite
// value above about 1.8e19 in the gradient), and the total is negated when it is
// in the scaled domain.  Every lane of the warp calls it.
__device__ __forceinline__ void warp_merge(const fa_stats *__restrict__ in, int64_t lo, int64_t hi,
                                           int64_t in_count, fa_stats *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    if (!fa_in_bounds(lo, hi - lo, in_count)) hi = lo;  // (bounds-checked build only)
    float sh = 0.f, sl = 0.f;
    bool ss = false;       // (sh, sl) in the scaled domain
    bool special = false;  // this lane's records need the domain-aware addition
    unsigned long long c = 0;
    lane_merge<false>(in, lo, hi, lane, sh, sl, ss, special, c);
    if (__any_sync(0xffffffffu, special || !(sh < kWarpTreeLimit))) {
        sh = sl = 0.f;
        lane_merge<true>(in, lo, hi, lane, sh, sl, ss, special, c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, sh, o);
            const float ol = __shfl_xor_sync(0xffffffffu, sl, o);
            const bool os = __shfl_xor_sync(0xffffffffu, static_cast<int>(ss), o) != 0;
            df_add_domain(sh, sl, ss, oh, ol, os);
        }
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, sh, o);
            const float ol = __shfl_xor_sync(0xffffffffu, sl, o);
            df_add(sh, sl, oh, ol);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) {
        const double ts = static_cast<double>(sh) + static_cast<double>(sl);
        fa_stats rec;
        rec.sum_sq = static_cast<float>(ts);
        rec.sum_sq_lo = static_cast<float>(ts - static_cast<double>(rec.sum_sq));
        if (ss) {
            rec.sum_sq = -rec.sum_sq;
            rec.sum_sq_lo = -rec.sum_sq_lo;
        }
        rec.nonfinite = c > 0xffffffffull ? 0xffffffffu : static_cast<uint32_t>(c);
        *out = rec;
    }
}

constexpr int kMergeWarps = kThreads / 32;  // groups (or chunks) per CTA

// One warp per group of kFanIn input records, eight groups per CTA: the 4096
// groups of the largest plan take 512 CTAs instead of 4096.
// ``post`` (the final level only; nullptr otherwise) is the device address of a
// report mailbox in pinned host memory: the report is also stored there, then, after
// a system-wide fence, ``seq``, so a host that sees seq reads the whole report.
__global__ void __launch_bounds__(kThreads)
merge_kernel(const fa_stats *__restrict__ in, int64_t count, fa_stats *__restrict__ out,
             fa_report_mailbox *post, uint32_t seq) {
    fa_grid_dependency_wait();  // (launched early: the records are not ready before this)
    fa_allow_dependents();
    const int64_t group = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    const int64_t lo = group * kFanIn;
    if (lo >= count) return;  // the whole warp
    const int64_t hi = lo + kFanIn < count ? lo + kFanIn : count;
    warp_merge(in, lo, hi, count, out + group);
    if (post != nullptr && group == 0 && (threadIdx.x & 31) == 0) {
        const fa_stats rec = out[0];  // written by this thread just above
        volatile uint32_t *w = reinterpret_cast<volatile uint32_t *>(&post->report);
        w[0] = __float_as_uint(rec.sum_sq);
        w[1] = rec.nonfinite;
        w[2] = __float_as_uint(rec.sum_sq_lo);
        __threadfence_system();
        *reinterpret_cast<volatile uint32_t *>(&post->seq) = seq;
    }
}

// Per-chunk merge, level A: one CTA per group of at most kFanIn records of one
// chunk (groups never span two chunks).
__device__ __forceinline__ int find_chunk(const ChunkMergeArgs &a, int64_t group) {
    int lo = 0, hi = a.nchunks - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.group_start[mid] <= group) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kThreads)
merge_chunks_a_kernel(const __grid_constant__ ChunkMergeArgs a) {
    fa_grid_dependency_wait();
    fa_allow_dependents();
    const int64_t b = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (b >= a.group_start[a.nchunks]) return;  // the whole warp
    const int k = find_chunk(a, b);
    const int64_t lo = a.row_start[k] + (b - a.group_start[k]) * kFanIn;
    const int64_t hi = lo + kFanIn < a.row_start[k + 1] ? lo + kFanIn : a.row_start[k + 1];
    warp_merge(a.in, lo, hi, a.row_start[a.nchunks], a.partial + b);
}

// Level B: one warp per chunk over its level-A records (an empty chunk gives a
// zero record).
__global__ void __launch_bounds__(kThreads)
merge_chunks_b_kernel(const __grid_constant__ ChunkMergeArgs a) {
    fa_grid_dependency_wait();
    fa_allow_dependents();
    const int k = static_cast<int>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (k >= a.nchunks) return;  // the whole warp
    warp_merge(a.partial, a.group_start[k], a.group_start[k + 1], a.group_start[a.nchunks],
               a.out + k);
}

// A single-segment buffer takes a full grid of 128-thread CTAs, each warp one
// iteration of R rows: on GB300 that read the 2.15 GB BF16 gradient of 1.07e9
// parameters in 0.316 ms against 0.338 ms for persistent 256-thread CTAs (CUDA
// events, bit-identical rows).  A segment table keeps the persistent grid, which
// measured as fast or faster there (0.419 against 0.417-0.435 ms for the 199-segment
// FP16 bucket of 1.2e9 parameters).
constexpr int kFastFullThreads = 128;

template <int GT, int CH, bool MULTI>
cudaError_t launch_fast(const AnalyzeArgs &a, int64_t need, int dev, cudaStream_t stream) {
    if constexpr (MULTI) {
        auto k = analyze_fast_kernel<GT, CH, MULTI, kThreads>;
        k<<<persistent_grid(k, need, dev), kThreads, 0, stream>>>(a);
        return cudaGetLastError();
    } else {
        (void)need;
        (void)dev;
        constexpr int64_t kRowsPerCta = (8 / CH) * (kFastFullThreads / 32);
        const int64_t ctas = (a.rows + kRowsPerCta - 1) / kRowsPerCta;
        auto k = analyze_fast_kernel<GT, CH, MULTI, kFastFullThreads>;
        const int grid = static_cast<int>(ctas < kMaxGridX ? ctas : kMaxGridX);
        if (grid == 0) return cudaSuccess;
        k<<<grid, kFastFullThreads, 0, stream>>>(a);
        return cudaGetLastError();
    }
}

template <int GT>
cudaError_t launch_analyze_typed(const AnalyzeArgs &a, bool vec, cudaStream_t stream) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (sm_count(dev) <= 0) return cudaErrorInvalidDevice;
    const int64_t row_bytes = a.row_len * (GT == FA_F32 ? 4 : 2);
    const int64_t ch = row_bytes % 512 == 0 ? row_bytes / 512 : 0;
    auto ctas_for = [&](int64_t rows_per_warp) {
        return (((a.rows + rows_per_warp - 1) / rows_per_warp) * 32 + kThreads - 1) / kThreads;
    };
    if (vec && (ch == 1 || ch == 2 || ch == 4 || ch == 8)) {
        const int64_t need = ctas_for(8 / ch);
        if (a.nseg == 1) {
            switch (ch) {
                case 1: return launch_fast<GT, 1, false>(a, need, dev, stream);
                case 2: return launch_fast<GT, 2, false>(a, need, dev, stream);
                case 4: return launch_fast<GT, 4, false>(a, need, dev, stream);
                default: return launch_fast<GT, 8, false>(a, need, dev, stream);
            }
        }
        switch (ch) {
            case 1: return launch_fast<GT, 1, true>(a, need, dev, stream);
            case 2: return launch_fast<GT, 2, true>(a, need, dev, stream);
            case 4: return launch_fast<GT, 4, true>(a, need, dev, stream);
            default: return launch_fast<GT, 8, true>(a, need, dev, stream);
        }
    } else if (vec) {
        auto k = analyze_kernel<GT, true>;
        k<<<persistent_grid(k, ctas_for(kRowsPerWarp), dev), kThreads, 0, stream>>>(a);
    } else {
        auto k = analyze_kernel<GT, false>;
        k<<<persistent_grid(k, ctas_for(kRowsPerWarp), dev), kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_analyze(const AnalyzeArgs &a, fa_dtype gdt, bool vector_ok,
                           cudaStream_t stream) {
    switch (gdt) {
        case FA_F32: return launch_analyze_typed<FA_F32>(a, vector_ok, stream);
        case FA_F16: return launch_analyze_typed<FA_F16>(a, vector_ok, stream);
        case FA_BF16: return launch_analyze_typed<FA_BF16>(a, vector_ok, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t stats_bounds_violations(unsigned long long *count, bool clear) {
#if FA_BOUNDS_CHECK
    cudaError_t err = cudaMemcpyFromSymbol(count, g_stats_oob, sizeof(*count));
    if (err != cudaSuccess || !clear) return err;
    const unsigned long long zero = 0;
    return cudaMemcpyToSymbol(g_stats_oob, &zero, sizeof(zero));
#else
    (void)clear;
    *count = 0;
    return cudaSuccess;
#endif
}

cudaError_t launch_merge_chunks(const ChunkMergeArgs &a, cudaStream_t stream) {
    const int64_t groups = a.group_start[a.nchunks];
    // both levels start early and wait for their input in the kernel
    if (groups > 0) {
        const cudaError_t err = launch_dependent(
            merge_chunks_a_kernel, dim3(static_cast<unsigned>((groups + kMergeWarps - 1) / kMergeWarps)),
            dim3(kThreads), 0, stream, a);
        if (err != cudaSuccess) return err;
    }
    if (a.nchunks > 0)
        return launch_dependent(merge_chunks_b_kernel,
                                dim3(static_cast<unsigned>((a.nchunks + kMergeWarps - 1) / kMergeWarps)),
                                dim3(kThreads), 0, stream, a);
    return cudaSuccess;
}

cudaError_t launch_merge(const fa_stats *in, int64_t count, fa_stats *out, cudaStream_t stream,
                         fa_report_mailbox *post, uint32_t seq) {
    const int64_t groups = (count + kFanIn - 1) / kFanIn;
    const int64_t grid = (groups + kMergeWarps - 1) / kMergeWarps;
    if (grid <= 0) return cudaSuccess;
    if (post != nullptr && groups != 1) return cudaErrorInvalidValue;  // final level only
    // starts early and waits for its input in the kernel
    return launch_dependent(merge_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                            stream, in, count, out, post, seq);
}

// ---- fixed merge scratch for callers that cannot allocate ------------------------
//
// One file-scope device array, large enough for the biggest reduction plan
// (4,194,304 rows -> 4096 + 4 intermediate 12-byte records = 12,300 floats,
// 49,200 bytes).  Every GPU that loads this library holds it until the
// process exits.  In host code the symbol is only a stand-in: its device
// address comes from cudaGetSymbolAddress, looked up once per device.

static __device__ __align__(256) float g_static_merge_scratch[kStaticMergeScratchFloats];

cudaError_t static_merge_scratch(int device, bool lookup_allowed, float **ptr,
                                 int64_t *capacity_floats) {
    static std::mutex mu;
    static float *addr[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        // the first lookup may load the module; it must not happen inside a capture
        if (!lookup_allowed) return cudaErrorStreamCaptureUnsupported;
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_static_merge_scratch);
        if (err != cudaSuccess) return err;
        addr[device] = static_cast<float *>(p);
    }
    *ptr = addr[device];
    *capacity_floats = kStaticMergeScratchFloats;
    return cudaSuccess;
}

}  // namespace fa
