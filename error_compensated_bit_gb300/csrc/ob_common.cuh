// Device helpers shared by the compression-stage kernels (sm_103a).
//
// Work decomposition used by the streaming kernels here: the flat buffer is cut into
// groups of 256 elements (one warp iteration: 8 consecutive elements per lane, i.e. two
// 16-byte loads of float32 or one 16-byte load of a 16-bit gradient), and the groups
// into P contiguous ranges of (nearly) equal length, each worked by one warp (server) or
// by one block whose warps take its groups in turn (worker). A 256-element group never
// straddles a chunk (chunk % 256 == 0), so a warp can accumulate a chunk's sum of squares
// in registers and flush it when it moves to a later chunk.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ob_internal.h"

namespace ob {

constexpr unsigned kFull = 0xffffffffu;

// n / f.d for 32-bit n (see FastDiv).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f)
{
    if (f.d == 1) return n;
    const uint32_t t = __umulhi(n, f.m);
    return (t + ((n - t) >> 1)) >> (f.l - 1);
}

// ---- range partition ---------------------------------------------------------------------

__device__ __forceinline__ int64_t range_begin(const Part& pt, int64_t q)
{
    return q * pt.NG / pt.P;
}

// Ranges that hold at least one group of chunk k: lo..hi inclusive. Every range is
// non-empty (P <= NG), so this is exactly the set of warps that flush a partial for k.
__device__ __forceinline__ void chunk_contributors(const Part& pt, int64_t k, int64_t& lo,
                                                   int64_t& hi)
{
    const int64_t a = (k * pt.CG + 1) * pt.P;
    const int64_t b = (k + 1) * pt.CG * pt.P;
    lo = (a + pt.NG - 1) / pt.NG - 1;
    hi = (b + pt.NG - 1) / pt.NG - 1;
    if (hi > pt.P - 1) hi = pt.P - 1;
}

// ---- 8-element loads and stores ------------------------------------------------------------

__device__ __forceinline__ void ld8_stream(const float* p, float (&v)[8])
{
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// The same 8 floats cached in the L2 only (for data read again soon).
__device__ __forceinline__ void ld8_l2(const float* p, float (&v)[8])
{
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void st8_stream(float* p, const float (&v)[8])
{
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// Gradient rows in their storage format, widened exactly to float32.
template <typename G>
struct Grad;

template <>
struct Grad<float> {
    static __device__ __forceinline__ void ld8(const void* base, int64_t idx, float (&v)[8])
    {
        ld8_stream(static_cast<const float*>(base) + idx, v);
    }
};

template <>
struct Grad<__half> {
    static __device__ __forceinline__ void ld8(const void* base, int64_t idx, float (&v)[8])
    {
        const uint4 r = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __half*>(base) + idx));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            const float2 f = __half22float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
};

template <>
struct Grad<__nv_bfloat16> {
    static __device__ __forceinline__ void ld8(const void* base, int64_t idx, float (&v)[8])
    {
        const uint4 r = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + idx));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {               // bfloat16 is the top half of a float32
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// The same loads split in two: raw() issues the 16- or 32-byte load and keeps the bits as
// loaded (four registers for a 16-bit format), widen() converts them when they are used,
// so that a kernel with several groups in flight holds the narrow form meanwhile.
template <typename G>
struct GradRaw {
    uint4 r;
    static __device__ __forceinline__ GradRaw load(const void* base, int64_t idx)
    {
        return GradRaw{__ldcs(reinterpret_cast<const uint4*>(static_cast<const G*>(base) + idx))};
    }
    // the same load kept in the L2 (read again soon)
    static __device__ __forceinline__ GradRaw load_l2(const void* base, int64_t idx)
    {
        return GradRaw{__ldcg(reinterpret_cast<const uint4*>(static_cast<const G*>(base) + idx))};
    }
    __device__ __forceinline__ void widen(float (&v)[8]) const;
};

template <>
struct GradRaw<float> {
    float4 a, b;
    static __device__ __forceinline__ GradRaw load(const void* base, int64_t idx)
    {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
        return GradRaw{__ldcs(p), __ldcs(p + 1)};
    }
    static __device__ __forceinline__ GradRaw load_l2(const void* base, int64_t idx)
    {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
        return GradRaw{__ldcg(p), __ldcg(p + 1)};
    }
    __device__ __forceinline__ void widen(float (&v)[8]) const
    {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

template <>
__device__ __forceinline__ void GradRaw<__half>::widen(float (&v)[8]) const
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h;
        memcpy(&h, &w[i], 4);
        const float2 f = __half22float2(h);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void GradRaw<__nv_bfloat16>::widen(float (&v)[8]) const
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// ---- sign bits ---------------------------------------------------------------------------------

// Lane `lane` holds the sign bits of elements 8*lane .. 8*lane+7 of a group in `byte`.
// After the two exchanges, the four lanes of a quad hold the 32-bit word of elements
// 32*(lane/4) .. 32*(lane/4)+31 (bit t <-> element t of the word).
__device__ __forceinline__ uint32_t quad_word(uint32_t byte, int lane)
{
    uint32_t v = byte << (8 * (lane & 3));
    v |= __shfl_xor_sync(kFull, v, 1);
    v |= __shfl_xor_sync(kFull, v, 2);
    return v;
}

// The 8 sign bits of this lane's elements inside a row of packed words.
__device__ __forceinline__ uint32_t lane_byte(const uint32_t* words, int64_t group, int lane)
{
    const uint32_t w = __ldcs(words + group * 8 + (lane >> 2));
    return (w >> (8 * (lane & 3))) & 0xffu;
}

__device__ __forceinline__ float signed_scale(float s, bool nonneg)
{
    return nonneg ? s : -s;
}

// ---- reductions --------------------------------------------------------------------------------

// Error-free accumulation of squares in float32: every z^2 is split exactly into
// p + r (p = fl(z*z), r = fma(z, z, -p)) and p is added with Knuth's two-sum, whose
// rounding error q is exact; the pair (s, e) carries the sum as s + e with an error of
// order u^2 * terms * sum, which keeps chunk sums within ~1e-12 of an exact double sum.
struct Sum2 {
    float s, e;
};

__device__ __forceinline__ void sum2_add_sq(Sum2& a, float z)
{
    const float p = __fmul_rn(z, z);
    const float r = __fmaf_rn(z, z, -p);
    const float t = __fadd_rn(a.s, p);
    const float bp = __fsub_rn(t, a.s);
    const float ap = __fsub_rn(t, bp);
    const float q = __fadd_rn(__fsub_rn(a.s, ap), __fsub_rn(p, bp));
    a.s = t;
    a.e = __fadd_rn(a.e, __fadd_rn(q, r));
}

// (a.s + a.e) + (b.s + b.e) as a float pair: the sum of the leading parts split exactly
// by two-sum, the trailing parts added to its error. Symmetric in a and b bit for bit.
__device__ __forceinline__ Sum2 sum2_add(const Sum2& a, const Sum2& b)
{
    const float t = __fadd_rn(a.s, b.s);
    const float bp = __fsub_rn(t, a.s);
    const float ap = __fsub_rn(t, bp);
    const float q = __fadd_rn(__fsub_rn(a.s, ap), __fsub_rn(b.s, bp));
    return Sum2{t, __fadd_rn(__fadd_rn(a.e, b.e), q)};
}

__device__ __forceinline__ Sum2 shfl_xor(const Sum2& v, int o)
{
    return Sum2{__shfl_xor_sync(kFull, v.s, o), __shfl_xor_sync(kFull, v.e, o)};
}

// Warp totals of R rows of float-pair sums, by reduce-scatter: at each of the first
// log2(P2) exchange distances (16, 8, ...) a lane hands its partner half of its remaining
// rows and keeps the other half, so the rows spread over the lanes; a butterfly over the
// remaining distances then leaves every lane with the total of one row, `row` (rows R and
// above of the power-of-two padding are zeros). 2(P2 - 1 + 5 - log2 P2) shuffles instead
// of the 10 R of R separate butterflies; the order of the additions is fixed.
template <int R>
__device__ __forceinline__ Sum2 warp_reduce_rows(const Sum2 (&v)[R], int lane, int& row)
{
    constexpr int P2 = R <= 1 ? 1 : (R <= 2 ? 2 : (R <= 4 ? 4 : (R <= 8 ? 8 : 16)));
    Sum2 x[P2];
#pragma unroll
    for (int i = 0; i < P2; ++i) x[i] = i < R ? v[i] : Sum2{0.0f, 0.0f};
    int base = 0;
    int o = 16;
#pragma unroll
    for (int half = P2 / 2; half >= 1; half >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const Sum2 recv = shfl_xor(upper ? x[i] : x[i + half], o);
            x[i] = sum2_add(upper ? x[i + half] : x[i], recv);
        }
        if (upper) base += half;
    }
#pragma unroll
    for (; o >= 1; o >>= 1) x[0] = sum2_add(x[0], shfl_xor(x[0], o));
    row = base;
    return x[0];
}

// After warp_reduce_rows<R>: whether this lane is the one that stores its row's total
// (the lowest lane of each group of lanes left holding the same row).
template <int R>
__device__ __forceinline__ bool row_holder(int lane, int row)
{
    constexpr int P2 = R <= 1 ? 1 : (R <= 2 ? 2 : (R <= 4 ? 4 : (R <= 8 ? 8 : 16)));
    return (lane & (32 / P2 - 1)) == 0 && row < R;
}

// sqrt(sum / C) rounded to float32, from a sum of squares held as a float pair, in
// double-float arithmetic (T. J. Dekker, "A floating-point technique for extending the
// available precision", 1971): the quotient's exact remainder by FMA gives its trailing
// part, and one Newton correction from the square root's exact residual gives the root
// to about 2^-46 relative before the single final rounding -- the float32 nearest the
// exact root except within that distance of a rounding tie. C must be exactly
// representable (C <= 2^24). Returns false for a mean square outside [2^-80, 2^127] or a
// non-finite sum (degenerate chunks: the caller recomputes them in double).
__device__ __forceinline__ bool rms_from_pair(const Sum2& t, float Cf, float& out)
{
    const float hi = __fadd_rn(t.s, t.e);
    const float lo = __fsub_rn(t.e, __fsub_rn(hi, t.s));        // |t.s| >= |t.e|: exact
    if (!(hi >= __fmul_rn(Cf, 0x1p-80f) && hi <= 0x1p127f)) return false;
    const float qh = __fdiv_rn(hi, Cf);
    const float r = __fmaf_rn(-qh, Cf, hi);                      // hi - qh*C, exact
    const float ql = __fdiv_rn(__fadd_rn(r, lo), Cf);
    const float sh = __fsqrt_rn(qh);
    const float d = __fadd_rn(__fmaf_rn(-sh, sh, qh), ql);      // qh - sh^2 exact, then + ql
    const float sl = __fdiv_rn(d, __fadd_rn(sh, sh));
    out = __fadd_rn(sh, sl);
    return true;
}

// A chunk's scale from its double sum of squares: the sum split into a float pair (its
// float rounding and the float rounding of the remainder, which is exact in double) and
// the root taken by rms_from_pair in float arithmetic -- double division and square root
// are slow on this part, and this runs on the launch's critical path (the last
// contributor of each chunk). Sums outside rms_from_pair's range take the double root.
__device__ __forceinline__ float rms_from_double(double sum, int64_t C)
{
    const float hi = (float)sum;
    const float lo = (float)(sum - (double)hi);
    float sc;
    if (C <= (1 << 24) && rms_from_pair(Sum2{hi, lo}, (float)C, sc)) return sc;
    return (float)sqrt(sum / (double)C);
}

// Butterfly sum: every lane ends with the same, order-fixed value.
__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// A chunk's float32 sum of squares is trusted when its mean square lies in
// [2^-80, float max): squares of elements below 2^-63 (that underflow in float32) then
// weigh less than 2^-46 of the total. Otherwise -- an all-zero or all-tiny chunk, or an
// overflow -- the last contributor recomputes the chunk in double from the stored
// buffer (a slow path taken only by such degenerate chunks).
__device__ __forceinline__ bool sumsq_trusted(double sum, int64_t C)
{
    return sum >= (double)C * 0x1p-80 && sum <= 0x1p127;
}

static __device__ __noinline__ double chunk_sumsq_exact(const float* row, int64_t C, int lane)
{
    double acc = 0.0;
    for (int64_t i = (int64_t)lane * 4; i < C; i += 128) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(row + i));
        acc += (double)v.x * v.x;
        acc += (double)v.y * v.y;
        acc += (double)v.z * v.z;
        acc += (double)v.w * v.w;
    }
    return warp_sum(acc);
}

// ---- per-chunk scales from partial sums ------------------------------------------------------
//
// A range q is worked by `wpr` warps (warp `wir` of them here); each flushes one double
// partial per row -- possibly zero -- for every chunk the range touches, into slot
//   part[((r * P + q) * wpr + wir) * J + j],   j = k - (first chunk of range q).
// Chunk k is touched by ranges lo..hi: range lo holds the chunk's first group (its slot is
// j = k - first chunk of lo), and every later one starts inside chunk k (slot j = 0). No
// warp waits on another: the last arrival combines, writes the chunk's RMS scales and
// resets the chunk's counter for the next launch. `rows` is the buffer the squares came
// from (row r at rows + r*row_stride), read only on the degenerate slow path.

// The last contributor's combination: every row's partials added range by range, warp by
// warp (a lane's running sums add their terms in ascending range order; the 32 lanes' sums
// are then combined by a fixed butterfly), then scale = sqrt(sum / C). Loads of several
// ranges are issued before they are added; a missing term adds +0.0, which leaves a sum of
// squares unchanged, so the unrolling does not change the result. (Wider unrolling
// shortens this on small buffers, where its L2 round trips are a large part of the worker's
// time, but the larger out-of-line body made the calling kernels spill.)
template <int R>
__device__ __forceinline__ void combine_chunk(const Part& pt, int wpr, int64_t k, const double* part,
                                              unsigned* cnt, float* scale_out, int64_t C,
                                              const float* rows, int64_t row_stride, int lane)
{
    int64_t lo, hi;
    chunk_contributors(pt, k, lo, hi);
    const int64_t jlo = k - range_begin(pt, lo) / pt.CG;
    if (wpr == 1) {
        // lanes take the ranges in turn, all rows at once
        constexpr int U = R == 1 ? 4 : (R <= 4 ? 2 : 1);
        double acc_r[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc_r[r] = 0.0;
        for (int64_t q0 = lo + lane; q0 <= hi; q0 += 32 * U) {
            double v[U][R];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t qq = q0 + 32 * u;
                const int64_t off = qq * pt.J + (qq == lo ? jlo : 0);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    v[u][r] = qq <= hi ? __ldcg(part + (int64_t)r * pt.P * pt.J + off) : 0.0;
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < R; ++r) acc_r[r] += v[u][r];
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            double sum = warp_sum(acc_r[r]);
            if (!sumsq_trusted(sum, C)) sum = chunk_sumsq_exact(rows + (int64_t)r * row_stride + k * C, C, lane);
            if (lane == 0) scale_out[(int64_t)r * pt.nchunks + k] = rms_from_double(sum, C);
        }
    } else {
        // several warps per range: lane l owns the (row, warp) pairs l, l+32, ... and adds
        // that pair's partials range by range; per-row totals are then formed in a fixed order
        constexpr int kSlots = (R * 16 + 31) / 32;   // pairs per lane (wpr <= 16)
        constexpr int U = kSlots <= 2 ? 4 : 2;
        const int pairs = R * wpr;
        const int64_t range_stride = (int64_t)wpr * pt.J;
        double acc_p[kSlots];
        int row_of[kSlots];
        int64_t base_of[kSlots];
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
            const int pi = lane + 32 * i;
            acc_p[i] = 0.0;
            row_of[i] = pi < pairs ? pi / wpr : -1;
            base_of[i] = pi < pairs ? ((int64_t)(pi / wpr) * pt.P * wpr + pi % wpr) * pt.J : 0;
        }
        for (int64_t q0 = lo; q0 <= hi; q0 += U) {
            double v[U][kSlots];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t qq = q0 + u;
                const int64_t off = qq * range_stride + (qq == lo ? jlo : 0);
#pragma unroll
                for (int i = 0; i < kSlots; ++i)
                    v[u][i] = (qq <= hi && row_of[i] >= 0) ? __ldcg(part + base_of[i] + off) : 0.0;
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < kSlots; ++i) acc_p[i] += v[u][i];
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            double v = 0.0;
#pragma unroll
            for (int i = 0; i < kSlots; ++i)
                if (row_of[i] == r) v += acc_p[i];
            double sum = warp_sum(v);
            if (!sumsq_trusted(sum, C)) sum = chunk_sumsq_exact(rows + (int64_t)r * row_stride + k * C, C, lane);
            if (lane == 0) scale_out[(int64_t)r * pt.nchunks + k] = rms_from_double(sum, C);
        }
    }
    if (lane == 0) cnt[k] = 0u;
}

// Scales of a chunk whose only contributor is this warp, straight from the lanes' float
// pairs: no partial is stored and no double arithmetic runs (double throughput is low on
// this part, and with short chunks this runs once per group). The rows' totals are first
// spread over the lanes (warp_reduce_rows, inline: the sums are in registers); then each
// row's holder forms and stores its scale. Rows whose sum is degenerate (or chunks too
// long for a float32 C, which never lie inside one warp's range in practice) are
// recomputed in double from the stored buffer.
template <int R>
__device__ __forceinline__ void sole_scales(Sum2 t, int row, const Part& pt, int64_t k, float* scale_out,
                                            int64_t C, const float* rows, int64_t row_stride, int lane)
{
    const bool holder = row_holder<R>(lane, row);   // one lane per row
    float sc = 0.0f;
    const bool ok = C <= (1 << 24) && rms_from_pair(t, (float)C, sc);
    unsigned bad = __ballot_sync(kFull, holder && !ok);
    if (holder && ok) scale_out[(int64_t)row * pt.nchunks + k] = sc;
    if (bad) __threadfence();       // the chunk's rows were just stored by this warp's lanes
    while (bad) {
        const int l = __ffs(bad) - 1;
        bad &= bad - 1;
        const int r = __shfl_sync(kFull, row, l);
        const double ex = chunk_sumsq_exact(rows + (int64_t)r * row_stride + k * C, C, lane);
        if (lane == 0) scale_out[(int64_t)r * pt.nchunks + k] = (float)sqrt(ex / (double)C);
    }
}

template <int R>
__device__ __noinline__ void sole_scales_outlined(float ts, float te, int row, const Part& pt, int64_t k,
                                                  float* scale_out, int64_t C, const float* rows,
                                                  int64_t row_stride, int lane)
{
    sole_scales<R>(Sum2{ts, te}, row, pt, k, scale_out, C, rows, row_stride, lane);
}

// After the partials are stored: every contributor counts itself in, and the last one
// combines.
template <int R>
__device__ __forceinline__ void flush_rest(const Part& pt, int wpr, int64_t k, double* part, unsigned* cnt,
                                           float* scale_out, int64_t C, const float* rows, int64_t row_stride,
                                           int lane)
{
    __threadfence();                // every lane's stores (partials, rows) before ...
    __syncwarp();                   // ... lane 0 counts this contributor in
    unsigned last = 0;
    if (lane == 0) {
        int64_t lo, hi;
        chunk_contributors(pt, k, lo, hi);
        const unsigned prev = atomicAdd(cnt + k, 1u);
        last = (prev == (unsigned)((hi - lo + 1) * wpr - 1)) ? 1u : 0u;
    }
    last = __shfl_sync(kFull, last, 0);
    if (last) combine_chunk<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
}

// Out-of-line forms, so that a register-hungry kernel does not carry this code's
// registers through its streaming loop (it runs once per chunk and range).
template <int R>
__device__ __noinline__ void flush_rest_outlined(const Part& pt, int wpr, int64_t k, double* part, unsigned* cnt,
                                                 float* scale_out, int64_t C, const float* rows,
                                                 int64_t row_stride, int lane)
{
    flush_rest<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
}

template <int R>
__device__ __noinline__ void combine_chunk_outlined(const Part& pt, int wpr, int64_t k, const double* part,
                                                    unsigned* cnt, float* scale_out, int64_t C,
                                                    const float* rows, int64_t row_stride, int lane)
{
    combine_chunk<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
}

// How flush_chunk's rarely run part is laid out; the best choice depends on the calling
// kernel's register pressure (measured per kernel).
enum FlushCode {
    kFlushInline,       // everything inline
    kFlushTailCall,     // one call for everything after the partial stores (and one for
                        // an only contributor's scales)
    kFlushLastCall      // counter inline; a call only for the last contributor's combination
};

// Flush this warp's sums of squares of chunk k (rows 0..R-1): if the chunk lies wholly
// inside the warp's range, form its scales at once (sole_scales); otherwise store one
// double partial per row and finish the chunk if this warp is its last contributor. The
// warp works range q (groups g0..g1, first chunk kfirst) as warp wir of wpr. A caller
// whose ranges are shared by several warps passes MAYBE_SOLE = false, which leaves the
// first branch out of its code.
template <int R, FlushCode CODE, bool MAYBE_SOLE = true>
__device__ __forceinline__ void flush_chunk(const Part& pt, int64_t q, int wpr, int wir, int64_t k,
                                            int64_t kfirst, int64_t g0, int64_t g1, Sum2 (&acc)[R],
                                            double* part, unsigned* cnt, float* scale_out, int64_t C,
                                            const float* rows, int64_t row_stride, int lane)
{
    const int64_t idx0 = (q * wpr + wir) * pt.J + (k - kfirst);     // row 0's slot
    if (MAYBE_SOLE && wpr == 1 && k * pt.CG >= g0 && (k + 1) * pt.CG <= g1) {
        // the chunk lies wholly inside this warp's range: it is the only contributor
        int row;
        const Sum2 t = warp_reduce_rows<R>(acc, lane, row);
        if (CODE == kFlushTailCall) sole_scales_outlined<R>(t.s, t.e, row, pt, k, scale_out, C, rows, row_stride, lane);
        else sole_scales<R>(t, row, pt, k, scale_out, C, rows, row_stride, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            acc[r].s = 0.0f;
            acc[r].e = 0.0f;
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const double d = warp_sum((double)acc[r].s + (double)acc[r].e);
        if (lane == 0) part[idx0 + (int64_t)r * pt.P * wpr * pt.J] = d;
        acc[r].s = 0.0f;
        acc[r].e = 0.0f;
    }
    if (CODE == kFlushInline) {
        flush_rest<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
    } else if (CODE == kFlushTailCall) {
        flush_rest_outlined<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
    } else {
        __threadfence();
        __syncwarp();
        unsigned last = 0;
        if (lane == 0) {
            int64_t lo, hi;
            chunk_contributors(pt, k, lo, hi);
            const unsigned prev = atomicAdd(cnt + k, 1u);
            last = (prev == (unsigned)((hi - lo + 1) * wpr - 1)) ? 1u : 0u;
        }
        last = __shfl_sync(kFull, last, 0);
        if (last) combine_chunk_outlined<R>(pt, wpr, k, part, cnt, scale_out, C, rows, row_stride, lane);
    }
}

}  // namespace ob
