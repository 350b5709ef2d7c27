// LoCo low-bit step: each worker compensates its gradient with the moving average of
// its past compression errors, quantizes it per chunk to signed `bits`-bit levels with
// an absmax scale, and updates the moving average; the mean of the dequantized
// gradients then drives a plain Adam step.
//
// Method: "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// "Method" (moving average of historical compensation errors, compensate before
// compression, then synchronise), key design item 2 (the proportion of the compensation
// is tuned: `ratio`, 1 by default) and the abstract (compatible with Adam).
//
// Passes. The absmax of c = g + ratio*e~ over a chunk must be known before any element of
// the chunk can be quantized, and a chunk spans up to n/W elements, so for long chunks c
// is formed twice (once for the absmax, once to quantize) instead of being stored:
//   absmax     amax[w][k] = max |c|                      (atomicMax on float bits: exact)
//   quantize   s = amax/L; q = clamp(rint(c/s), -L, L) (0 when s = 0); e = c - q*s;
//              e~ = beta*e~ + (1-beta)*e
//   server     gbar = (sum over w of q_w*s_w)/W; Adam on m, v, x
// Long chunks: the absmax pass (W*(grad+4) bytes per element), then quantize and server
// in one pass over all W rows of each group (k_loco_qs: W*(grad+8) + 24; the codes stay
// in registers). Chunks of up to 4096 elements: absmax and quantize in one kernel whose
// warps own whole chunks (k_loco_fused_small, k_loco_fused: W*(grad+8+bits/8), reading
// the gradients and errors from DRAM once), then the server pass (k_loco_server:
// W*bits/8 + 24).
#include "ob_common.cuh"
#include "ob_div.cuh"
#include "ob_tma.cuh"

namespace ob {

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Work items are the W*n/256 groups of 256 elements of the [W][n] rows, numbered in
// memory order (item t starts at element t*256 of the flat array; n is a multiple of the
// chunk, so item t lies in scale slot t / (chunk/256) = w*nchunks + k). Each warp owns one
// contiguous, balanced range of items (the grid is one resident wave) and keeps kLocoU
// groups' loads in flight per iteration.
constexpr int kLocoU = 4;

__device__ __forceinline__ void warp_items(int64_t total, int64_t& t0, int64_t& t1)
{
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    t0 = warp * total / nwarps;
    t1 = (warp + 1) * total / nwarps;
}

template <typename G>
__global__ void __launch_bounds__(kBlock) k_loco_absmax(LocoArgs a)
{
    constexpr int U = kLocoU;
    const int lane = threadIdx.x & 31;
    int64_t t0, t1;
    warp_items((int64_t)a.W * a.NG, t0, t1);
    // the running max of the scale slot the warp is in, published (atomicMax on the float
    // bits, exact and order-free) only when the slot changes
    int64_t cur = t0 < t1 ? (int64_t)fast_div((uint32_t)t0, a.cg_div) : -1;
    float run = 0.0f;
    for (int64_t tb = t0; tb < t1; tb += U) {
        GradRaw<G> gr[U];
        float ev[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u < t1) {
                const int64_t e0 = (tb + u) * 256 + lane * 8;
                gr[u] = GradRaw<G>::load(a.g, e0);
                ld8_stream(a.err + e0, ev[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u < t1) {
                const int64_t key = fast_div((uint32_t)(tb + u), a.cg_div);
                if (key != cur) {
                    const float mx = warp_max(run);
                    if (lane == 0) atomicMax(a.amax_bits + cur, __float_as_uint(mx));
                    cur = key;
                    run = 0.0f;
                }
                float gv[8];
                gr[u].widen(gv);
#pragma unroll
                for (int j = 0; j < 8; ++j) run = fmaxf(run, fabsf(__fadd_rn(gv[j], __fmul_rn(a.ratio, ev[u][j]))));
            }
        }
    }
    if (cur >= 0) {
        const float mx = warp_max(run);
        if (lane == 0) atomicMax(a.amax_bits + cur, __float_as_uint(mx));
    }
}

// Quantize one lane's 8 elements of a group with scale s (inv = rn(1/s)) and update the
// moving average of the errors in place; returns the levels.
template <int BITS>
__device__ __forceinline__ void quantize8_levels(const float (&gv)[8], float (&ev)[8], float s, float inv,
                                                 float ratio, float beta, float keep, int (&qv)[8])
{
    const float L = (float)((1 << (BITS - 1)) - 1);
    constexpr float kTieMargin = (float)(1 << (BITS - 1)) * 0x1p-21f;   // (L + 1) 2^-21
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float c = __fadd_rn(gv[j], __fmul_rn(ratio, ev[j]));
        int qi = 0;
        if (s > 0.0f) {
            // rint(c/s) with c/s correctly rounded, as defined. |c/s| <= L(1+u), and
            // c * rn(1/s) lies within 3u|c/s| < (L+1) 2^-22 of rn(c/s); unless it is that
            // close to a half-integer, both round to the same integer. Near a half-integer
            // (the test keeps twice that distance) or when 1/s overflows, the quotient is
            // formed exactly.
            const float qq = __fmul_rn(c, inv);
            float r = rintf(qq);
            if (!(fabsf(__fsub_rn(qq, r)) < 0.5f - kTieMargin)) r = rintf(__fdiv_rn(c, s));
            r = fminf(fmaxf(r, -L), L);
            qi = (int)r;
        }
        qv[j] = qi;
        const float e = __fsub_rn(c, __fmul_rn((float)qi, s));
        ev[j] = __fadd_rn(__fmul_rn(beta, ev[j]), __fmul_rn(keep, e));
    }
}

// The levels packed as stored: 4 bits two per byte (even element in the low nibble) or
// one signed byte each, two's complement.
template <int BITS>
__device__ __forceinline__ void pack_codes(const int (&qv)[8], uint32_t& lo, uint32_t& hi)
{
    lo = 0;
    hi = 0;
    if (BITS == 4) {
#pragma unroll
        for (int j = 0; j < 8; ++j) lo |= ((uint32_t)qv[j] & 0xfu) << (4 * j);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo |= ((uint32_t)qv[j] & 0xffu) << (8 * j);
            hi |= ((uint32_t)qv[j + 4] & 0xffu) << (8 * j);
        }
    }
}

template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t* out, uint32_t lo, uint32_t hi)
{
    if (BITS == 4) __stcs(reinterpret_cast<unsigned int*>(out), lo);
    else __stcs(reinterpret_cast<uint2*>(out), make_uint2(lo, hi));
}

// quantize8_levels, then the levels packed as stored.
template <int BITS>
__device__ __forceinline__ void quantize8(const float (&gv)[8], float (&ev)[8], float s, float inv,
                                          float ratio, float beta, float keep, uint32_t& lo, uint32_t& hi)
{
    int qv[8];
    quantize8_levels<BITS>(gv, ev, s, inv, ratio, beta, keep, qv);
    pack_codes<BITS>(qv, lo, hi);
}

// Absmax and quantization in one kernel, for chunks short enough that a warp owns whole
// ones: the (row, chunk) slots -- slot w*nchunks + k covers elements [slot*C, (slot+1)*C)
// of the flat [W][n] arrays -- are split into contiguous ranges per warp. Each slot is
// read twice, first for its absmax (kept in the L2, as the slots the warps hold in flight
// together stay well inside it) and straight after to quantize, so DRAM sees the
// gradients and errors once. Scale, codes and errors are those of the two-pass form
// exactly: the same maximum (the warp's maximum of |c| is the chunk's) and the same
// quantize8.
constexpr int kLocoOnePassU = 2;     // groups in flight per sweep (both sweeps share registers)

template <typename G, int BITS>
__global__ void __launch_bounds__(kBlock) k_loco_fused(LocoArgs a)
{
    constexpr int U = kLocoOnePassU;      // second sweep (from the L2)
    constexpr int UA = kLocoU;            // first sweep (from DRAM): more groups in flight
    const int lane = threadIdx.x & 31;
    const float L = (float)((1 << (BITS - 1)) - 1);
    int64_t s0, s1;
    warp_items((int64_t)a.W * a.nchunks, s0, s1);
    const int64_t CG = a.C / 256;
    for (int64_t slot = s0; slot < s1; ++slot) {
        const int64_t t0 = slot * CG;
        float run = 0.0f;
        for (int64_t tb = 0; tb < CG; tb += UA) {
            GradRaw<G> gr[UA];
            float ev[UA][8];
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                if (tb + u < CG) {
                    const int64_t e0 = (t0 + tb + u) * 256 + lane * 8;
                    gr[u] = GradRaw<G>::load_l2(a.g, e0);
                    ld8_l2(a.err + e0, ev[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                if (tb + u < CG) {
                    float gv[8];
                    gr[u].widen(gv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) run = fmaxf(run, fabsf(__fadd_rn(gv[j], __fmul_rn(a.ratio, ev[u][j]))));
                }
            }
        }
        const float s = __fdiv_rn(warp_max(run), L);
        const float inv = __frcp_rn(s);
        if (lane == 0) a.scale[slot] = s;
        for (int64_t tb = 0; tb < CG; tb += U) {
            GradRaw<G> gr[U];
            float ev[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (tb + u < CG) {
                    const int64_t e0 = (t0 + tb + u) * 256 + lane * 8;
                    gr[u] = GradRaw<G>::load(a.g, e0);
                    ld8_stream(a.err + e0, ev[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (tb + u < CG) {
                    float gv[8];
                    gr[u].widen(gv);
                    uint32_t lo, hi;
                    quantize8<BITS>(gv, ev[u], s, inv, a.ratio, a.beta, a.keep, lo, hi);
                    const int64_t e0 = (t0 + tb + u) * 256 + lane * 8;
                    st8_stream(a.err + e0, ev[u]);
                    store_codes<BITS>(a.codes + e0 * BITS / 8, lo, hi);
                }
            }
        }
    }
}

// The same for chunks of one, two or four groups (C = 256, 512, 1024; not 768): each warp
// takes kLocoU groups at a time -- whole chunks, as the chunk size divides kLocoU groups
// and a warp's range starts on a chunk -- and keeps them in registers: the maxima of the
// groups, combined per chunk, give the scales, and the groups are quantized from the
// registers they were loaded into. One read, and kLocoU groups in flight per warp.
// Residency (measured): three blocks per SM for 16-bit gradients (80 registers), two for
// float32 ones, whose wider rows spill at 80.
template <typename G, int BITS>
__global__ void __launch_bounds__(kBlock, sizeof(G) == 4 ? 2 : 3) k_loco_fused_small(LocoArgs a)
{
    constexpr int U = kLocoU;
    const int lane = threadIdx.x & 31;
    const float L = (float)((1 << (BITS - 1)) - 1);
    int64_t s0, s1;
    warp_items((int64_t)a.W * a.nchunks, s0, s1);
    const int CG = (int)(a.C / 256);                  // 1, 2 or 4
    const int64_t t1 = s1 * CG;
    for (int64_t tb = s0 * CG; tb < t1; tb += U) {
        GradRaw<G> gr[U];
        float ev[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u < t1) {
                const int64_t e0 = (tb + u) * 256 + lane * 8;
                gr[u] = GradRaw<G>::load(a.g, e0);
                ld8_stream(a.err + e0, ev[u]);
            }
        }
        float mx[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float run = 0.0f;
            if (tb + u < t1) {
                float gv[8];
                gr[u].widen(gv);
#pragma unroll
                for (int j = 0; j < 8; ++j) run = fmaxf(run, fabsf(__fadd_rn(gv[j], __fmul_rn(a.ratio, ev[u][j]))));
            }
            mx[u] = warp_max(run);
        }
        // the maximum of each group's chunk (groups u..u+CG-1 with u a multiple of CG)
        if (CG >= 2) {
#pragma unroll
            for (int u = 0; u < U; u += 2) mx[u] = mx[u + 1] = fmaxf(mx[u], mx[u + 1]);
        }
        if (CG == 4) mx[0] = mx[1] = mx[2] = mx[3] = fmaxf(mx[0], mx[2]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u < t1) {
                const float sc = __fdiv_rn(mx[u], L);
                const float inv = __frcp_rn(sc);
                if (lane == 0 && (u % CG) == 0) a.scale[(tb + u) / CG] = sc;
                float gv[8];
                gr[u].widen(gv);
                uint32_t lo, hi;
                quantize8<BITS>(gv, ev[u], sc, inv, a.ratio, a.beta, a.keep, lo, hi);
                const int64_t e0 = (tb + u) * 256 + lane * 8;
                st8_stream(a.err + e0, ev[u]);
                store_codes<BITS>(a.codes + e0 * BITS / 8, lo, hi);
            }
        }
    }
}

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t* p, int (&q)[8])
{
    if (BITS == 4) {
        const uint32_t word = __ldcs(reinterpret_cast<const unsigned int*>(p));
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = ((int)(word << (28 - 4 * j))) >> 28;   // sign-extend nibble j
    } else {
        const uint2 r = __ldcs(reinterpret_cast<const uint2*>(p));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            q[j] = ((int)(r.x << (24 - 8 * j))) >> 24;
            q[j + 4] = ((int)(r.y << (24 - 8 * j))) >> 24;
        }
    }
}

// The Adam step on one lane's 8 elements from the sum over workers of the dequantized
// gradients (gbar = acc/W): m, v, x updated in place.
__device__ __forceinline__ void loco_adam8(const float (&acc)[8], float fW, float (&mv)[8], float (&vv)[8],
                                           float (&xv)[8], const LocoArgs& a)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float gbar = div_rn_zero_fast(acc[j], fW);
        mv[j] = __fadd_rn(__fmul_rn(a.b1, mv[j]), __fmul_rn(a.c1, gbar));
        vv[j] = __fadd_rn(__fmul_rn(a.b2, vv[j]), __fmul_rn(a.c2, __fmul_rn(gbar, gbar)));
        const float denom = __fadd_rn(__fsqrt_rn(vv[j]), a.eps);
        float u = div_rn_zero_fast(mv[j], denom);
        if (a.wd != 0.0f) u = __fadd_rn(u, __fmul_rn(a.wd, xv[j]));
        xv[j] = __fsub_rn(xv[j], __fmul_rn(a.lr, u));
    }
}

template <int BITS>
__global__ void __launch_bounds__(kBlock) k_loco_server(LocoArgs a)
{
    const int64_t nvec = a.n / 8;
    const int64_t row_bytes = a.n * BITS / 8;
    const float fW = (float)a.W;
    for (int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i8 < nvec;
         i8 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e0 = i8 * 8;
        const int64_t k = fast_div((uint32_t)(i8 >> 5), a.cg_div);   // e0 / C
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int w = 0; w < a.W; ++w) {
            const float s = __ldg(a.scale + (int64_t)w * a.nchunks + k);
            int q[8];
            load_codes<BITS>(a.codes + (int64_t)w * row_bytes + e0 * BITS / 8, q);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn((float)q[j], s));
        }
        float mv[8], vv[8], xv[8];
        ld8_stream(a.m + e0, mv);
        ld8_stream(a.v + e0, vv);
        ld8_stream(a.x + e0, xv);
        loco_adam8(acc, fW, mv, vv, xv, a);
        st8_stream(a.m + e0, mv);
        st8_stream(a.v + e0, vv);
        st8_stream(a.x + e0, xv);
    }
}

// Long chunks, after the absmax pass: the quantization of every worker row and the server
// step in one pass. Each block works one contiguous, balanced range of groups (the grid is
// one resident wave) and its warps take the range's groups in turn; per group a warp
// quantizes the W rows in ascending order, with the next row's loads in flight while one
// row is quantized, adds each dequantized row into the sum in that order, and takes the
// Adam step on x, m, v. The codes stay in registers (stored only when a.keep_codes is set),
// so DRAM sees neither their write nor their read-back: W*(grad + 8) + 24 bytes per
// element instead of W*(grad + 8 + bits/4) + 24 for a quantize pass and a server pass.
// Scales, codes, errors and the Adam state are those of the separate passes exactly: the
// same quantize8_levels, the same sums in the same order.
template <typename G, int BITS>
__global__ void __launch_bounds__(kBlock, 2) k_loco_qs(LocoArgs a)
{
    __shared__ float2 s_sc[kBlock / 32][16];   // per warp: (s, rn(1/s)) of each row in its chunk
    const int lane = threadIdx.x & 31;
    float2* sc = s_sc[threadIdx.x >> 5];
    const float L = (float)((1 << (BITS - 1)) - 1);
    const int wpb = blockDim.x >> 5;
    const int64_t g_end = ((int64_t)blockIdx.x + 1) * a.NG / gridDim.x;
    const int64_t CG = a.C / 256;
    const float fW = (float)a.W;
    int64_t cur = -1;
    for (int64_t gi = (int64_t)blockIdx.x * a.NG / gridDim.x + (threadIdx.x >> 5); gi < g_end; gi += wpb) {
        const int64_t k = fast_div((uint32_t)gi, a.cg_div);
        if (k != cur) {
            // the rows' scales of chunk k, formed once per chunk the warp enters; the warp
            // holding the chunk's first group stores them
            cur = k;
            __syncwarp();
            if (lane < a.W) {
                const float s = __fdiv_rn(__uint_as_float(__ldcg(a.amax_bits + (int64_t)lane * a.nchunks + k)), L);
                sc[lane] = make_float2(s, __frcp_rn(s));
                if (gi == k * CG) a.scale[(int64_t)lane * a.nchunks + k] = s;
            }
            __syncwarp();
        }
        const int64_t e0 = gi * 256 + lane * 8;
        float mv[8], vv[8], xv[8], ev[8], acc[8];
        ld8_stream(a.m + e0, mv);
        ld8_stream(a.v + e0, vv);
        ld8_stream(a.x + e0, xv);
        GradRaw<G> gr = GradRaw<G>::load(a.g, e0);
        ld8_stream(a.err + e0, ev);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int w = 0; w < a.W; ++w) {
            const int64_t ew = (int64_t)w * a.n + e0;
            GradRaw<G> gn = gr;
            float en[8];
            if (w + 1 < a.W) {
                gn = GradRaw<G>::load(a.g, ew + a.n);
                ld8_stream(a.err + ew + a.n, en);
            }
            float gv[8];
            gr.widen(gv);
            const float2 si = sc[w];
            int qv[8];
            quantize8_levels<BITS>(gv, ev, si.x, si.y, a.ratio, a.beta, a.keep, qv);
            st8_stream(a.err + ew, ev);
            if (a.keep_codes) {
                uint32_t lo, hi;
                pack_codes<BITS>(qv, lo, hi);
                store_codes<BITS>(a.codes + ew * BITS / 8, lo, hi);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn((float)qv[j], si.x));
            gr = gn;
#pragma unroll
            for (int j = 0; j < 8; ++j) ev[j] = en[j];
        }
        loco_adam8(acc, fW, mv, vv, xv, a);
        st8_stream(a.m + e0, mv);
        st8_stream(a.v + e0, vv);
        st8_stream(a.x + e0, xv);
    }
}

cudaError_t launch_loco_absmax(int dtype, const LocoArgs& a, int grid, cudaStream_t s)
{
    if (dtype == 0) k_loco_absmax<float><<<grid, kBlock, 0, s>>>(a);
    else if (dtype == 1) k_loco_absmax<__half><<<grid, kBlock, 0, s>>>(a);
    else k_loco_absmax<__nv_bfloat16><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename K>
static int occ_of(K kernel)
{
    int blocks = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kBlock, 0) == cudaSuccess ? blocks : 0;
}

int occupancy_loco_absmax(int dtype)
{
    if (dtype == 0) return occ_of(k_loco_absmax<float>);
    if (dtype == 1) return occ_of(k_loco_absmax<__half>);
    return occ_of(k_loco_absmax<__nv_bfloat16>);
}

// The register kernel needs the chunk's group count to divide kLocoU (1, 2 or 4 groups):
// its blocks of kLocoU groups then hold whole chunks. Other short chunks (3 groups, or 5 to
// 16) take the two-sweep kernel.
static bool loco_small_chunks(int64_t C)
{
    const int64_t cg = C / 256;
    return cg == 1 || cg == 2 || cg == 4;
}

cudaError_t launch_loco_fused(int dtype, const LocoArgs& a, int grid, cudaStream_t s)
{
    const bool small = loco_small_chunks(a.C);
#define OB_LOCO_FUSED(G, B)                                              \
    do {                                                                 \
        if (small) k_loco_fused_small<G, B><<<grid, kBlock, 0, s>>>(a);  \
        else k_loco_fused<G, B><<<grid, kBlock, 0, s>>>(a);              \
    } while (0)
    if (a.bits == 4) {
        if (dtype == 0) OB_LOCO_FUSED(float, 4);
        else if (dtype == 1) OB_LOCO_FUSED(__half, 4);
        else OB_LOCO_FUSED(__nv_bfloat16, 4);
    } else {
        if (dtype == 0) OB_LOCO_FUSED(float, 8);
        else if (dtype == 1) OB_LOCO_FUSED(__half, 8);
        else OB_LOCO_FUSED(__nv_bfloat16, 8);
    }
#undef OB_LOCO_FUSED
    return cudaGetLastError();
}

int occupancy_loco_fused(int dtype, int bits, int64_t C)
{
    const bool small = loco_small_chunks(C);
#define OB_LOCO_OCC(G, B) return small ? occ_of(k_loco_fused_small<G, B>) : occ_of(k_loco_fused<G, B>)
    if (bits == 4) {
        if (dtype == 0) OB_LOCO_OCC(float, 4);
        if (dtype == 1) OB_LOCO_OCC(__half, 4);
        OB_LOCO_OCC(__nv_bfloat16, 4);
    }
    if (dtype == 0) OB_LOCO_OCC(float, 8);
    if (dtype == 1) OB_LOCO_OCC(__half, 8);
    OB_LOCO_OCC(__nv_bfloat16, 8);
#undef OB_LOCO_OCC
}

// The same pass for 16-bit gradients and W <= 4, with each lane's data staged in shared
// memory: every lane copies its own 8 elements of a group -- the W rows' gradients and
// errors, then x, m, v -- into a stage of its warp's ring by 16-byte asynchronous copies
// and reads back only what it copied, so the copies need only the lane's own wait, and
// kQsStages groups' loads are in flight per warp without holding registers. On the
// bfloat16 GPT-like buffer (W = 4) it runs at 0.92 of the copy peak where the register
// form, which waits about one memory round trip per group, ran at 0.885; with float32
// gradients (larger stages, 10 warps per SM) the register form measured faster.
// Stage layout: gradients [4 rows][32 lanes][8], errors [4][32][8], then x, m, v [32][8].
constexpr int kQsStages = 2;
constexpr int kQsMaxRows = 4;
constexpr int kQsSmemBudget = 227 * 1024;   // dynamic shared memory one block may take

template <typename G>
struct QsStage {
    static constexpr uint32_t kG = 8 * sizeof(G);                  // a lane's gradients
    static constexpr uint32_t kGOff = 0;
    static constexpr uint32_t kEOff = kQsMaxRows * 32 * kG;
    static constexpr uint32_t kXOff = kEOff + kQsMaxRows * 32 * 32;
    static constexpr uint32_t kBytes = kXOff + 3 * 32 * 32;       // + x, m, v
    // warps per block: as many rings as fit (one block per SM; 12 for 16-bit gradients)
    static constexpr int kWarps = kQsSmemBudget / (kQsStages * (int)kBytes) < 16
                                      ? kQsSmemBudget / (kQsStages * (int)kBytes) : 16;
    static constexpr size_t kSmem = (size_t)kWarps * kQsStages * kBytes;
};

template <typename G, int BITS>
__global__ void __launch_bounds__(QsStage<G>::kWarps * 32, 1) k_loco_qs_staged(LocoArgs a)
{
    using St = QsStage<G>;
    constexpr int S = kQsStages;
    constexpr int NW = St::kWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 s_sc[NW][kQsMaxRows];   // per warp: (s, rn(1/s)) of each row
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    float2* sc = s_sc[wib];
    const unsigned char* ring = smem + (size_t)wib * S * St::kBytes;
    const uint32_t ring_u32 = smem_u32(ring);
    const uint64_t pol = policy_evict_first();
    const float L = (float)((1 << (BITS - 1)) - 1);
    const int64_t b0 = (int64_t)blockIdx.x * a.NG / gridDim.x;
    const int64_t b1 = ((int64_t)blockIdx.x + 1) * a.NG / gridDim.x;
    const int64_t count = b1 - b0 > wib ? (b1 - b0 - wib + NW - 1) / NW : 0;
    const int64_t CG = a.C / 256;
    const float fW = (float)a.W;

    // this lane's copies of the warp's item i (group b0 + wib + i*NW) into stage s
    auto issue = [&](int s, int64_t i) {
        const int64_t e0 = (b0 + wib + i * NW) * 256 + lane * 8;
        const uint32_t st = ring_u32 + (uint32_t)s * St::kBytes;
        for (int w = 0; w < a.W; ++w) {
            const int64_t ew = (int64_t)w * a.n + e0;
            const unsigned char* gsrc = static_cast<const unsigned char*>(a.g) + ew * (int64_t)sizeof(G);
            const uint32_t gdst = st + St::kGOff + ((uint32_t)w * 32 + lane) * St::kG;
#pragma unroll
            for (uint32_t c = 0; c < St::kG; c += 16) cp_async16(gdst + c, gsrc + c, pol);
            const uint32_t edst = st + St::kEOff + ((uint32_t)w * 32 + lane) * 32;
            cp_async16(edst, a.err + ew, pol);
            cp_async16(edst + 16, a.err + ew + 4, pol);
        }
        const uint32_t xdst = st + St::kXOff + lane * 32;
        cp_async16(xdst, a.x + e0, pol);
        cp_async16(xdst + 16, a.x + e0 + 4, pol);
        cp_async16(xdst + 1024, a.m + e0, pol);
        cp_async16(xdst + 1040, a.m + e0 + 4, pol);
        cp_async16(xdst + 2048, a.v + e0, pol);
        cp_async16(xdst + 2064, a.v + e0 + 4, pol);
    };
    auto ld8s = [&](const unsigned char* p, float (&v)[8]) {
        const float4 lo = reinterpret_cast<const float4*>(p)[0];
        const float4 hi = reinterpret_cast<const float4*>(p)[1];
        v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
        v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
    };

#pragma unroll
    for (int s = 0; s < S; ++s) {
        if (s < count) issue(s, s);
        cp_async_commit();
    }
    int64_t cur = -1;
    for (int64_t i = 0; i < count; ++i) {
        const int s = (int)(i % S);
        const int64_t gi = b0 + wib + i * NW;
        const int64_t k = fast_div((uint32_t)gi, a.cg_div);
        if (k != cur) {
            // the rows' scales of chunk k, formed once per chunk the warp enters; the warp
            // holding the chunk's first group stores them
            cur = k;
            __syncwarp();
            if (lane < a.W) {
                const float sv = __fdiv_rn(__uint_as_float(__ldcg(a.amax_bits + (int64_t)lane * a.nchunks + k)), L);
                sc[lane] = make_float2(sv, __frcp_rn(sv));
                if (gi == k * CG) a.scale[(int64_t)lane * a.nchunks + k] = sv;
            }
            __syncwarp();
        }
        cp_async_wait<S - 1>();         // this lane's copies of item i have landed
        const unsigned char* stg = ring + (size_t)s * St::kBytes;
        const int64_t e0 = gi * 256 + lane * 8;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int w = 0; w < a.W; ++w) {
            const int64_t ew = (int64_t)w * a.n + e0;
            GradRaw<G> gr;
            gr = *reinterpret_cast<const GradRaw<G>*>(stg + St::kGOff + ((uint32_t)w * 32 + lane) * St::kG);
            float gv[8], ev[8];
            gr.widen(gv);
            ld8s(stg + St::kEOff + ((uint32_t)w * 32 + lane) * 32, ev);
            const float2 si = sc[w];
            int qv[8];
            quantize8_levels<BITS>(gv, ev, si.x, si.y, a.ratio, a.beta, a.keep, qv);
            st8_stream(a.err + ew, ev);
            if (a.keep_codes) {
                uint32_t lo, hi;
                pack_codes<BITS>(qv, lo, hi);
                store_codes<BITS>(a.codes + ew * BITS / 8, lo, hi);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn((float)qv[j], si.x));
        }
        float xv[8], mv[8], vv[8];
        ld8s(stg + St::kXOff + lane * 32, xv);
        ld8s(stg + St::kXOff + 1024 + lane * 32, mv);
        ld8s(stg + St::kXOff + 2048 + lane * 32, vv);
        loco_adam8(acc, fW, mv, vv, xv, a);
        st8_stream(a.m + e0, mv);
        st8_stream(a.v + e0, vv);
        st8_stream(a.x + e0, xv);
        // the lane has read all it copied into stage s: it may fill it again
        if (i + S < count) issue(s, i + S);
        cp_async_commit();
    }
    cp_async_wait<0>();
}

static bool loco_qs_staged(int W, int dtype)
{
    return W <= kQsMaxRows && dtype != 0;
}

cudaError_t prepare_loco()
{
#define OB_QS_ATTR(G, B)                                                                                     \
    if (cudaError_t e = cudaFuncSetAttribute(k_loco_qs_staged<G, B>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             (int)QsStage<G>::kSmem))                                         \
        return e;
    OB_QS_ATTR(__half, 4) OB_QS_ATTR(__half, 8) OB_QS_ATTR(__nv_bfloat16, 4) OB_QS_ATTR(__nv_bfloat16, 8)
#undef OB_QS_ATTR
    return cudaSuccess;
}

cudaError_t launch_loco_qs(int dtype, const LocoArgs& a, int grid, cudaStream_t s)
{
    if (loco_qs_staged(a.W, dtype)) {
#define OB_QS_STAGED(G, B) k_loco_qs_staged<G, B><<<grid, QsStage<G>::kWarps * 32, QsStage<G>::kSmem, s>>>(a)
        if (a.bits == 4) {
            if (dtype == 1) OB_QS_STAGED(__half, 4);
            else OB_QS_STAGED(__nv_bfloat16, 4);
        } else {
            if (dtype == 1) OB_QS_STAGED(__half, 8);
            else OB_QS_STAGED(__nv_bfloat16, 8);
        }
#undef OB_QS_STAGED
        return cudaGetLastError();
    }
    if (a.bits == 4) {
        if (dtype == 0) k_loco_qs<float, 4><<<grid, kBlock, 0, s>>>(a);
        else if (dtype == 1) k_loco_qs<__half, 4><<<grid, kBlock, 0, s>>>(a);
        else k_loco_qs<__nv_bfloat16, 4><<<grid, kBlock, 0, s>>>(a);
    } else {
        if (dtype == 0) k_loco_qs<float, 8><<<grid, kBlock, 0, s>>>(a);
        else if (dtype == 1) k_loco_qs<__half, 8><<<grid, kBlock, 0, s>>>(a);
        else k_loco_qs<__nv_bfloat16, 8><<<grid, kBlock, 0, s>>>(a);
    }
    return cudaGetLastError();
}

template <typename G, int B>
static int occ_staged()
{
    int blocks = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_loco_qs_staged<G, B>, QsStage<G>::kWarps * 32,
                                                         QsStage<G>::kSmem) == cudaSuccess ? blocks : 0;
}

int occupancy_loco_qs(int dtype, int bits, int W)
{
    if (loco_qs_staged(W, dtype)) {
        if (bits == 4) return dtype == 1 ? occ_staged<__half, 4>() : occ_staged<__nv_bfloat16, 4>();
        return dtype == 1 ? occ_staged<__half, 8>() : occ_staged<__nv_bfloat16, 8>();
    }
    if (bits == 4) {
        if (dtype == 0) return occ_of(k_loco_qs<float, 4>);
        if (dtype == 1) return occ_of(k_loco_qs<__half, 4>);
        return occ_of(k_loco_qs<__nv_bfloat16, 4>);
    }
    if (dtype == 0) return occ_of(k_loco_qs<float, 8>);
    if (dtype == 1) return occ_of(k_loco_qs<__half, 8>);
    return occ_of(k_loco_qs<__nv_bfloat16, 8>);
}

cudaError_t launch_loco_server(const LocoArgs& a, int grid, cudaStream_t s)
{
    if (a.bits == 4) k_loco_server<4><<<grid, kBlock, 0, s>>>(a);
    else k_loco_server<8><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ob
