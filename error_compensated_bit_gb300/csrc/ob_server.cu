// Server side of the compression-stage step and the final update.
//
// Method: DeepSpeed 1-bit Adam training guide, §4 (compressed_allreduce: a server_error
// per GPU, the averaged momentum recompressed and sent back; then
// update = exp_avg/(sqrt(exp_avg_sq)+eps), weight decay and learning rate), §3.5
// (exp_avg multiplied by exp_avg_mask after the exchange); "1-bit Adam" review,
// "Proposed method" (the variance frozen after the warm-up preconditions the update).
//
// The exchange is a gather inside device memory: the server pass reads, for its
// elements, every worker's packed words (the all-to-all), and the update pass reads
// the server's words (the all-gather). Nothing is copied.
#include "ob_common.cuh"
#include "ob_tma.cuh"

namespace ob {

// All elements of a chunk share the W scales, so the server average depends only on the
// element's W sign bits. A warp tabulates, once per chunk, the running sum over the first
// min(W, 8) workers for all their sign patterns -- each entry summed in the same order as
// the definition, so it is exactly the float32 partial sum the definition reaches after
// those workers. For W <= 8 the entry is already divided by W (the final average); for
// W > 8 the element continues the sum over the remaining workers in order.
template <int W>
__device__ __forceinline__ void build_average_table(float* tab, const float (&sw)[W], int lane)
{
    constexpr int T = W < 8 ? W : 8;
    __syncwarp();                       // the previous chunk's table is no longer read
    for (uint32_t e = lane; e < (1u << T); e += 32) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < T; ++w) sum = __fadd_rn(sum, signed_scale(sw[w], (e >> w) & 1u));
        if (W <= 8) sum = (W & (W - 1)) == 0 ? __fmul_rn(sum, 1.0f / (float)W) : __fdiv_rn(sum, (float)W);
        tab[e] = sum;
    }
    __syncwarp();
}

// 8x8 bit-matrix transpose (three delta swaps, as in Hacker's Delight): in, byte r bit c
// is entry (r, c); out, byte c bit r. With byte w = worker w's signs of this lane's 8
// elements, output byte j is element j's sign pattern (bit w = worker w).
__device__ __forceinline__ uint64_t transpose8x8(uint64_t x)
{
    uint64_t t;
    t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
    x = x ^ t ^ (t << 7);
    t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
    x = x ^ t ^ (t << 14);
    t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
    x = x ^ t ^ (t << 28);
    return x;
}

// a = (sum over w ascending of +-S_wk)/W;  e_s = yprev - T_prev*sign(yprev);  y = a + e_s;
// bit = (y >= 0); ybuf = y; chunk sums of y^2 -> T_next.
// Memory per element: W/8 (worker bits) + 4 + 4 (y) + 1/8 (server bits).
// This lane's sign bytes from the words holding its elements' sign bits in each worker
// row (word lane >> 2 of the group's eight; zero for rows W and above): byte (lane & 3)
// of row w's word becomes byte w of the result. Two rounds of byte permutes gather four
// rows into one word.
__device__ __forceinline__ uint64_t pack_sign_bytes(const uint32_t (&wv)[8], int lane)
{
    const uint32_t b = (uint32_t)lane & 3u;
    const uint32_t pick = b | ((b + 4u) << 4);        // byte b of the first and of the second word
    const uint32_t lo = __byte_perm(__byte_perm(wv[0], wv[1], pick), __byte_perm(wv[2], wv[3], pick), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(wv[4], wv[5], pick), __byte_perm(wv[6], wv[7], pick), 0x5410);
    return ((uint64_t)hi << 32) | lo;
}

// Used for W <= 8: one group's y per warp in flight, 64 registers (four blocks per SM). The
// worker sign words come in one coalesced 128-byte load per row for four groups at a time
// (lane l holds word l), and each group takes its words from the holding lanes by
// shuffles: a quarter of the load requests of a 32-byte load per row and group, 5-6%
// faster. Keeping several groups in flight through shared memory (cp.async copies as in
// k_server_staged, or bulk copies) measured slower here; it pays for W > 8.
template <int W>
__global__ void __launch_bounds__(kBlock, 4) k_server(ServerArgs a)
{
    static_assert(W <= 8, "the register server pass covers up to eight workers");
    __shared__ float s_tab[(kBlock / 32) << W];
    float* tab = s_tab + ((threadIdx.x >> 5) << W);
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const Part pt = a.pt;
    const int64_t words_per_row = a.n / 32;
    pdl_wait();             // the worker pass has finished
    pdl_allow_next();

    // group and chunk indices fit 32 bits (W * n / 256 < 2^32 is checked at init)
    const uint32_t CG = (uint32_t)pt.CG;
    for (int64_t q = warp; q < pt.P; q += nwarps) {
        const uint32_t g0 = (uint32_t)range_begin(pt, q);
        const uint32_t g1 = (uint32_t)range_begin(pt, q + 1);
        uint32_t k = g0 / CG;
        const uint32_t kfirst = k;
        uint32_t kend = (k + 1) * CG;

        float sw[W];
#pragma unroll
        for (int w = 0; w < W; ++w) sw[w] = __ldg(a.s_next + (int64_t)w * pt.nchunks + k);
        float tp = __ldg(a.t_prev + k);
        build_average_table<W>(tab, sw, lane);
        Sum2 acc[1] = {{0.0f, 0.0f}};
        uint32_t blk[8];    // row w: word `lane` of the 32 words of groups 4b .. 4b + 3

        for (uint32_t gi = g0; gi < g1; ++gi) {
            if (gi == kend) {
                flush_chunk<1, kFlushInline>(pt, q, 1, 0, k, kfirst, g0, g1, acc, a.part, a.cnt, a.t_next, a.C, a.ybuf, a.n, lane);
                ++k;
                kend += CG;
#pragma unroll
                for (int w = 0; w < W; ++w) sw[w] = __ldg(a.s_next + (int64_t)w * pt.nchunks + k);
                tp = __ldg(a.t_prev + k);
                build_average_table<W>(tab, sw, lane);
            }
            const int jg = (int)(gi & 3u);
            if (jg == 0 || gi == g0) {
                // one coalesced 128-byte load per row covers this group and the next three
                const int64_t wb = (int64_t)(gi & ~3u) * 8 + lane;
                const bool in = wb < words_per_row;
#pragma unroll
                for (int w = 0; w < W; ++w) blk[w] = in ? __ldcs(a.wbits + (int64_t)w * words_per_row + wb) : 0u;
            }
            uint32_t wv[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) wv[w] = w < W ? __shfl_sync(kFull, blk[w], jg * 8 + (lane >> 2)) : 0u;
            const uint64_t raw = pack_sign_bytes(wv, lane);
            float yv[8];
            ld8_stream(a.ybuf + (int64_t)gi * 256 + lane * 8, yv);
            const uint64_t pat = transpose8x8(raw);   // byte j: element j's signs, bit w = worker w
            uint32_t byte = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float avg = tab[(uint32_t)(pat >> (8 * j)) & 0xffu];
                const float es = __fsub_rn(yv[j], signed_scale(tp, yv[j] >= 0.0f));
                const float y = __fadd_rn(avg, es);
                yv[j] = y;
                byte |= (y >= 0.0f ? 1u : 0u) << j;
                sum2_add_sq(acc[0], y);
            }
            st8_stream(a.ybuf + (int64_t)gi * 256 + lane * 8, yv);
            const uint32_t word = quad_word(byte, lane);
            if ((lane & 3) == 0) __stcs(a.sbits + (int64_t)gi * 8 + (lane >> 2), word);
        }
        flush_chunk<1, kFlushInline>(pt, q, 1, 0, k, kfirst, g0, g1, acc, a.part, a.cnt, a.t_next, a.C, a.ybuf, a.n, lane);
    }
}

// The same pass for W > 8, where the per-element work grows and one group in flight per
// warp no longer covers the memory latency. Each warp works one contiguous range of groups through a ring of kServerStages(W)
// shared-memory stages: a stage holds one group's previous y (1 KB) and the group's 32
// bytes of sign words from each worker row, copied by per-lane 16-byte asynchronous copies
// (two per lane for y, one per lane for the first 2W lanes for the signs), so that several
// groups' loads are in flight per warp without holding registers. Dynamic shared memory:
// the warps' average tables, then the warps' rings.
template <int W>
struct ServerStage {
    static constexpr int kStages = W > 8 ? 3 : 4;
    static constexpr uint32_t kSignOff = 1024;                    // after the 256 y values
    static constexpr uint32_t kBytes = 1024 + 32 * W;
    static constexpr uint32_t kTabBytes = 4u << (W < 8 ? W : 8);  // one table per warp
    static constexpr size_t kSmem = (size_t)(kBlock / 32) * (kTabBytes + kStages * kBytes);
};

template <int W>
__global__ void __launch_bounds__(kBlock, 4) k_server_staged(ServerArgs a)
{
    static_assert(W > 8, "the staged server pass covers more than eight workers");
    using St = ServerStage<W>;
    constexpr int S = St::kStages;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    float* tab = reinterpret_cast<float*>(smem + (size_t)wib * St::kTabBytes);
    unsigned char* ring = smem + (size_t)(kBlock / 32) * St::kTabBytes + (size_t)wib * S * St::kBytes;
    const uint32_t ring_u32 = smem_u32(ring);
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const Part pt = a.pt;
    const int64_t words_per_row = a.n / 32;
    const uint64_t pol = policy_evict_first();
    pdl_wait();             // the worker pass has finished
    pdl_allow_next();

    // this lane's copies of group gi into stage s: two 16-byte pieces of y, and piece
    // (lane & 1) of worker row (lane >> 1)'s 32 bytes of sign words
    auto issue = [&](int s, int64_t gi) {
        const uint32_t dst = ring_u32 + (uint32_t)s * St::kBytes;
        const float* ysrc = a.ybuf + gi * 256 + lane * 8;
        cp_async16(dst + lane * 32, ysrc, pol);
        cp_async16(dst + lane * 32 + 16, ysrc + 4, pol);
        if (lane < 2 * W) {
            const uint32_t* wsrc = a.wbits + (int64_t)(lane >> 1) * words_per_row + gi * 8 + (lane & 1) * 4;
            cp_async16(dst + St::kSignOff + lane * 16, wsrc, pol);
        }
    };

    for (int64_t q = warp; q < pt.P; q += nwarps) {
        const int64_t g0 = range_begin(pt, q);
        const int64_t g1 = range_begin(pt, q + 1);
        int64_t k = g0 / pt.CG;
        const int64_t kfirst = k;
        int64_t kend = (k + 1) * pt.CG;

        __syncwarp();                       // the previous range's last stage is read
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if (g0 + s < g1) issue(s, g0 + s);
            cp_async_commit();
        }
        float sw[W];
#pragma unroll
        for (int w = 0; w < W; ++w) sw[w] = __ldg(a.s_next + (int64_t)w * pt.nchunks + k);
        float tp = __ldg(a.t_prev + k);
        build_average_table<W>(tab, sw, lane);
        Sum2 acc[1] = {{0.0f, 0.0f}};

        for (int64_t gi = g0; gi < g1; ++gi) {
            if (gi == kend) {
                flush_chunk<1, kFlushLastCall>(pt, q, 1, 0, k, kfirst, g0, g1, acc, a.part, a.cnt, a.t_next, a.C, a.ybuf, a.n, lane);
                ++k;
                kend += pt.CG;
#pragma unroll
                for (int w = 0; w < W; ++w) sw[w] = __ldg(a.s_next + (int64_t)w * pt.nchunks + k);
                tp = __ldg(a.t_prev + k);
                build_average_table<W>(tab, sw, lane);
            }
            const int s = (int)((gi - g0) % S);
            cp_async_wait<S - 1>();         // this lane's copies of group gi have landed
            __syncwarp();                   // ... and every other lane's
            const unsigned char* stg = ring + (size_t)s * St::kBytes;
            float yv[8];
            {
                const float4 y0 = reinterpret_cast<const float4*>(stg)[2 * lane];
                const float4 y1 = reinterpret_cast<const float4*>(stg)[2 * lane + 1];
                yv[0] = y0.x; yv[1] = y0.y; yv[2] = y0.z; yv[3] = y0.w;
                yv[4] = y1.x; yv[5] = y1.y; yv[6] = y1.z; yv[7] = y1.w;
            }
            // byte (lane & 3) of word (lane >> 2) of each row: this lane's 8 sign bits
            uint64_t lo = 0, hi = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) lo |= (uint64_t)stg[St::kSignOff + w * 32 + lane] << (8 * w);
#pragma unroll
            for (int w = 8; w < W; ++w) hi |= (uint64_t)stg[St::kSignOff + w * 32 + lane] << (8 * (w - 8));
            __syncwarp();                   // every lane is done with stage s
            if (gi + S < g1) issue(s, gi + S);
            cp_async_commit();
            lo = transpose8x8(lo);
            hi = transpose8x8(hi);
            uint32_t byte = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // the table's partial sum over workers 0..7, then workers 8.. in order
                float avg = tab[(uint32_t)(lo >> (8 * j)) & 0xffu];
                const uint32_t pat = (uint32_t)(hi >> (8 * j)) & 0xffu;
#pragma unroll
                for (int w = 8; w < W; ++w) avg = __fadd_rn(avg, signed_scale(sw[w], (pat >> (w - 8)) & 1u));
                avg = (W & (W - 1)) == 0 ? __fmul_rn(avg, 1.0f / (float)W) : __fdiv_rn(avg, (float)W);
                const float es = __fsub_rn(yv[j], signed_scale(tp, yv[j] >= 0.0f));
                const float y = __fadd_rn(avg, es);
                yv[j] = y;
                byte |= (y >= 0.0f ? 1u : 0u) << j;
                sum2_add_sq(acc[0], y);
            }
            st8_stream(a.ybuf + gi * 256 + lane * 8, yv);
            const uint32_t word = quad_word(byte, lane);
            if ((lane & 3) == 0) __stcs(a.sbits + gi * 8 + (lane >> 2), word);
        }
        cp_async_wait<0>();                 // nothing of this range is left in flight
        flush_chunk<1, kFlushLastCall>(pt, q, 1, 0, k, kfirst, g0, g1, acc, a.part, a.cnt, a.t_next, a.C, a.ybuf, a.n, lane);
    }
}

// m = T_k*sign(y) [* mask];  x -= lr*(m/(sqrt(v)+eps) [+ wd*x]).
// Memory per element: 1/8 (server bits) [+ 1/8 mask bits] + 4 (v) + 8 (x) + 4 (m).
// Block 0 also moves this step's scales into the "previous" slots for the next step:
// every kernel that reads the previous slots (worker, server) has finished by now.
// Groups per warp iteration (all their loads in flight together): four without a mask,
// two with one (measured faster there: the mask words add loads per group).
template <bool MASKED>
__global__ void __launch_bounds__(kBlock) k_update(UpdateArgs a)
{
    constexpr int U = MASKED ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    constexpr bool masked = MASKED;
    // one contiguous, balanced range of groups per warp (the grid is one resident wave)
    const int64_t g_end = (warp + 1) * a.NG / nwarps;
    pdl_wait();             // the server pass has finished
    pdl_allow_next();

    for (int64_t gb = warp * a.NG / nwarps; gb < g_end; gb += U) {
        float vv[U][8], xv[U][8];
        float T[U];
        uint32_t sb[U];
        // masked: the U groups' server and mask words in one coalesced load per bit row
        // (lane l holds word l of the 8U words from group gb on; measured faster there,
        // and slower than one word per lane and group without a mask)
        const int64_t wb = gb * 8 + lane;
        const bool win = masked && lane < 8 * U && wb < g_end * 8;
        const uint32_t swd = win ? __ldcs(a.sbits + wb) : 0u;
        const uint32_t mwd = win ? __ldcs(a.maskbits + wb) : 0u;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t gi = gb + u;
            if (gi < g_end) {
                const int64_t e0 = gi * 256 + lane * 8;
                T[u] = __ldg(a.t_next + fast_div((uint32_t)gi, a.cg_div));
                if (!masked) sb[u] = lane_byte(a.sbits, gi, lane);
                ld8_stream(a.v + e0, vv[u]);
                ld8_stream(a.x + e0, xv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t gi = gb + u;
            uint32_t sbu, mbu;
            if (masked) {
                // this lane's 8 bits of group gi: byte (lane & 3) of the group's word lane >> 2
                const int src = u * 8 + (lane >> 2);
                sbu = (__shfl_sync(kFull, swd, src) >> (8 * (lane & 3))) & 0xffu;
                mbu = (__shfl_sync(kFull, mwd, src) >> (8 * (lane & 3))) & 0xffu;
            } else {
                sbu = sb[u];
                mbu = 0xffu;
            }
            if (gi < g_end) {
                const int64_t e0 = gi * 256 + lane * 8;
                float mv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float st = signed_scale(T[u], (sbu >> j) & 1u);
                    const float denom = __fadd_rn(__fsqrt_rn(vv[u][j]), a.eps);
                    float mi = st, uu;
                    if (masked) {
                        // a masked element has mi = st*0 = +-0 and mi/denom = mi (denom > 0);
                        // the quotient is formed from st and then selected, so the division
                        // never sees the zero numerators that send it down its slow path
                        const bool on = ((mbu >> j) & 1u) != 0u;
                        mi = __fmul_rn(st, on ? 1.0f : 0.0f);
                        const float q = __fdiv_rn(st, denom);
                        uu = on ? q : mi;
                    } else {
                        uu = __fdiv_rn(mi, denom);
                    }
                    mv[j] = mi;
                    if (a.wd != 0.0f) uu = __fadd_rn(uu, __fmul_rn(a.wd, xv[u][j]));
                    xv[u][j] = __fsub_rn(xv[u][j], __fmul_rn(a.lr, uu));
                }
                st8_stream(a.m + e0, mv);
                st8_stream(a.x + e0, xv[u]);
            }
        }
    }

    // this step's scales become the previous ones (nothing in the update reads those); when
    // they are many, k_scales does it instead and the counts here are zero
    if (blockIdx.x == 0) {
        for (int64_t i = threadIdx.x; i < a.nscales_w; i += blockDim.x) a.s_prev[i] = a.s_next[i];
        for (int64_t i = threadIdx.x; i < a.nchunks; i += blockDim.x) a.t_prev[i] = a.t_next[i];
    }
}

// This step's scales become the previous ones, over the whole grid (many scales).
__global__ void __launch_bounds__(kBlock) k_scales(UpdateArgs a)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    pdl_wait();             // the update pass has finished
    pdl_allow_next();
    for (int64_t i = tid; i < a.nscales_w; i += nthreads) a.s_prev[i] = a.s_next[i];
    for (int64_t i = tid; i < a.nchunks; i += nthreads) a.t_prev[i] = a.t_next[i];
}

// Momentum mask (float 0/1) -> packed bits, bit = (mask != 0).
__global__ void __launch_bounds__(kBlock) k_mask(MaskArgs a)
{
    const int64_t nwords = a.n / 32;
    for (int64_t wi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; wi < nwords;
         wi += (int64_t)gridDim.x * blockDim.x) {
        uint32_t word = 0;
        for (int t = 0; t < 32; ++t) word |= (a.mask01[wi * 32 + t] != 0.0f ? 1u : 0u) << t;
        a.bits[wi] = word;
    }
}

// True residuals from the stored (z, S) and (y, T): e = z - S*sign(z).
__global__ void __launch_bounds__(kBlock) k_export(ExportArgs a)
{
    const int64_t total = (int64_t)(a.W + 1) * a.n;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i / a.n, e = i % a.n;
        const int64_t k = e / a.C;
        if (w < a.W) {
            const float z = a.zbuf[i];
            a.ew_out[i] = __fsub_rn(z, signed_scale(a.s_prev[w * a.nchunks + k], z >= 0.0f));
        } else {
            const float y = a.ybuf[e];
            a.es_out[e] = __fsub_rn(y, signed_scale(a.t_prev[k], y >= 0.0f));
        }
    }
}

template <int W>
static cudaError_t launch_s(const ServerArgs& a, int grid, cudaStream_t s)
{
    if constexpr (W > 8) return launch_pdl(k_server_staged<W>, grid, kBlock, ServerStage<W>::kSmem, s, a);
    else return launch_pdl(k_server<W>, grid, kBlock, 0, s, a);
}

template <int W>
static cudaError_t prepare_s()
{
    if constexpr (W <= 8) return cudaSuccess;
    else return cudaFuncSetAttribute(k_server_staged<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)ServerStage<W>::kSmem);
}

template <int W>
static int occ_s()
{
    int blocks = 0;
    if (prepare_s<W>() != cudaSuccess) return 0;
    cudaError_t e;
    if constexpr (W > 8)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_server_staged<W>, kBlock, ServerStage<W>::kSmem);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_server<W>, kBlock, 0);
    return e == cudaSuccess ? blocks : 0;
}

#define OB_FOR_EACH_W(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14) X(15) X(16)

cudaError_t launch_server(int W, const ServerArgs& a, int grid, cudaStream_t s)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return launch_s<w>(a, grid, s);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t prepare_server(int W)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return prepare_s<w>();
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return cudaErrorInvalidValue;
}

int occupancy_server(int W)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return occ_s<w>();
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return 0;
}

cudaError_t launch_update(const UpdateArgs& a, int grid, cudaStream_t s)
{
    if (a.maskbits) return launch_pdl(k_update<true>, grid, kBlock, 0, s, a);
    return launch_pdl(k_update<false>, grid, kBlock, 0, s, a);
}

int occupancy_update()
{
    int b0 = 0, b1 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, k_update<false>, kBlock, 0) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k_update<true>, kBlock, 0) != cudaSuccess) return 0;
    return b0 < b1 ? b0 : b1;
}

cudaError_t launch_scales(const UpdateArgs& a, int grid, cudaStream_t s)
{
    return launch_pdl(k_scales, grid, kBlock, 0, s, a);
}

cudaError_t launch_mask(const MaskArgs& a, int grid, cudaStream_t s)
{
    k_mask<<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_export(const ExportArgs& a, int grid, cudaStream_t s)
{
    k_export<<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ob
