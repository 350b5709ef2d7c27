// Worker side of the compression-stage step: momentum, error compensation, chunk RMS
// scale, sign packing and residual, fused in one pass over the W gradient rows.
//
// The kernel template and its launch shape; ob_worker_f32.cu, ob_worker_f16.cu and
// ob_worker_bf16.cu instantiate it per gradient type (in parallel translation units),
// ob_worker.cu dispatches.
//
// Method: "1-bit Adam" review, "Proposed method" (error compensation on the momentum,
// 1-bit compression); DeepSpeed 1-bit Adam training guide, §4 (exp_avg update, then
// compressed_allreduce with a per-worker error buffer), §1 (one sign bit per value).
//
// Per element i (chunk k) and worker w, as single float32 operations in this order:
//   old = b1*m[i];  new = c1*g[w][i];  p = old + new
//   e   = zprev[w][i] - S_prev[w][k]*sign(zprev)      (the stored residual of last step)
//   z   = p + e;  bit = (z >= 0);  zbuf[w][i] = z      (this step's residual is z - S*sign)
// and sum z^2 over each chunk for S[w][k] = sqrt(sum/chunk). The residual of this step
// cannot be written in the same pass (S needs the whole chunk), so z itself is kept and
// the residual is rebuilt from (z, S) when the next step reads it: the state streams
// through HBM once per step instead of twice.
//
// Memory per element: W*(grad bytes + 4 read + 4 write + 1/8 bits) + 4 (m), all
// coalesced 16-byte accesses with streaming cache hints; m is read once for all W.
#pragma once

#include "ob_common.cuh"
#include "ob_tma.cuh"

namespace ob {

// Shared-memory pipeline. A stage holds one 256-element group of up to four gradient
// rows and the matching z rows (plus m in a group's first stage), filled by bulk copies
// (TMA) issued by lane 0 and counted by one mbarrier; with W > 4 a group takes several
// stages. Small stages let up to 16 warps share one SM's shared memory.
// Each warp owns `stages` consecutive stages. Bytes in flight then scale with shared
// memory (up to ~200 KB per SM) rather than with the registers that plain loads need,
// which is what a streaming kernel needs to reach HBM bandwidth.
template <int W, typename G>
struct WorkerStage {
    static constexpr int kRows = W < 4 ? W : 4;                 // rows per stage
    static constexpr int kBlocks = (W + kRows - 1) / kRows;     // stages per group
    static constexpr uint32_t kGradRow = 256 * sizeof(G);
    static constexpr uint32_t kZRow = 256 * 4;
    static constexpr uint32_t kZOff = kRows * kGradRow;
    static constexpr uint32_t kMOff = kRows * (kGradRow + kZRow);
    static constexpr uint32_t kBytes = kMOff + 256 * 4;
};

constexpr int kMaxWarps = 16;
constexpr int kMaxStages = 8;

// Dynamic shared memory of a worker block: [block partials: double [2][kMaxWarps][W], when
// the block pre-combines][two counters][mbarriers: warps x stages x 8 B][stages, 128-byte
// aligned]. The offsets come from config_w through WorkerArgs.
template <int W>
constexpr uint32_t block_part_bytes()
{
    return 2u * kMaxWarps * W * 8u;
}

// Whether the interleaved kernel for (W, G) pre-combines its partials in the block (see
// below): chosen per instantiation, so each kernel carries one flush path. With one block
// of up to 227 KB per SM it fits beside the stages without costing a warp or a stage
// except for 16-bit gradients with W >= 11 (16 warps x 7 KB stages fill the block).
template <int W, typename G>
constexpr bool block_combine_fits()
{
    return !(W >= 11 && sizeof(G) == 2);
}

// Interleaved mode: the warps of a block share one range, so their partial sums of chunk k
// are first combined inside the block. Each warp stores its row totals in shared memory
// and counts itself in; the block's last warp adds them in warp order and flushes one
// partial per row for the block's range (the slot layout of one warp per range), after
// which the chunk's last range combines as usual. A chunk then has one partial per range
// and row instead of one per range, warp and row, so the combination on the step's
// critical path takes about one round of loads instead of one per few ranges. Slot j = k -
// (the range's first chunk) is 0 or 1 (interleaved ranges touch at most two chunks), and a
// block works one range per launch, so no slot is reused within a launch.
template <int W>
__device__ __noinline__ void block_flush(const Part& pt, int64_t q, int wpb, int j, int64_t k, const double* bpart,
                                         double* part, unsigned* cnt, float* scale_out, int64_t C, const float* rows,
                                         int64_t row_stride, int lane)
{
    __syncwarp();
    __threadfence_block();
    for (int r = lane; r < W; r += 32) {
        double sum = 0.0;
        for (int w = 0; w < wpb; ++w) sum += bpart[(j * kMaxWarps + w) * W + r];
        part[((int64_t)r * pt.P + q) * pt.J + j] = sum;
    }
    // lanes 0..W-1 wrote the block's partials; each makes its own writes visible before
    // lane 0 counts the range in (in flush_rest)
    __threadfence();
    __syncwarp();
    flush_rest<W>(pt, 1, k, part, cnt, scale_out, C, rows, row_stride, lane);
}

template <int W>
__device__ __forceinline__ void flush_chunk_block(const Part& pt, int64_t q, int wpb, int wib, int64_t k, int64_t kfirst,
                                                  Sum2 (&acc)[W], double* bpart, unsigned* bcnt, double* part,
                                                  unsigned* cnt, float* scale_out, int64_t C, const float* rows,
                                                  int64_t row_stride, int lane)
{
    const int j = (int)(k - kfirst);
    if constexpr (W <= 4) {
        // few rows: the warp's row totals as float pairs spread over the lanes, each row's
        // holder storing its total as one double. Double operations are slow on this part
        // (per-row double butterflies kept its double pipe busy for about a quarter of a
        // small launch's worker time), and up to four rows reduce-scatter in registers.
        int row;
        const Sum2 t = warp_reduce_rows<W>(acc, lane, row);
        if (row_holder<W>(lane, row)) bpart[(j * kMaxWarps + wib) * W + row] = (double)t.s + (double)t.e;
    } else {
#pragma unroll
        for (int r = 0; r < W; ++r) {
            const double d = warp_sum((double)acc[r].s + (double)acc[r].e);
            if (lane == 0) bpart[(j * kMaxWarps + wib) * W + r] = d;
        }
    }
#pragma unroll
    for (int r = 0; r < W; ++r) {
        acc[r].s = 0.0f;
        acc[r].e = 0.0f;
    }
    unsigned prev = 0;
    if (lane == 0) {
        __threadfence_block();
        prev = atomicAdd(bcnt + j, 1u);
        __threadfence_block();
    }
    prev = __shfl_sync(kFull, prev, 0);
    if (prev == (unsigned)(wpb - 1)) block_flush<W>(pt, q, wpb, j, k, bpart, part, cnt, scale_out, C, rows, row_stride, lane);
}

template <typename G>
__device__ __forceinline__ void ld8_shared(const unsigned char* row, int lane, float (&v)[8]);

template <>
__device__ __forceinline__ void ld8_shared<float>(const unsigned char* row, int lane, float (&v)[8])
{
    const float4 a = reinterpret_cast<const float4*>(row)[2 * lane];
    const float4 b = reinterpret_cast<const float4*>(row)[2 * lane + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void ld8_shared<__half>(const unsigned char* row, int lane, float (&v)[8])
{
    const uint4 r = reinterpret_cast<const uint4*>(row)[lane];
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
__device__ __forceinline__ void ld8_shared<__nv_bfloat16>(const unsigned char* row, int lane, float (&v)[8])
{
    const uint4 r = reinterpret_cast<const uint4*>(row)[lane];
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int W, typename G, bool INTER>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) k_worker(WorkerArgs a)
{
    using St = WorkerStage<W, G>;
    constexpr int R = St::kRows;
    constexpr int NB = St::kBlocks;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int wpb = (int)(blockDim.x >> 5);
    const int S = a.stages;
    const Part pt = a.pt;
    const int64_t words_per_row = a.n / 32;
    const uint32_t bar0 = smem_u32(smem) + a.bars_off + 8u * (uint32_t)(wib * S);
    unsigned char* stage0 = smem + a.stages_off + (size_t)wib * S * St::kBytes;
    const uint32_t st0 = smem_u32(stage0);
    constexpr bool bcomb = INTER && block_combine_fits<W, G>();
    double* bpart = reinterpret_cast<double*>(smem);
    unsigned* bcnt = reinterpret_cast<unsigned*>(smem + a.bcnt_off);
    if (bcomb) {
        if (threadIdx.x == 0) {
            bcnt[0] = 0u;
            bcnt[1] = 0u;
        }
        __syncthreads();
    }

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }
    __syncwarp();
    pdl_wait();             // the previous step's kernels have finished with the buffers
    pdl_allow_next();
    const uint64_t pol = policy_evict_first();
    uint32_t phase = 0;   // bit s: parity of stage s's next completion

    // Interleaved mode (chunks much longer than a block's range): each block works one
    // contiguous range of groups and its warps take the range's groups in turn (warp wib:
    // g0 + wib, g0 + wib + wpb, ...), so the warps of a block stream neighbouring rows
    // together. Otherwise (short chunks) each warp works its own contiguous range, so
    // that no warp has to account for chunks it never touches.
    constexpr bool inter = INTER;
    const int wpr = inter ? wpb : 1;            // warps per range
    const int wir = inter ? wib : 0;            // this warp's index within its range
    const int64_t q0 = inter ? (int64_t)blockIdx.x : (int64_t)blockIdx.x * wpb + wib;
    const int64_t qstep = inter ? (int64_t)gridDim.x : (int64_t)gridDim.x * wpb;
    for (int64_t q = q0; q < pt.P; q += qstep) {
        const int64_t g0 = range_begin(pt, q);
        const int64_t g1 = range_begin(pt, q + 1);
        const int64_t count = g1 - g0 > wir ? (g1 - g0 - wir + wpr - 1) / wpr : 0;
        const int64_t items = count * NB;   // (group, row block) pairs, in order
        const int64_t klast = (g1 - 1) / pt.CG;

        // lane 0: fill stage s with item `it` of this range
        auto issue = [&](int s, int64_t it) {
            const uint32_t bar = bar0 + 8u * s;
            const uint32_t dst = st0 + (uint32_t)s * St::kBytes;
            const int64_t e0 = (g0 + wir + (it / NB) * wpr) * 256;
            const int b = (int)(it % NB);
            const int rows = (W - b * R) < R ? (W - b * R) : R;
            mbar_arrive_expect(bar, (uint32_t)rows * (St::kGradRow + St::kZRow) + (b == 0 ? 256u * 4u : 0u));
            for (int r = 0; r < rows; ++r) {
                const int64_t row = (int64_t)(b * R + r) * a.n + e0;
                bulk_load_hint(dst + r * St::kGradRow, static_cast<const G*>(a.g) + row, St::kGradRow, bar, pol);
                bulk_load_hint(dst + St::kZOff + r * St::kZRow, a.zbuf + row, St::kZRow, bar, pol);
            }
            if (b == 0) bulk_load(dst + St::kMOff, a.m + e0, 256 * 4, bar);
        };

        int64_t k = g0 / pt.CG;
        const int64_t kfirst = k;
        float sp[W];
        Sum2 acc[W];
#pragma unroll
        for (int w = 0; w < W; ++w) {
            sp[w] = __ldg(a.s_prev + (int64_t)w * pt.nchunks + k);
            acc[w].s = 0.0f;
            acc[w].e = 0.0f;
        }
        if (lane == 0)
            for (int64_t it = 0; it < S && it < items; ++it) issue((int)it, it);

        for (int64_t i = 0; i < count; ++i) {
            const int64_t gi = g0 + wir + i * wpr;
            const int64_t kg = fast_div((uint32_t)gi, a.cg_div);
            if (kg != k) {
                // this warp's part of chunks k .. kg-1 is done (possibly empty)
                while (k < kg) {
                    if constexpr (bcomb) flush_chunk_block<W>(pt, q, wpb, wib, k, kfirst, acc, bpart, bcnt, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
                    else flush_chunk<W, kFlushTailCall, !INTER>(pt, q, wpr, wir, k, kfirst, g0, g1, acc, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
                    ++k;
                }
#pragma unroll
                for (int w = 0; w < W; ++w) sp[w] = __ldg(a.s_prev + (int64_t)w * pt.nchunks + k);
            }
            const int64_t e0 = gi * 256 + lane * 8;
            float bm[8];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const int64_t it = i * NB + b;
                const int s = (int)(it % S);
                const bool landed = __all_sync(kFull, mbar_wait(bar0 + 8u * s, (phase >> s) & 1u));
                if (!landed) {
                    // record the failure, let every copy still in flight land, and stop
                    if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
                    for (int64_t t = it; t < items && t < it + S; ++t) {
                        const int st = (int)(t % S);
                        mbar_wait(bar0 + 8u * st, (phase >> st) & 1u);
                    }
                    return;
                }
                phase ^= 1u << s;
                const unsigned char* stg = stage0 + (size_t)s * St::kBytes;
                if (b == 0) {
                    ld8_shared<float>(stg + St::kMOff, lane, bm);
#pragma unroll
                    for (int j = 0; j < 8; ++j) bm[j] = __fmul_rn(a.b1, bm[j]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int w = b * R + r;
                    if (w < W) {
                        float gv[8], zv[8];
                        ld8_shared<G>(stg + r * St::kGradRow, lane, gv);
                        ld8_shared<float>(stg + St::kZOff + r * St::kZRow, lane, zv);
                        uint32_t byte = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float e = __fsub_rn(zv[j], signed_scale(sp[w], zv[j] >= 0.0f));
                            const float p = __fadd_rn(bm[j], __fmul_rn(a.c1, gv[j]));
                            const float z = __fadd_rn(p, e);
                            zv[j] = z;
                            byte |= (z >= 0.0f ? 1u : 0u) << j;
                            sum2_add_sq(acc[w], z);
                        }
                        st8_stream(a.zbuf + (int64_t)w * a.n + e0, zv);
                        const uint32_t word = quad_word(byte, lane);
                        if ((lane & 3) == 0) __stcs(a.wbits + (int64_t)w * words_per_row + gi * 8 + (lane >> 2), word);
                    }
                }
                __syncwarp();               // every lane is done with stage s
                if (lane == 0 && it + S < items) issue(s, it + S);
            }
        }
        for (;;) {
            if constexpr (bcomb) flush_chunk_block<W>(pt, q, wpb, wib, k, kfirst, acc, bpart, bcnt, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
            else flush_chunk<W, kFlushTailCall, !INTER>(pt, q, wpr, wir, k, kfirst, g0, g1, acc, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
            if (k == klast) break;
            ++k;
        }
    }
}

// Launch shape for (W, gradient type): warps per block and stages per warp chosen so that
// the stages fill the shared memory of one block (one block per SM): at least two stages
// per warp, up to sixteen warps, and as many stages as then fit (at most eight), after
// the block-level partials of the interleaved kernels that pre-combine.
template <int W, typename G>
WorkerConfig config_w(int smem_budget)
{
    using St = WorkerStage<W, G>;
    auto fit = [&](uint32_t reserve) {
        WorkerConfig c{};
        const int per = (int)St::kBytes + 8;                 // a stage and its mbarrier
        const int usable = smem_budget - (int)reserve - 128;
        int warps = usable / (2 * per);
        warps = warps > kMaxWarps ? kMaxWarps : (warps < 1 ? 1 : warps);
        int stages = usable / (warps * per);
        stages = stages > kMaxStages ? kMaxStages : (stages < 2 ? 2 : stages);
        c.warps_per_block = warps;
        c.stages = stages;
        c.stage_bytes = St::kBytes;
        c.bars_off = reserve;
        c.stages_off = (reserve + 8u * (uint32_t)(warps * stages) + 127u) & ~127u;
        c.smem_bytes = c.stages_off + (size_t)warps * stages * St::kBytes;
        return c;
    };
    if (!block_combine_fits<W, G>()) return fit(0);
    WorkerConfig c = fit(block_part_bytes<W>() + 16u);
    c.block_combine = 1;
    c.bcnt_off = block_part_bytes<W>();
    return c;
}

template <int W, typename G>
cudaError_t launch_wg(const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget)
{
    const WorkerConfig c = config_w<W, G>(smem_budget);
    if ((int)c.smem_bytes > smem_budget) return cudaErrorInvalidConfiguration;
    WorkerArgs b = a;
    b.stages = c.stages;
    b.bars_off = c.bars_off;
    b.stages_off = c.stages_off;
    b.bcnt_off = c.bcnt_off;
    // the block-level partial slots of the interleaved kernel assume one range per block
    if (a.interleave && c.block_combine && a.pt.P > grid) return cudaErrorInvalidConfiguration;
    if (a.interleave) return launch_pdl(k_worker<W, G, true>, grid, c.warps_per_block * 32, c.smem_bytes, s, b);
    return launch_pdl(k_worker<W, G, false>, grid, c.warps_per_block * 32, c.smem_bytes, s, b);
}

// The shared-memory opt-in of the worker kernels for W, on the current device. It is a
// property of the kernel in the current device's context, so it is set for every context
// (see prepare_worker), not once per process.
template <int W, typename G>
cudaError_t prepare_wg(int smem_budget)
{
    const WorkerConfig c = config_w<W, G>(smem_budget);
    if ((int)c.smem_bytes > smem_budget) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(k_worker<W, G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c.smem_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_worker<W, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)c.smem_bytes);
    return e;
}

#define OB_FOR_EACH_W(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14) X(15) X(16)

// The per-type entry points, defined in the instantiating files.
cudaError_t launch_worker_f32(int W, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget);
cudaError_t launch_worker_f16(int W, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget);
cudaError_t launch_worker_bf16(int W, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget);
cudaError_t prepare_worker_f32(int W, int smem_budget);
cudaError_t prepare_worker_f16(int W, int smem_budget);
cudaError_t prepare_worker_bf16(int W, int smem_budget);
WorkerConfig worker_config_f32(int W, int smem_budget);
WorkerConfig worker_config_f16(int W, int smem_budget);
WorkerConfig worker_config_bf16(int W, int smem_budget);

}  // namespace ob
