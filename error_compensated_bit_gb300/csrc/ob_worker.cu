// Worker side of the compression-stage step: momentum, error compensation, chunk RMS
// scale, sign packing and residual, fused in one pass over the W gradient rows.
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
#include "ob_common.cuh"

namespace ob {

template <int W, typename G>
__global__ void __launch_bounds__(kBlock) k_worker(WorkerArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const Part pt = a.pt;
    const int64_t words_per_row = a.n / 32;

    for (int64_t q = warp; q < pt.P; q += nwarps) {
        const int64_t g0 = range_begin(pt, q);
        const int64_t g1 = range_begin(pt, q + 1);
        int64_t k = g0 / pt.CG;
        const int64_t kfirst = k;
        int64_t kend = (k + 1) * pt.CG;

        float sp[W];
        Sum2 acc[W];
#pragma unroll
        for (int w = 0; w < W; ++w) {
            sp[w] = __ldg(a.s_prev + (int64_t)w * pt.nchunks + k);
            acc[w].s = 0.0f;
            acc[w].e = 0.0f;
        }

        for (int64_t gi = g0; gi < g1; ++gi) {
            if (gi == kend) {
                flush_chunk<W>(pt, q, k, kfirst, acc, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
                ++k;
                kend += pt.CG;
#pragma unroll
                for (int w = 0; w < W; ++w) sp[w] = __ldg(a.s_prev + (int64_t)w * pt.nchunks + k);
            }
            const int64_t e0 = gi * 256 + lane * 8;
            float bm[8];
            ld8_stream(a.m + e0, bm);
#pragma unroll
            for (int j = 0; j < 8; ++j) bm[j] = __fmul_rn(a.b1, bm[j]);

#pragma unroll
            for (int w = 0; w < W; ++w) {
                const int64_t row = (int64_t)w * a.n + e0;
                float gv[8], zv[8];
                Grad<G>::ld8(a.g, row, gv);
                ld8_stream(a.zbuf + row, zv);
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
                st8_stream(a.zbuf + row, zv);
                const uint32_t word = quad_word(byte, lane);
                if ((lane & 3) == 0) __stcs(a.wbits + (int64_t)w * words_per_row + gi * 8 + (lane >> 2), word);
            }
        }
        flush_chunk<W>(pt, q, k, kfirst, acc, a.part, a.cnt, a.s_next, a.C, a.zbuf, a.n, lane);
    }
}

template <int W>
static cudaError_t launch_w(int dtype, const WorkerArgs& a, int grid, cudaStream_t s)
{
    if (dtype == 0) k_worker<W, float><<<grid, kBlock, 0, s>>>(a);
    else if (dtype == 1) k_worker<W, __half><<<grid, kBlock, 0, s>>>(a);
    else k_worker<W, __nv_bfloat16><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

template <int W>
static int occ_w(int dtype)
{
    int blocks = 0;
    cudaError_t e;
    if (dtype == 0) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_worker<W, float>, kBlock, 0);
    else if (dtype == 1) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_worker<W, __half>, kBlock, 0);
    else e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_worker<W, __nv_bfloat16>, kBlock, 0);
    return e == cudaSuccess ? blocks : 0;
}

#define OB_FOR_EACH_W(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14) X(15) X(16)

cudaError_t launch_worker(int W, int dtype, const WorkerArgs& a, int grid, cudaStream_t s)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return launch_w<w>(dtype, a, grid, s);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return cudaErrorInvalidValue;
}

int occupancy_worker(int W, int dtype)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return occ_w<w>(dtype);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return 0;
}

}  // namespace ob
