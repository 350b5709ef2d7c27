// Full-precision warm-up step: the W gradients are averaged (the full-precision
// AllReduce of the warm-up phase) and plain Adam updates m, v and x.
//
// Method: DeepSpeed 1-bit Adam training guide, §3.1 (freeze_step: full-precision Adam
// until the variance is estimated) and §4 (phase one, standard Adam on exp_avg and
// exp_avg_sq); "1-bit Adam" review, "Proposed method" (Adam warm-up).
//
// Per element, single float32 operations in this order:
//   acc = 0; acc = acc + g_w (w ascending); gbar = acc / W
//   m = b1*m + c1*gbar;  v = b2*v + c2*(gbar*gbar)
//   [mh = m / bc1; vh = v / bc2 when bias correction is on]
//   x = x - lr*(mh/(sqrt(vh)+eps) [+ wd*x])
// Memory per element: W*(grad bytes) + 24 (m, v, x read and written).
#include "ob_common.cuh"
#include "ob_div.cuh"

namespace ob {

template <typename G>
__global__ void __launch_bounds__(kBlock) k_warmup(WarmupArgs a)
{
    const int64_t nvec = a.n / 8;
    const float fW = (float)a.W;
    for (int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i8 < nvec;
         i8 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e0 = i8 * 8;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll 4
        for (int w = 0; w < a.W; ++w) {
            float gv[8];
            Grad<G>::ld8(a.g, (int64_t)w * a.n + e0, gv);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], gv[j]);
        }
        float mv[8], vv[8], xv[8];
        ld8_stream(a.m + e0, mv);
        ld8_stream(a.v + e0, vv);
        ld8_stream(a.x + e0, xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float gbar = div_rn_zero_fast(acc[j], fW);
            mv[j] = __fadd_rn(__fmul_rn(a.b1, mv[j]), __fmul_rn(a.c1, gbar));
            vv[j] = __fadd_rn(__fmul_rn(a.b2, vv[j]), __fmul_rn(a.c2, __fmul_rn(gbar, gbar)));
            float mh = mv[j], vh = vv[j];
            if (a.corrected) {
                mh = div_rn_zero_fast(mh, a.bc1);
                vh = div_rn_zero_fast(vh, a.bc2);
            }
            const float denom = __fadd_rn(__fsqrt_rn(vh), a.eps);
            float u = div_rn_zero_fast(mh, denom);
            if (a.wd != 0.0f) u = __fadd_rn(u, __fmul_rn(a.wd, xv[j]));
            xv[j] = __fsub_rn(xv[j], __fmul_rn(a.lr, u));
        }
        st8_stream(a.m + e0, mv);
        st8_stream(a.v + e0, vv);
        st8_stream(a.x + e0, xv);
    }
}

cudaError_t launch_warmup(int dtype, const WarmupArgs& a, int grid, cudaStream_t s)
{
    if (dtype == 0) k_warmup<float><<<grid, kBlock, 0, s>>>(a);
    else if (dtype == 1) k_warmup<__half><<<grid, kBlock, 0, s>>>(a);
    else k_warmup<__nv_bfloat16><<<grid, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ob
