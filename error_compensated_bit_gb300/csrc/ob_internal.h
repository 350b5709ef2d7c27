// Internal launch interface between the C ABI (ob_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace ob {

// Division by a run-time constant for 32-bit operands, by a precomputed multiplier -- the
// unsigned division by an invariant integer of T. Granlund and P. L. Montgomery, "Division
// by Invariant Integers using Multiplication" (PLDI 1994):
// n / d == (t + ((n - t) >> 1)) >> (l - 1) with t = high 32 bits of n * m,
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1 (d >= 2; d == 1 is passed through).
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f{d, 0u, 0u};
    if (d > 1) {
        uint32_t l = 0;
        while ((1ull << l) < d) ++l;
        f.l = l;
        f.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    }
    return f;
}

// Partition of the buffer into 256-element groups and P contiguous warp ranges.
struct Part {
    int64_t NG;       // groups (n / 256)
    int64_t P;        // ranges (one warp each), 1 <= P <= NG
    int64_t CG;       // groups per chunk (chunk / 256)
    int64_t J;        // partial slots per range (most chunks one range touches)
    int64_t nchunks;  // n / chunk
};

struct WorkerArgs {
    const void* g;          // [W][n] gradients
    const float* m;         // [n] momentum of the previous step
    float* zbuf;            // [W][n] in: previous z, out: this step's z
    uint32_t* wbits;        // [W][n/32]
    const float* s_prev;    // [W][nchunks] scales of the previous step
    float* s_next;          // [W][nchunks] scales of this step (written by the last contributor)
    double* part;           // [W][P][warps per range][J] partial sums of squares
    unsigned* cnt;          // [nchunks] arrival counters (zero between launches)
    unsigned* status;       // status word (0 = fine; see ob_tma.cuh)
    FastDiv cg_div;         // division by the groups per chunk
    Part pt;
    int64_t n, C;
    float b1, c1;
    int stages;             // pipeline stages per warp (set by the launcher)
    int interleave;         // 1: one range per block, warps interleaved; 0: one range per warp
    uint32_t bars_off, stages_off, bcnt_off;   // dynamic shared-memory layout (set by the launcher)
};

// Launch shape of the worker kernel for one (W, gradient type).
struct WorkerConfig {
    int warps_per_block;
    int stages;
    size_t smem_bytes;
    uint32_t stage_bytes;
    int block_combine;      // room for the block-level partials without fewer warps or stages
    uint32_t bars_off, stages_off, bcnt_off;
};

struct ServerArgs {
    const uint32_t* wbits;  // [W][n/32]
    const float* s_next;    // [W][nchunks]
    float* ybuf;            // [n] in: previous y, out: this step's y
    uint32_t* sbits;        // [n/32]
    const float* t_prev;    // [nchunks]
    float* t_next;          // [nchunks]
    double* part;           // [P][J]
    unsigned* cnt;          // [nchunks]
    Part pt;
    int64_t n, C;
};

struct UpdateArgs {
    const uint32_t* sbits;     // [n/32]
    const float* t_next;       // [nchunks]
    const uint32_t* maskbits;  // [n/32] or null
    const float* v;            // [n] frozen variance
    float* x;                  // [n]
    float* m;                  // [n] out
    float* s_prev;             // [W][nchunks] <- s_next (no reader of s_prev runs in this step's update)
    const float* s_next;
    float* t_prev;             // [nchunks] <- t_next
    int64_t NG, CG;
    int64_t nscales_w, nchunks; // scales to move (W*nchunks and nchunks, or 0 when k_scales moves them)
    FastDiv cg_div;            // division by the groups per chunk
    float lr, eps, wd;
};

struct WarmupArgs {
    const void* g;  // [W][n]
    float* x;
    float* m;
    float* v;
    int64_t n;
    int W;
    float b1, c1, b2, c2, eps, lr, wd, bc1, bc2;
    int corrected;
};

struct MaskArgs {
    const float* mask01;  // [n]
    uint32_t* bits;       // [n/32]
    int64_t n;
};

struct ExportArgs {
    const float* zbuf;     // [W][n]
    const float* ybuf;     // [n]
    const float* s_prev;   // [W][nchunks]
    const float* t_prev;   // [nchunks]
    float* ew_out;         // [W][n]
    float* es_out;         // [n]
    int64_t n, C, nchunks;
    int W;
};

struct LocoArgs {
    const void* g;         // [W][n]
    float* err;            // [W][n] moving average of compensation errors
    uint8_t* codes;        // [W][n*bits/8]
    float* scale;          // [W][nchunks]
    unsigned* amax_bits;   // [W][nchunks] running absmax as float bits (pass 1)
    float* x;
    float* m;
    float* v;
    int64_t n, C, nchunks, NG;
    FastDiv ng_div, cg_div;    // division by the groups per row / per chunk
    int W, bits;
    int keep_codes;        // long chunks: also store the codes (they are otherwise kept in registers)
    float ratio, beta, keep, b1, c1, b2, c2, eps, lr, wd;
};

// Launchers (return the launch status). `grid` blocks of kBlock threads.
constexpr int kBlock = 256;
cudaError_t launch_worker(int W, int dtype, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget);
WorkerConfig worker_config(int W, int dtype, int smem_budget);
// Opt the worker / server kernels for W into their dynamic shared memory on the current
// device (a property of the kernel in that device's context).
cudaError_t prepare_worker(int W, int smem_budget);
cudaError_t prepare_server(int W);
cudaError_t prepare_loco();
cudaError_t launch_server(int W, const ServerArgs& a, int grid, cudaStream_t s);
cudaError_t launch_update(const UpdateArgs& a, int grid, cudaStream_t s);
cudaError_t launch_scales(const UpdateArgs& a, int grid, cudaStream_t s);
cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_warmup(int dtype, const WarmupArgs& a, int grid, cudaStream_t s);
cudaError_t launch_mask(const MaskArgs& a, int grid, cudaStream_t s);
cudaError_t launch_export(const ExportArgs& a, int grid, cudaStream_t s);
cudaError_t launch_loco_absmax(int dtype, const LocoArgs& a, int grid, cudaStream_t s);
cudaError_t launch_loco_server(const LocoArgs& a, int grid, cudaStream_t s);
cudaError_t launch_loco_qs(int dtype, const LocoArgs& a, int grid, cudaStream_t s);
cudaError_t launch_loco_fused(int dtype, const LocoArgs& a, int grid, cudaStream_t s);

// Resident blocks per SM of the server kernel for W / of the update kernel; 0 on error.
int occupancy_server(int W);
int occupancy_update();
int occupancy_loco_absmax(int dtype);
int occupancy_loco_qs(int dtype, int bits, int W);
int occupancy_loco_fused(int dtype, int bits, int64_t C);

// Launch `kernel` with the programmatic stream-serialization attribute (see pdl_wait in
// ob_tma.cuh): it may begin while the previous kernel on the stream finishes.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), int grid, int block, size_t smem, cudaStream_t s,
                              Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ob
