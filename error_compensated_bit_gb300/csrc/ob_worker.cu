// Dispatch of the worker kernels by gradient type (the kernels are in ob_worker.cuh,
// instantiated in ob_worker_f32.cu, ob_worker_f16.cu, ob_worker_bf16.cu), and the
// self-test of the bounded pipeline wait.
#include "ob_worker.cuh"

namespace ob {

// Self-test of the failure path: one warp waits, with the given limit, on an mbarrier that
// expects one arrival and never gets it; the wait runs out and the warp records the same
// status the pipelines record. No copy is in flight, so returning is safe.
__global__ void __launch_bounds__(32, 1) k_wait_probe(unsigned* status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const bool landed = __all_sync(kFull, mbar_wait_for(b, 0u, limit_ns));
    if (!landed && threadIdx.x == 0) atomicOr(status, kStatusWaitTimeout);
}

cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s)
{
    k_wait_probe<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_worker(int W, int dtype, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget)
{
    if (dtype == 0) return launch_worker_f32(W, a, grid, s, smem_budget);
    if (dtype == 1) return launch_worker_f16(W, a, grid, s, smem_budget);
    return launch_worker_bf16(W, a, grid, s, smem_budget);
}

cudaError_t prepare_worker(int W, int smem_budget)
{
    cudaError_t e = prepare_worker_f32(W, smem_budget);
    if (e == cudaSuccess) e = prepare_worker_f16(W, smem_budget);
    if (e == cudaSuccess) e = prepare_worker_bf16(W, smem_budget);
    return e;
}

WorkerConfig worker_config(int W, int dtype, int smem_budget)
{
    if (dtype == 0) return worker_config_f32(W, smem_budget);
    if (dtype == 1) return worker_config_f16(W, smem_budget);
    return worker_config_bf16(W, smem_budget);
}

}  // namespace ob
