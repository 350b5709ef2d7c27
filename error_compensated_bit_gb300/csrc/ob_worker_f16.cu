// Worker kernels for __half gradients (all W, both range modes); see ob_worker.cuh.
#include "ob_worker.cuh"

namespace ob {

cudaError_t launch_worker_f16(int W, const WorkerArgs& a, int grid, cudaStream_t s, int smem_budget)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return launch_wg<w, __half>(a, grid, s, smem_budget);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t prepare_worker_f16(int W, int smem_budget)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return prepare_wg<w, __half>(smem_budget);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return cudaErrorInvalidValue;
}

WorkerConfig worker_config_f16(int W, int smem_budget)
{
    switch (W) {
#define OB_CASE(w) \
    case w:        \
        return config_w<w, __half>(smem_budget);
        OB_FOR_EACH_W(OB_CASE)
#undef OB_CASE
    }
    return WorkerConfig{};
}

}  // namespace ob
