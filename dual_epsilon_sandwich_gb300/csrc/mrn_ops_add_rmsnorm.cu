// mrn_ops_add_rmsnorm.cu -- kernel instantiations and launcher for
// the residual add then RMSNorm.
// One translation unit per operation so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_add_rmsnorm(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                               cudaStream_t stream, uint64_t *launches) {
    return launch_op<kAddRmsnorm>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_add_rmsnorm() { return take_wait_timeouts<kAddRmsnorm>(); }

}  // namespace mrn
