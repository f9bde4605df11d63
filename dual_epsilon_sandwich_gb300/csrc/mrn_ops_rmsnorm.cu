// mrn_ops_rmsnorm.cu -- kernel instantiations and launcher for the RMSNorm.
// One translation unit per operation so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_rmsnorm(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                           cudaStream_t stream, uint64_t *launches) {
    return launch_op<kRmsnorm>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_rmsnorm() { return take_wait_timeouts<kRmsnorm>(); }

}  // namespace mrn
