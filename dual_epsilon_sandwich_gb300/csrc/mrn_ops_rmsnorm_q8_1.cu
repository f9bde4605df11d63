// mrn_ops_rmsnorm_q8_1.cu -- kernel instantiations and launcher for
// RMSNorm fused with Q8_1 block quantisation.
// One translation unit per operation so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_rmsnorm_q8_1(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                                cudaStream_t stream, uint64_t *launches) {
    return launch_op<kRmsnormQ8>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_rmsnorm_q8_1() { return take_wait_timeouts<kRmsnormQ8>(); }

}  // namespace mrn
