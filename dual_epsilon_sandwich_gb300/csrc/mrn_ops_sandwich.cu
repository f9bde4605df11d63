// mrn_ops_sandwich.cu -- kernel instantiations and launcher for the dual-epsilon sandwich tail.
// One translation unit per operation so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_sandwich(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                            cudaStream_t stream, uint64_t *launches) {
    return launch_op<kSandwich>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_sandwich() { return take_wait_timeouts<kSandwich>(); }

}  // namespace mrn
