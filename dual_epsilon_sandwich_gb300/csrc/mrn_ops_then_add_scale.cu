// mrn_ops_then_add_scale.cu -- kernel instantiations and launcher for
// the post norm, residual add and broadcast scale.
// One translation unit per operation so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_then_add_scale(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                                  cudaStream_t stream, uint64_t *launches) {
    return launch_op<kThenAddScale>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_then_add_scale() { return take_wait_timeouts<kThenAddScale>(); }

}  // namespace mrn
