// mrn_ops_rmsnorm_q8_1.cu -- kernel instantiations and launcher for
// RMSNorm fused with Q8_1 block quantisation.
// One translation unit per operation so the library builds in parallel.
#include "mrn_q8_kernels.cuh"

namespace mrn {

cudaError_t launch_rmsnorm_q8_1(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                                cudaStream_t stream, uint64_t *launches) {
    if (g.kind == kQ8Blocks && g.stages > 0) {
        return bf16 ? launch_q8_tma<BF16>(g, a, rows, stream, launches)
                    : launch_q8_tma<F32>(g, a, rows, stream, launches);
    }
    if (g.kind == kQ8Blocks) {
        return bf16 ? launch_q8_blocks<BF16>(g, a, rows, stream, launches)
                    : launch_q8_blocks<F32>(g, a, rows, stream, launches);
    }
    return launch_op<kRmsnormQ8>(bf16, g, a, rows, stream, launches);
}

int take_wait_timeouts_rmsnorm_q8_1() { return take_wait_timeouts<kRmsnormQ8>(); }

}  // namespace mrn
