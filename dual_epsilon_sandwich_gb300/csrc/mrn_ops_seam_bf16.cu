// mrn_ops_seam_bf16.cu -- kernel instantiations and launcher for the split-norm
// seam with a bf16 publication format: the fused form
// y = bf16(bf16(x * inv) * gamma) and the weightless first half u = bf16(x * inv).
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_seam_bf16(int op, bool bf16, const Geometry &g, const KernelArgs &a,
                             int64_t rows, cudaStream_t stream, uint64_t *launches) {
    if (op == kSeamBF16) return launch_op<kSeamBF16>(bf16, g, a, rows, stream, launches);
    if (op == kUnweightedBF16)
        return launch_op<kUnweightedBF16>(bf16, g, a, rows, stream, launches);
    return cudaErrorInvalidValue;
}

int take_wait_timeouts_seam_bf16() { return take_wait_timeouts<kSeamBF16>(); }

}  // namespace mrn
