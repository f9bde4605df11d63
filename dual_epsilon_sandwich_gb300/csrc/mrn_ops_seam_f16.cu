// mrn_ops_seam_f16.cu -- kernel instantiations and launcher for the split-norm
// seam with a binary16 publication format: the fused form
// y = f16(f16(x * inv) * gamma) and the weightless first half u = f16(x * inv).
// One translation unit per format so the library builds in parallel.
#include "mrn_kernels.cuh"

namespace mrn {

cudaError_t launch_seam_f16(int op, bool bf16, const Geometry &g, const KernelArgs &a,
                            int64_t rows, cudaStream_t stream, uint64_t *launches) {
    if (op == kSeamF16) return launch_op<kSeamF16>(bf16, g, a, rows, stream, launches);
    if (op == kUnweightedF16)
        return launch_op<kUnweightedF16>(bf16, g, a, rows, stream, launches);
    return cudaErrorInvalidValue;
}

int take_wait_timeouts_seam_f16() { return take_wait_timeouts<kSeamF16>(); }

}  // namespace mrn
