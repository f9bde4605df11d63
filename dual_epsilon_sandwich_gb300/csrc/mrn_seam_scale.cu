// mrn_seam_scale.cu -- the split route's second operation at the norm seam
// ("Chapter 12 -- RMSNorm and the dual-epsilon sandwich", section 12.7: the
// learned-weight multiply applied as a separate operation in the publication
// format): y[r,j] = S(u[r,j] * gamma[j]) over 16-bit values of S.
//
// Element-wise and HBM-bound: each thread owns one column vector (gamma read
// once per thread) and walks the rows r = blockIdx.y, + gridDim.y, ...,
// kScaleUnroll rows per step so that several 16-byte loads are in flight.
#include "mrn_kernels.cuh"

namespace mrn {

constexpr int kScaleThreads = 256;
constexpr int kScaleUnroll = 4;
constexpr int kScaleCtasPerSm = 8;
constexpr int kMaxGridY = 65535;

template <bool BF, int VEC>
__global__ void __launch_bounds__(kScaleThreads)
mrn_seam_scale_kernel(const void *u, const void *gamma, void *y, int64_t rows, int64_t n,
                      int64_t nvec) {
    pdl_enter();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= nvec) return;
    H16<VEC> g;
    ld_h16(g, static_cast<const char *>(gamma) + c * VEC * 2);
    const int64_t step = gridDim.y;
    for (int64_t r0 = blockIdx.y; r0 < rows; r0 += step * kScaleUnroll) {
        H16<VEC> v[kScaleUnroll];
#pragma unroll
        for (int i = 0; i < kScaleUnroll; ++i) {
            const int64_t r = r0 + i * step;
            if (r < rows) ld_stream_h16(v[i], static_cast<const char *>(u) + (r * n + c * VEC) * 2);
        }
#pragma unroll
        for (int i = 0; i < kScaleUnroll; ++i) {
            const int64_t r = r0 + i * step;
            if (r < rows)
                st_h16(static_cast<char *>(y) + (r * n + c * VEC) * 2, seam_scale_frag<BF, VEC>(v[i], g));
        }
    }
}

template <bool BF, int VEC>
cudaError_t launch_scale_typed(const void *u, const void *gamma, void *y, int64_t rows, int64_t n,
                               int sms, bool pdl, cudaStream_t stream, uint64_t *launches) {
    const int64_t nvec = n / VEC;
    const int64_t threads = nvec < kScaleThreads ? ((nvec + 31) / 32) * 32 : kScaleThreads;
    const int64_t gx = (nvec + threads - 1) / threads;
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    int64_t gy = static_cast<int64_t>(sms) * kScaleCtasPerSm / gx;
    gy = gy < 1 ? 1 : gy;
    gy = gy > rows ? rows : gy;
    gy = gy > kMaxGridY ? kMaxGridY : gy;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.stream = stream;
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, mrn_seam_scale_kernel<BF, VEC>, u, gamma, y, rows, n, nvec);
    if (err == cudaSuccess) ++*launches;
    return err;
}

cudaError_t launch_seam_scale(bool seam_bf16, const void *u, const void *gamma, void *y,
                              int64_t rows, int64_t n, int vec, int sms, bool pdl,
                              cudaStream_t stream, uint64_t *launches) {
    if (vec == 8) {
        return seam_bf16 ? launch_scale_typed<true, 8>(u, gamma, y, rows, n, sms, pdl, stream, launches)
                         : launch_scale_typed<false, 8>(u, gamma, y, rows, n, sms, pdl, stream, launches);
    }
    return seam_bf16 ? launch_scale_typed<true, 1>(u, gamma, y, rows, n, sms, pdl, stream, launches)
                     : launch_scale_typed<false, 1>(u, gamma, y, rows, n, sms, pdl, stream, launches);
}

}  // namespace mrn
