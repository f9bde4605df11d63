// mrn_internal.h -- host-side interface between the C ABI layer (mrn_api.cpp)
// and the kernel launchers (mrn_ops_*.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

// Helpers used both by the host layer and inside kernels.
#if defined(__CUDACC__)
#define MRN_HOST_DEVICE __host__ __device__
#else
#define MRN_HOST_DEVICE
#endif

namespace mrn {

enum Op : int {
    kRmsnorm = 0,
    kThenAdd = 1,
    kSandwich = 2,
    kAddRmsnorm = 3,
    kThenAddScale = 4,
    kRmsnormQ8 = 5,   // RMSNorm then Q8_1 blocks: 32 codes + (f16 d, f16 s) per 36 bytes
    // Split-norm seam: the weightless norm rounded to a 16-bit format S, and
    // (the weighted forms) the weight multiply as a second S operation.
    kSeamF16 = 6,          // y = f16(f16(x * inv) * gamma), gamma in f16
    kSeamBF16 = 7,         // the same with S = bf16
    kUnweightedF16 = 8,    // u = f16(x * inv): the split route's first operation
    kUnweightedBF16 = 9,   // the same with S = bf16
};
constexpr int kQ8Block = 32;        // elements per Q8_1 block
constexpr int kQ8BlockBytes = 36;   // f16 d, f16 s, int8 q[32]

// The seam operations (their output and gamma are 16-bit values of S).
MRN_HOST_DEVICE constexpr bool op_is_seam(int op) { return op >= kSeamF16 && op <= kUnweightedBF16; }
MRN_HOST_DEVICE constexpr bool op_seam_bf16(int op) { return op == kSeamBF16 || op == kUnweightedBF16; }
MRN_HOST_DEVICE constexpr bool op_seam_weighted(int op) { return op == kSeamF16 || op == kSeamBF16; }

// Row operands each operation reads, and the gamma vectors it uses.
MRN_HOST_DEVICE constexpr int op_row_inputs(int op) {
    return (op == kRmsnorm || op == kRmsnormQ8 || op_is_seam(op)) ? 1 : 2;
}
MRN_HOST_DEVICE constexpr int op_gammas(int op) {
    return op == kSandwich ? 2 : (op == kUnweightedF16 || op == kUnweightedBF16) ? 0 : 1;
}
// Gammas the staged (kTma) kernel copies into shared memory: the seam's
// 16-bit gamma is read through L1 instead (its rows need not be a multiple
// of 16 bytes when x is f32).
MRN_HOST_DEVICE constexpr int op_staged_gammas(int op) { return op_is_seam(op) ? 0 : op_gammas(op); }
enum Kind : int { kAuto = 0, kRowsPerWarp = 1, kCta = 2, kStream = 3, kTma = 4, kQ8Blocks = 5 };

// Launch-time view of one call.  Pointers are device pointers; row operands
// are [rows x n] row-major.  For the sandwich, x = block_out, res = residual,
// g1 = gamma_post, g2 = gamma_pre, y = out_stream, y2 = normed.  For the
// residual add + norm, x = a, res = b, y = residual_out, y2 = normed.  For
// then-add-scale, scale points at the one broadcast element.  For Q8_1, y
// points at the output blocks.  For the seam operations, y is the 16-bit
// output (u or y of the seam) and g1 the 16-bit gamma of the weighted forms.
struct KernelArgs {
    const void *x;
    const void *res;
    const void *g1;
    const void *g2;
    const void *scale;
    void *y;
    void *y2;
    int64_t n;         // elements per row
    int64_t nvec;      // loads per row = ceil(n / vec)
    int64_t row0;      // first row of this launch
    int64_t rows_end;  // one past the last row of this launch
    float eps1;        // eps (rmsnorm, then-add) or eps_post (sandwich)
    float eps2;        // eps_pre (sandwich)
    uint32_t stall_bytes;   // test hook: bytes a CTA's first wait expects beyond its
                            // copies or messages (0 in use; see MRN_LAUNCH_TEST_WAIT_TIMEOUT)
    uint32_t stage_bytes;   // staged kernel, rows not 16-byte aligned (Geometry::edge):
                            // bytes between its shared-memory slots (edge_stage_bytes)
};

struct Geometry {
    int kind;          // Kind
    int vec;           // elements per load
    int k;             // loads per operand per thread
    int threads;       // threads per CTA
    int cluster;       // CTAs per row (kCta)
    int lanes;         // threads per row (kRowsPerWarp)
    int rows_per_cta;
    int stages;        // shared-memory row stages (kTma)
    int ctas;          // CTAs launched (kTma: persistent grid), 0 = from rows
    int groups;        // warp groups per CTA (kTma), each on its own rows
    int pdl;           // launch with programmatic stream serialisation
    int edge;          // kTma: rows not 16-byte aligned, staged as the 16-byte granules
                       // that cover them (every row operand at the same offset)
};

// Register-slot limits per thread count: the kernels are compiled with these
// launch bounds so that every (k, threads <= max) pair can launch.
constexpr int kMaxK = 8;
constexpr int kWarpKernelThreads = 256;     // rows-per-warp kernel: at most (launch bounds)
constexpr int kWarpKernelCtaThreads = 128;  // ... and the automatic choice
constexpr int kStreamMaxThreads = 512;
constexpr int kMaxCluster = 16;
constexpr int kTmaMaxStages = 8;
constexpr int kSharedBytesPerCta = 232448;    // 227 KB opt-in limit on sm_100 / sm_103
constexpr int cta_max_threads(int k) { return k <= 2 ? 1024 : (k <= 4 ? 512 : 256); }
// Staged kernel: threads per warp group, and per CTA for 1 or 2 groups.
constexpr int kTmaMaxGroups = 2;
// RMSNorm + Q8_1 with whole blocks per thread (kQ8Blocks): k = 1 or 2 blocks
// per thread, at most this many threads per CTA (one row per CTA); with
// stages > 0 the staged form: 1 or 2 warp groups of at most
// kQ8TmaGroupThreads threads, persistent CTAs.
constexpr int kQ8BlockMaxThreads = 512;
constexpr int kQ8BlockMaxK = 2;
constexpr int kQ8TmaGroupThreads = 256;
// A row's Q8_1 blocks in shared memory, rounded up to 16 bytes.
MRN_HOST_DEVICE constexpr int64_t q8_out_stride(int64_t blocks) {
    return (blocks * 36 + 15) / 16 * 16;
}
// Dynamic shared memory of the staged Q8_1 kernel: gamma and `stages` rows of
// x, plus one block buffer per group.
MRN_HOST_DEVICE constexpr int64_t q8_tma_shared_bytes(int64_t n, int elem_bytes, int stages,
                                                      int groups) {
    return n * elem_bytes * (1 + stages) + groups * q8_out_stride(n / 32);
}
constexpr int tma_group_max_threads(int k) { return k <= 2 ? 512 : (k <= 4 ? 416 : 256); }
constexpr int tma_max_threads(int k, int groups) {
    return groups == 1 ? cta_max_threads(k) : groups * tma_group_max_threads(k);
}

// One launcher per operation; each returns the CUDA error of the launch(es).
cudaError_t launch_rmsnorm(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                           cudaStream_t stream, uint64_t *launches);
cudaError_t launch_then_add(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                            cudaStream_t stream, uint64_t *launches);
cudaError_t launch_sandwich(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                            cudaStream_t stream, uint64_t *launches);
cudaError_t launch_add_rmsnorm(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                               cudaStream_t stream, uint64_t *launches);
cudaError_t launch_then_add_scale(bool bf16, const Geometry &g, const KernelArgs &a,
                                  int64_t rows, cudaStream_t stream, uint64_t *launches);
cudaError_t launch_rmsnorm_q8_1(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                                cudaStream_t stream, uint64_t *launches);
// The seam operations: op is kSeamF16 or kUnweightedF16 (f16 launcher),
// kSeamBF16 or kUnweightedBF16 (bf16 launcher); bf16 is the input dtype.
cudaError_t launch_seam_f16(int op, bool bf16, const Geometry &g, const KernelArgs &a,
                            int64_t rows, cudaStream_t stream, uint64_t *launches);
cudaError_t launch_seam_bf16(int op, bool bf16, const Geometry &g, const KernelArgs &a,
                             int64_t rows, cudaStream_t stream, uint64_t *launches);
// The split route's second operation: y[r,j] = S(u[r,j] * gamma[j]) over
// 16-bit values of S; vec is 8 (16-byte aligned rows) or 1.
cudaError_t launch_seam_scale(bool seam_bf16, const void *u, const void *gamma, void *y,
                              int64_t rows, int64_t n, int vec, int sms, bool pdl,
                              cudaStream_t stream, uint64_t *launches);

// Dynamic shared memory of the staged (kTma) kernel for one operation: the
// gammas once, plus each stage's row operands.
constexpr int64_t tma_shared_bytes(int op, int64_t row_bytes, int stages) {
    return row_bytes * (op_staged_gammas(op) + stages * op_row_inputs(op));
}
// The staged kernel with a cluster of `cluster` CTAs per row (each stages a
// slice of row_bytes / cluster): plain, then-add, then-add-scale, sandwich.
MRN_HOST_DEVICE constexpr bool op_has_cluster_staging(int op) {
    return op == kRmsnorm || op == kThenAdd || op == kSandwich || op == kThenAddScale;
}
// The staged kernel for rows that are not 16-byte aligned (Geometry::edge):
// the same operations, whose outputs have the row operands' element size.
MRN_HOST_DEVICE constexpr bool op_has_edge_staging(int op) { return op_has_cluster_staging(op); }
// Bytes between the shared-memory slots of the edge-staged kernel: a row of
// row_bytes starting anywhere within a 16-byte granule spans at most this
// many bytes of granules.
MRN_HOST_DEVICE constexpr int64_t edge_stage_bytes(int64_t row_bytes) {
    return (row_bytes + 15) / 16 * 16 + 16;
}
// Granules (16-byte loads) of such a row at most.
MRN_HOST_DEVICE constexpr int64_t edge_granules(int64_t row_bytes) {
    return edge_stage_bytes(row_bytes) / 16;
}
// The edge-staged kernel's persistent grid is a multiple of this many CTAs:
// rows that far apart start at the same offset within 16 bytes for any n.
constexpr int kEdgeGridMultiple = 8;

// Number of bounded waits that ran out since the last call (and reset them).
int take_wait_timeouts_rmsnorm();
int take_wait_timeouts_then_add();
int take_wait_timeouts_sandwich();
int take_wait_timeouts_add_rmsnorm();
int take_wait_timeouts_then_add_scale();
int take_wait_timeouts_rmsnorm_q8_1();
int take_wait_timeouts_seam_f16();
int take_wait_timeouts_seam_bf16();

}  // namespace mrn
