// mrn_api.cpp -- the C ABI declared in include/mrn.h: argument validation,
// geometry choice and the launch of one kernel on the caller's stream.
//
// Operations: RMSNorm ("Chapter 12 -- RMSNorm and the dual-epsilon
// sandwich", section 12.1), post norm then residual add (Hesper "RMSNorm
// Layer", rmsNormThenAddKernel), the dual-epsilon sandwich tail (section
// 12.4.3), residual add then norm (Hesper residualAddRmsNormKernel), post
// norm, add, broadcast scale (Hesper rmsNormThenAddThenBroadcastScaleKernel),
// RMSNorm with Q8_1 quantisation (Hesper fusedRMSNormQ8_1Kernel) and the
// split-norm seam (section 12.7: the weightless norm published in F16 or
// bf16, the weight applied as a second operation in that format).  This layer
// holds no arithmetic of the method; it checks arguments, picks a register
// geometry from (n, rows, dtype, alignment) and hands the call to the
// launcher of the operation.
#include "mrn.h"

#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <cmath>
#include <cstdint>

#include "mrn_internal.h"

namespace {

using mrn::Geometry;
using mrn::KernelArgs;

std::atomic<uint64_t> g_launch_count{0};
thread_local int t_last_cuda_error = 0;
thread_local bool t_forced = false;
thread_local Geometry t_forced_geometry = {};
thread_local uint32_t t_launch_options = MRN_LAUNCH_PDL;   // the default

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
constexpr int kDefaultSmCount = 152;   // GB300

int elem_bytes(mrn_dtype dt) { return dt == MRN_F32 ? 4 : 2; }

int sm_count_of_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return kDefaultSmCount;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
    }
    int count = 0;
    if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        count <= 0) {
        (void)cudaGetLastError();
        return kDefaultSmCount;
    }
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(count, std::memory_order_relaxed);
    return count;
}

int64_t pow2_ceil(int64_t v) {
    int64_t p = 1;
    while (p < v) p <<= 1;
    return p;
}

int64_t pow2_floor(int64_t v) {
    int64_t p = 1;
    while (p * 2 <= v) p <<= 1;
    return p;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int natural_vec(mrn_dtype dt) { return 16 / elem_bytes(dt); }

// Register slots k and threads t for `per` loads of a row in one CTA (or one
// warp group): the least waste (t*k - per), then t nearest `target`.
void pick_threads(int64_t per, int *k_out, int *t_out, int (*max_threads)(int) = nullptr,
                  double target = 256.0) {
    double best = 1e30;
    for (int k = 1; k <= mrn::kMaxK; ++k) {
        const int64_t t = ceil_div(ceil_div(per, k), 32) * 32;
        const int cap = max_threads ? max_threads(k) : mrn::cta_max_threads(k);
        if (t > cap) continue;
        const double waste = static_cast<double>(t * k - per) / static_cast<double>(per);
        const double shape = 0.02 * std::fabs(std::log2(static_cast<double>(t) / target));
        const double score = waste + shape;
        if (score < best) {
            best = score;
            *k_out = k;
            *t_out = static_cast<int>(t);
        }
    }
}

int tma_group_cap(int k) { return mrn::tma_group_max_threads(k); }

// For batches in the register kernel: among (k, t) with at most 1/8 of the
// slots idle, the one with t nearest `target` (measured best on GB300: 256
// for the residual add + norm, 7 x 256 at n = 6656 f32; 128 for the Q8_1
// pass, 4 x 128 at n = 4096 bf16, whose more registers per slot want fewer
// threads per CTA).
void pick_threads_batch(int64_t per, int *k_out, int *t_out, double target) {
    double best = 1e30;
    for (int k = 1; k <= mrn::kMaxK; ++k) {
        const int64_t t = ceil_div(ceil_div(per, k), 32) * 32;
        if (t > mrn::cta_max_threads(k) || (t * k - per) * 8 > per) continue;
        const double d = std::fabs(std::log2(static_cast<double>(t) / target));
        if (d < best) {
            best = d;
            *k_out = k;
            *t_out = static_cast<int>(t);
        }
    }
    if (best > 1e29) pick_threads(per, k_out, t_out);
}

// Batches (rows >= #SMs, aligned rows of at most 2048 loads) that run faster
// in the register kernel -- one row per CTA, many CTAs per SM, no persistent
// grid to drain -- than in the staged one.  From sweeps on GB300 (CUDA events,
// back to back; register vs staged or rows-per-warp, TB/s):
//  * always: the residual add + norm and the Q8_1 pass (they store or compute
//    more per byte); the f32 sandwich from 2048 rows (one reduction per row);
//  * rows of at most 512 loads, any batch: 16384 x 4096 bf16 plain 6.47 vs
//    6.16, then-add 6.90 vs 6.47, sandwich 6.30 vs 6.03; 65536 x 2048 f32
//    plain 7.04 vs 6.57, then-add 7.12 vs 6.73; 1216 x 4096 bf16 then-add
//    6.22 vs 5.28; rows of 129..256 loads too, against rows per warp (65536 x
//    2048 bf16: plain 6.81 vs 6.32, then-add 7.02 vs 5.02, sandwich 6.76 vs 5.30);
//  * plain f32 rows from 2048 rows up to 2048 loads, eight slots per thread
//    (65536 x 6656 7.08 vs 6.47; 65536 x 8192 7.13 vs 6.73; 4096 x 6656 6.41
//    vs 5.84); the f32 seam the same way (16384 x 8192 7.03 vs 6.41, 16384 x
//    6656 6.68 vs 6.48);
//  * wider rows from 2048 rows: then-add up to 1664 loads (16384 x 8192 bf16
//    7.01 vs 6.51, 65536 x 6656 f32 6.95 vs 6.84; at 2048 loads staged, 6.86
//    vs 6.11), then-add-scale the same in bf16 but up to 1280 loads in f32
//    (at 1664, 4096 x 6656: 58.8 us against 50.8 for the staged then-add);
//    bf16 plain up to 896 loads (4096 x 6656 5.45 vs 4.21); the bf16 seam from 4096
//    rows up to 896 loads (16384 x 4096 6.57 vs 6.20).  The bf16 sandwich
//    keeps the staged kernel past 512 loads (4096 x 8192: 4.71 vs 6.01).
bool register_batch_pays(mrn::Op op, mrn_dtype dt, int64_t nvec, int64_t rows) {
    if (op == mrn::kAddRmsnorm || op == mrn::kRmsnormQ8) return true;
    if (op == mrn::kSandwich && dt == MRN_F32 && rows >= 2048) return true;
    if (nvec > 2048) return false;
    const bool f32 = dt == MRN_F32;
    if (mrn::op_is_seam(op)) {
        if (f32) return nvec <= 2048 && (nvec <= 512 || rows >= 2048);
        return nvec <= 896 && rows >= 4096;
    }
    if (nvec <= 512) return true;
    if (rows < 2048 || op == mrn::kSandwich) return false;
    if (op == mrn::kThenAdd) return nvec <= 1664;
    if (op == mrn::kThenAddScale) return nvec <= (f32 ? 1280 : 1664);
    if (op == mrn::kRmsnorm && f32) return true;   // (eight slots per thread, below)
    return nvec <= (f32 ? 1280 : 896);
}

// Dynamic shared memory the staged kernel may use (the rest of the 227 KB
// holds its static reduction slots and barriers).
constexpr int64_t kTmaSharedBudget = mrn::kSharedBytesPerCta - 1024;

// Automatic geometry.  Loads per row: nvec = ceil(n / vec).
//  * nvec <= 256: several rows per warp (lanes = next power of two of nvec up
//    to 32, k = ceil(nvec / 32)); no shared memory, no barrier.
//  * at least one row per SM, 16-byte aligned rows, nvec <= 2048, and two
//    rows' operands fit in shared memory: the persistent TMA-staged kernel,
//    two warp groups, one stage each;
//  * at least one row per SM, 16-byte aligned slices, 2048 < nvec <= 16 *
//    2048 (plain, then-add, then-add-scale, sandwich): the persistent
//    cluster-staged kernel, a cluster of 2..16 CTAs per row;
//  * nvec <= 16 * 2048: the row in registers of one CTA or of a cluster of up
//    to 16 CTAs (2048 loads per CTA at most).  Few rows (decode) are spread
//    over up to 8 CTAs of a cluster so that more SMs pull the row in.
//  * wider: the looped fallback.
Geometry choose_geometry(mrn::Op op, int64_t rows, int64_t n, mrn_dtype dt, bool aligned16,
                         int sms, bool same_offset = false) {
    Geometry g = {};
    g.vec = aligned16 ? natural_vec(dt) : 1;
    g.cluster = 1;
    const int64_t nvec = ceil_div(n, g.vec);
    // Batches of rows that are not 16-byte aligned but whose row operands all
    // sit at one offset within 16 bytes (a row pitch that is not a multiple of
    // 16 bytes, or operands offset alike): the staged kernel on the 16-byte
    // granules that cover each row, as for aligned rows (measured on GB300:
    // see the edge-staged kernel's notes).
    if (!aligned16 && same_offset && mrn::op_has_edge_staging(op) && rows >= sms) {
        const int64_t stage = mrn::edge_stage_bytes(n * elem_bytes(dt));
        const int64_t gran = mrn::edge_granules(n * elem_bytes(dt));
        if (gran <= 2 * 1024 && nvec > 32 * mrn::kMaxK &&   // (shorter rows: rows per warp)
            mrn::tma_shared_bytes(op, stage, 2) <= kTmaSharedBudget) {
            g.kind = mrn::kTma;
            g.vec = natural_vec(dt);
            // (plain f32 rows keep four rows in flight per CTA where they fit:
            // 4096 x 6655 39.1 vs 40.1 us with two; aligned rows ran slower so)
            g.stages = op == mrn::kRmsnorm && dt == MRN_F32 &&
                               mrn::tma_shared_bytes(op, stage, 4) <= kTmaSharedBudget
                           ? 4 : 2;
            g.ctas = 0;
            g.groups = 2;
            g.edge = 1;
            // (measured on GB300, TB/s: 4096 x 6655 f32 sandwich 5.93 at 256 threads x
            // 7 granules per group vs 5.86 at 224 x 8; 16384 x 4095 bf16 sandwich 5.87
            // at 192 x 3 vs 5.68 at 96 x 6 and 4.18 at 288 x 2, where fewer CTAs fit
            // on an SM)
            int per_group = 0;
            pick_threads(gran, &g.k, &per_group, tma_group_cap,
                         n * elem_bytes(dt) > 16384 ? 256.0 : 192.0);
            g.threads = 2 * per_group;
            g.lanes = 0;
            g.rows_per_cta = 2;
            return g;
        }
    }
    // RMSNorm + Q8_1 batches of aligned rows: whole 32-element blocks per
    // thread (no shuffles; one reciprocal and one header per block).
    // RMSNorm + Q8_1 batches of aligned rows use the whole-block kernels
    // (measured on GB300, TB/s, rows >= 4096):
    //   f32: staged (persistent, x bulk-copied two stages ahead) everywhere --
    //        n = 1024: 4.2, 2048: 6.4, 4096: 6.3 (2 blocks per thread),
    //        16384: 5.6 (one group: two do not fit in shared memory);
    //   bf16: staged from n = 2048 (1 block per thread at 2048: 5.1 vs 4.8 for
    //        one row per CTA; 2 blocks per thread from 4096: 5.9 at 4096, 4.9 at
    //        4096 rows of 6656); below, the lane-layout kernels (n = 1024: 4.0
    //        vs 3.1 staged).
    const int64_t nblocks = n / mrn::kQ8Block;
    const int64_t max_staged = static_cast<int64_t>(mrn::kQ8BlockMaxK) * mrn::kQ8TmaGroupThreads;
    if (op == mrn::kRmsnormQ8 && aligned16 && rows >= sms && nblocks >= 32) {
        g.kind = mrn::kQ8Blocks;
        g.lanes = 0;
        if ((dt == MRN_F32 || nblocks >= 64) && nblocks <= max_staged) {
            g.k = nblocks >= 128 ? 2 : 1;
            const int per = static_cast<int>(ceil_div(ceil_div(nblocks, g.k), 32) * 32);
            for (int groups = 2; groups >= 1; --groups) {
                if (mrn::q8_tma_shared_bytes(n, elem_bytes(dt), 2, groups) <= kTmaSharedBudget) {
                    g.threads = groups * per;
                    g.stages = 2;
                    g.groups = groups;
                    g.ctas = 0;
                    g.rows_per_cta = groups;
                    return g;
                }
            }
        }
        if (dt == MRN_BF16 && nblocks >= 64 &&
            nblocks <= static_cast<int64_t>(mrn::kQ8BlockMaxK) * mrn::kQ8BlockMaxThreads) {
            g.k = nblocks <= mrn::kQ8BlockMaxThreads ? 1 : 2;
            g.threads = static_cast<int>(ceil_div(ceil_div(nblocks, g.k), 32) * 32);
            g.stages = 0;
            g.rows_per_cta = 1;
            return g;
        }
        g = Geometry{};   // the lane-layout kernels below
        g.vec = natural_vec(dt);
        g.cluster = 1;
    }
    const bool register_batch = aligned16 && rows >= sms && register_batch_pays(op, dt, nvec, rows);
    if (nvec <= 32 * mrn::kMaxK && !(register_batch && nvec > 128)) {
        // About four loads per thread (measured on GB300: per-head n = 128 rows
        // run ~15% faster with 4 slots x 4..8 lanes than with 1 slot x 16..32),
        // at least 4 lanes from 8 loads (163840 x 64 bf16: 4 x 2 7.0 us, 2 x 4
        // 8.1 us), in CTAs of 128 threads (163840 x 128 bf16: 13.8 us against
        // 14.6 us with 256; 655360 rows 49.0 vs 52.3 us: smaller CTAs drain
        // the grid's tail sooner).
        g.kind = mrn::kRowsPerWarp;
        g.threads = mrn::kWarpKernelCtaThreads;
        g.lanes = static_cast<int>(std::min<int64_t>(32, pow2_ceil(ceil_div(nvec, 4))));
        if (nvec >= 8 && g.lanes < 4) g.lanes = 4;
        if (op == mrn::kRmsnormQ8)   // a Q8_1 block must sit on consecutive lanes
            g.lanes = std::max(g.lanes, mrn::kQ8Block / g.vec);
        g.k = static_cast<int>(ceil_div(nvec, g.lanes));
        g.rows_per_cta = g.threads / g.lanes;
        return g;
    }
    // Many rows of aligned data whose staged copies fit in shared memory: the
    // persistent TMA-staged kernel with two warp groups (two rows reduced at a
    // time) and one stage per group; the occupancy calculator then puts as many
    // CTAs on an SM as fit.  (Measured on GB300: more rows in flight per SM beat
    // deeper per-CTA prefetch; groups of about 128 threads with more register
    // slots each beat wider groups.)
    const int64_t row_bytes = n * elem_bytes(dt);
    // The residual add + norm stores its sum before its only reduction, and the
    // Q8_1 pass has more arithmetic per byte; both run faster in the register
    // kernel with many CTAs per SM than in the staged one (measured on GB300:
    // add+norm 6.45 vs 6.03 TB/s at 4096 x 6656 f32).
    // Batches of 2048 rows or more of the f32 sandwich run the register kernel
    // too: there its two norms need only one reduction (the one-exchange form),
    // and one row per CTA with many CTAs per SM beat the staged kernel.  Measured
    // on GB300, back to back, register vs staged: 4096 x 6656 67.4 vs 69.9 us
    // (torch's own copy of the same 436 MB: 66.9 us), 8192 x 6656 128.2 vs 136.8,
    // 16384 x 4096 155.1 vs 170.7, 4096 x 8192 81.8 vs 86.2, 65536 x 2048 323.6
    // vs 337.5; but 1216 x 6656 23.9 vs 22.8 (a fit over rows: 15.1 ns per row +
    // 5.3 us against 16.4 ns + 2.6 us: equal at about 2060 rows).
    const bool one_exchange_sandwich = op == mrn::kSandwich && dt == MRN_F32;
    if (!register_batch && aligned16 && rows >= sms && nvec <= 2 * 1024) {
        // The seam from f32 rows reads twice the bytes it writes; a second
        // stage per group keeps more of those reads in flight (measured on
        // GB300, 4096 rows: 5.56 vs 4.75 TB/s at n = 6656, 5.45 vs 5.22 at
        // n = 4096).  The other operations ran slower with deeper stages.
        int stages = 2;
        if (mrn::op_is_seam(op) && dt == MRN_F32 &&
            mrn::tma_shared_bytes(op, row_bytes, 4) <= kTmaSharedBudget)
            stages = 4;
        if (mrn::tma_shared_bytes(op, row_bytes, stages) <= kTmaSharedBudget) {
            g.kind = mrn::kTma;
            g.stages = stages;
            g.ctas = 0;
            g.groups = 2;
            int per_group = 0;
            // (the seam's output pass is lighter: more slots per thread, 64-thread
            // groups, measured 5.88 vs 5.70 TB/s at 16384 x 4096 bf16)
            pick_threads(nvec, &g.k, &per_group, tma_group_cap,
                         mrn::op_is_seam(op) ? 64.0 : 128.0);
            g.threads = 2 * per_group;
            g.lanes = 0;
            g.rows_per_cta = 2;
            return g;
        }
    }
    // Batches of rows wider than 2048 loads: a cluster of C CTAs per row (C the
    // smallest power of two giving slices of at most 2048 loads = 32 KB), each
    // staging its slice of future rows in shared memory, the partial sums sent
    // as st.async messages.  Stages: plain 3 at C = 2, else 2; then-add (and
    // -scale) 2 up to C = 4, then 3; sandwich 2, with C doubled from 8 so two
    // CTAs fit per SM.  Measured on GB300 (TB/s; staged vs the register
    // cluster kernel it replaces): f32 4096 x 16384 plain 6.41 vs 5.06,
    // then-add 6.62 vs 5.52; 65536 x 16384 plain 6.79 vs 5.28; 8192 x 32768
    // plain 6.43 vs 4.91, then-add 6.77 vs 5.14; 4096 x 65536 plain 6.64 vs
    // 4.31, then-add 6.88 vs 4.93, sandwich 5.94 vs 3.03; sandwich 16384 x
    // 16384 6.55 vs 4.65; bf16 8192 x 32768 plain 6.27 vs 4.73, then-add 6.72
    // vs 4.06.  (The other stage counts lost 5-20 %: with one CTA per SM a
    // cluster of 8 packs the GPCs less well, and deeper staging of two
    // operands overfilled the SM.)
    // Plain f32 batches of wider rows: the register kernel at eight slots per
    // thread (three CTAs per SM), a cluster of ceil(nvec / 1024) CTAs per row, up
    // to 8 (measured on GB300 against the cluster-staged kernel: 4096 x 16384
    // 78.9 vs 83.6 us, 65536 x 16384 1190.6 vs 1258.1, 4096 x 32768 156.3 vs
    // 171.6; at 16 CTAs, 4096 x 65536, no clear gain: 337-338 vs 340 us in one
    // measurement, 6.35 vs 6.55 TB/s in the bench's).
    if (op == mrn::kRmsnorm && dt == MRN_F32 && aligned16 && rows >= 2048 && nvec > 2048 &&
        nvec <= 8 * 1024) {
        const int64_t ccl = ceil_div(nvec, 1024);
        const int64_t per = ceil_div(ceil_div(nvec, ccl), 32) * 32;   // loads per CTA
        g.kind = mrn::kCta;
        g.cluster = static_cast<int>(ccl);
        g.k = mrn::kMaxK;
        g.threads = static_cast<int>(ceil_div(per, 32 * mrn::kMaxK) * 32);
        g.lanes = 0;
        g.rows_per_cta = 1;
        return g;
    }
    if (mrn::op_has_cluster_staging(op) && aligned16 && rows >= sms && nvec > 2048 &&
        nvec <= static_cast<int64_t>(mrn::kMaxCluster) * 2048) {
        int64_t ccl = 2;
        while (ccl * 2048 < nvec) ccl *= 2;
        if (op == mrn::kSandwich && ccl >= 8 && ccl < mrn::kMaxCluster) ccl *= 2;
        int stages = 2;
        if (op == mrn::kRmsnorm && ccl == 2) stages = 3;
        if ((op == mrn::kThenAdd || op == mrn::kThenAddScale) && ccl >= 8) stages = 3;
        const int64_t slice = row_bytes / ccl;
        auto fits = [&](int st) {
            return (mrn::op_gammas(op) + st * mrn::op_row_inputs(op)) * slice <= kTmaSharedBudget;
        };
        if (!fits(stages)) stages = 2;
        if (row_bytes % (16 * ccl) == 0 && fits(stages)) {
            g.kind = mrn::kTma;
            g.cluster = static_cast<int>(ccl);
            g.groups = 1;
            g.stages = stages;
            g.ctas = 0;
            pick_threads(nvec / ccl, &g.k, &g.threads);
            g.lanes = 0;
            g.rows_per_cta = 1;
            return g;
        }
    }
    constexpr int64_t kCtaLoads = 2048;
    int64_t cl = ceil_div(nvec, kCtaLoads);
    // Batches of wide f32 rows: half the loads per CTA (four register slots),
    // up to clusters of 8 (measured on GB300: 65536 x 16384 plain 5.28 vs 4.94
    // TB/s, then-add 5.91 vs 5.47; 8192 x 32768 plain 4.91 vs 4.68).  bf16
    // rows were faster with the full 2048 loads per CTA.
    if (dt == MRN_F32 && rows >= sms && cl >= 2 && ceil_div(nvec, kCtaLoads / 2) <= 8)
        cl = ceil_div(nvec, kCtaLoads / 2);
    if (cl > mrn::kMaxCluster) {
        // Rows past what registers and staged slices hold: the looped kernel, a
        // cluster of CTAs per row, each looping over its slice, so that few rows
        // are in flight and each slice's second read comes from L2.  Measured on
        // GB300 (plain f32, 256 x 262144; ncu, one launch): clusters of 8 read
        // 1.008x the input from DRAM in 118 us, of 16 1.004x in 138 us, of 4
        // 1.19x in 113 us, of 2 1.75x in 117 us, one row per CTA 1.56x in 128 us;
        // 16 x 2^20: 16 CTAs 43 us, 8 47 us.
        g.kind = mrn::kStream;
        g.threads = mrn::kStreamMaxThreads;
        g.k = 1;
        g.cluster = rows >= 32 ? 8 : mrn::kMaxCluster;
        g.lanes = 0;
        g.rows_per_cta = 1;
        return g;
    }
    if (rows * 2 <= sms) {
        // Few rows (decode): spread each row over up to 8 CTAs of a cluster,
        // keeping at least ~192 loads per CTA, so that more SMs pull it in.
        // The f32 sandwich, with one exchange, goes to 16 CTAs of ~104 loads
        // (measured on GB300, 1 x 6656 in a CUDA graph over rotating buffers:
        // 16 x 128 threads 2.08 us, 8 x 224 threads 2.22 us per call).
        const int64_t cap = one_exchange_sandwich ? 16 : 8;
        const int64_t by_rows = pow2_floor(std::max<int64_t>(1, sms / rows));
        const int64_t by_width =
            pow2_floor(std::max<int64_t>(1, nvec / (one_exchange_sandwich ? 96 : 192)));
        cl = std::max(cl, std::min(cap, std::min(by_rows, by_width)));
    }
    if (register_batch) {
        // about four register slots per thread (two for the bf16 sandwich, whose
        // slots hold more), 64..256 threads; 256 for the residual add + norm,
        // 128 for the Q8_1 pass (measured best)
        double target = std::min(256.0, std::max(64.0, static_cast<double>(nvec) /
                                     (op == mrn::kSandwich && dt == MRN_BF16 ? 2.0 : 4.0)));
        // plain f32 rows past 512 loads: eight slots per thread, the kernel then
        // fitting three CTAs per SM (65536 x 6656: 224 x 8 492.8 us, 256 x 7 551.6,
        // staged 539.5; 65536 x 5120: 160 x 8 378.0 vs 256 x 5 395.5); then-add up
        // to 512 threads of four slots (65536 x 6656: 416 x 4 743.8 us, 256 x 7 764.9)
        if ((op == mrn::kRmsnorm || mrn::op_is_seam(op)) && dt == MRN_F32 && nvec > 512)
            target = std::min(256.0, static_cast<double>(nvec) / 8.0);
        if (op == mrn::kThenAdd)
            target = std::min(512.0, std::max(64.0, static_cast<double>(nvec) / 4.0));
        if (op == mrn::kAddRmsnorm) target = 256.0;
        if (op == mrn::kRmsnormQ8) target = 128.0;
        pick_threads_batch(ceil_div(nvec, cl), &g.k, &g.threads, target);
    } else {
        pick_threads(ceil_div(nvec, cl), &g.k, &g.threads);
    }
    g.kind = mrn::kCta;
    g.cluster = static_cast<int>(cl);
    g.lanes = 0;
    g.rows_per_cta = 1;
    return g;
}

bool geometry_is_consistent(const Geometry &g) {
    // the edge-staged kernel exists with two warp groups and no cluster only
    if (g.edge && (g.kind != mrn::kTma || g.groups != 2 || g.cluster != 1)) return false;
    if (g.kind == mrn::kRowsPerWarp) {
        const bool pow2 = g.lanes >= 1 && g.lanes <= 32 && (g.lanes & (g.lanes - 1)) == 0;
        return pow2 && g.k >= 1 && g.k <= mrn::kMaxK && g.threads >= 32 && g.threads % 32 == 0 &&
               g.threads <= mrn::kWarpKernelThreads;
    }
    if (g.kind == mrn::kCta) {
        return g.k >= 1 && g.k <= mrn::kMaxK && g.threads >= 32 && g.threads % 32 == 0 &&
               g.threads <= mrn::cta_max_threads(g.k) && g.cluster >= 1 &&
               g.cluster <= mrn::kMaxCluster;
    }
    if (g.kind == mrn::kStream) {
        return g.threads >= 32 && g.threads % 32 == 0 && g.threads <= mrn::kStreamMaxThreads &&
               g.cluster >= 1 && g.cluster <= mrn::kMaxCluster;
    }
    if (g.kind == mrn::kQ8Blocks) {
        if (g.k < 1 || g.k > mrn::kQ8BlockMaxK || g.threads < 32 || g.threads % 32 != 0)
            return false;
        if (g.stages == 0) return g.threads <= mrn::kQ8BlockMaxThreads;
        // staged: one stage per group per row, as for kTma
        return g.groups >= 1 && g.groups <= 2 && g.threads % (32 * g.groups) == 0 &&
               g.threads / g.groups <= mrn::kQ8TmaGroupThreads && g.stages >= g.groups &&
               g.stages % g.groups == 0 && g.stages <= mrn::kTmaMaxStages && g.ctas >= 0;
    }
    if (g.kind == mrn::kTma) {
        if (g.groups < 1 || g.groups > mrn::kTmaMaxGroups) return false;
        if (g.cluster < 1 || g.cluster > mrn::kMaxCluster) return false;
        if (g.cluster > 1 && g.groups != 1) return false;   // one group per CTA of a cluster
        const int per_group = g.threads / g.groups;
        return g.k >= 1 && g.k <= mrn::kMaxK && g.threads % (32 * g.groups) == 0 &&
               per_group >= 32 && g.threads <= mrn::tma_max_threads(g.k, g.groups) &&
               g.stages >= g.groups && g.stages % g.groups == 0 &&
               g.stages <= mrn::kTmaMaxStages && g.ctas >= 0;
    }
    return false;
}

// Resolve the thread's forced geometry for one call; false if it cannot
// cover the row or asks for vectors the pointers do not allow.
bool resolve_forced(Geometry g, mrn::Op op, int64_t n, mrn_dtype dt, bool aligned16,
                    Geometry *out, bool same_offset = false) {
    if (g.edge) {
        // the edge-staged kernel: 16-byte granules of rows at one offset
        // (aligned rows are the case of offset 0)
        if (!mrn::op_has_edge_staging(op) || !(aligned16 || same_offset)) return false;
        if (g.vec == 0) g.vec = natural_vec(dt);
        if (g.vec != natural_vec(dt)) return false;
        const int64_t stage = mrn::edge_stage_bytes(n * elem_bytes(dt));
        if (static_cast<int64_t>(g.threads / g.groups) * g.k < mrn::edge_granules(n * elem_bytes(dt)))
            return false;
        if (mrn::tma_shared_bytes(op, stage, g.stages) > kTmaSharedBudget) return false;
        g.cluster = 1;
        g.lanes = 0;
        g.rows_per_cta = g.groups;
        *out = g;
        return true;
    }
    if (g.vec == 0) g.vec = aligned16 ? natural_vec(dt) : 1;
    if (g.vec != 1 && !(g.vec == natural_vec(dt) && aligned16)) return false;
    const int64_t nvec = ceil_div(n, g.vec);
    if (g.kind == mrn::kQ8Blocks) {
        if (op != mrn::kRmsnormQ8 || !aligned16 || g.vec != natural_vec(dt)) return false;
        const int per = g.stages > 0 ? g.threads / g.groups : g.threads;
        if (static_cast<int64_t>(per) * g.k * mrn::kQ8Block < n) return false;
        if (g.stages > 0 &&
            mrn::q8_tma_shared_bytes(n, elem_bytes(dt), g.stages, g.groups) > kTmaSharedBudget)
            return false;
        g.cluster = 1;
        g.lanes = 0;
        g.rows_per_cta = g.stages > 0 ? g.groups : 1;
    } else if (g.kind == mrn::kTma && g.cluster > 1) {
        // a cluster per row: each CTA stages a 16-byte-aligned slice
        if (!mrn::op_has_cluster_staging(op)) return false;
        if (!aligned16 || g.vec != natural_vec(dt)) return false;
        const int64_t row_bytes = n * elem_bytes(dt);
        if (row_bytes % (16 * g.cluster) != 0) return false;
        if (static_cast<int64_t>(g.threads) * g.k < nvec / g.cluster) return false;
        if ((mrn::op_gammas(op) + g.stages * mrn::op_row_inputs(op)) * (row_bytes / g.cluster) >
            kTmaSharedBudget)
            return false;
        g.lanes = 0;
        g.rows_per_cta = 1;
    } else if (g.kind == mrn::kTma) {
        if (!aligned16 || g.vec != natural_vec(dt)) return false;
        if (static_cast<int64_t>(g.threads / g.groups) * g.k < nvec) return false;
        if (mrn::tma_shared_bytes(op, n * elem_bytes(dt), g.stages) > kTmaSharedBudget)
            return false;
        g.cluster = 1;
        g.lanes = 0;
        g.rows_per_cta = g.groups;
    } else if (g.kind == mrn::kRowsPerWarp) {
        if (static_cast<int64_t>(g.lanes) * g.k < nvec) return false;
        if (op == mrn::kRmsnormQ8 && g.lanes < mrn::kQ8Block / g.vec) return false;
        g.cluster = 1;
        g.rows_per_cta = g.threads / g.lanes;
    } else if (g.kind == mrn::kCta) {
        if (static_cast<int64_t>(g.cluster) * g.threads * g.k < nvec) return false;
        g.lanes = 0;
        g.rows_per_cta = 1;
    } else {   // the looped kernel: any width, one row per CTA or per cluster
        g.k = 1;
        g.lanes = 0;
        g.rows_per_cta = 1;
    }
    *out = g;
    return true;
}

struct Span {
    uintptr_t lo;
    uintptr_t hi;
};

Span span_of(const void *p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// An output may coincide exactly with a row input or be disjoint from it.
bool output_vs_row_input_ok(Span out, Span in) { return !overlaps(out, in) || out.lo == in.lo; }

mrn_status check_common(int64_t rows, int64_t n, mrn_dtype dt, float eps1, float eps2) {
    if (dt != MRN_F32 && dt != MRN_BF16) return MRN_ERR_UNSUPPORTED_DTYPE;
    if (n < 1 || rows < 0) return MRN_ERR_INVALID_SIZE;
    const int64_t e = elem_bytes(dt);
    if (n > INT64_MAX / e) return MRN_ERR_INVALID_SIZE;
    if (rows > 0 && rows > INT64_MAX / (n * e)) return MRN_ERR_INVALID_SIZE;
    if (!(eps1 > 0.0f) || !std::isfinite(eps1)) return MRN_ERR_INVALID_EPS;
    if (!(eps2 > 0.0f) || !std::isfinite(eps2)) return MRN_ERR_INVALID_EPS;
    return MRN_OK;
}

bool aligned_to(const void *p, int64_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// True when every given pointer sits at the same offset within 16 bytes (then
// every row of the call starts at one offset in all its row operands).
bool same_offset16(std::initializer_list<const void *> ptrs) {
    const uintptr_t m = reinterpret_cast<uintptr_t>(*ptrs.begin()) & 15u;
    for (const void *p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != m) return false;
    return true;
}

struct Call {
    mrn::Op op;
    mrn_dtype dt;
    int64_t rows;
    int64_t n;
    KernelArgs args;
    bool same_offset;   // every row operand at one offset within 16 bytes
};

mrn_status launch(const Call &c, bool aligned16, cudaStream_t stream) {
    Geometry g;
    if (t_forced) {
        if (!resolve_forced(t_forced_geometry, c.op, c.n, c.dt, aligned16, &g, c.same_offset))
            return MRN_ERR_INVALID_GEOMETRY;
    } else {
        g = choose_geometry(c.op, c.rows, c.n, c.dt, aligned16, sm_count_of_current_device(),
                            c.same_offset);
    }
    g.pdl = (t_launch_options & MRN_LAUNCH_PDL) ? 1 : 0;
    KernelArgs a = c.args;
    a.stall_bytes = (t_launch_options & MRN_LAUNCH_TEST_WAIT_TIMEOUT) ? 16u : 0u;
    a.n = c.n;
    a.nvec = ceil_div(c.n, g.vec);
    const bool bf16 = c.dt == MRN_BF16;
    uint64_t launched = 0;
    cudaError_t err;
    switch (c.op) {
    case mrn::kRmsnorm: err = mrn::launch_rmsnorm(bf16, g, a, c.rows, stream, &launched); break;
    case mrn::kThenAdd: err = mrn::launch_then_add(bf16, g, a, c.rows, stream, &launched); break;
    case mrn::kSandwich: err = mrn::launch_sandwich(bf16, g, a, c.rows, stream, &launched); break;
    case mrn::kAddRmsnorm:
        err = mrn::launch_add_rmsnorm(bf16, g, a, c.rows, stream, &launched);
        break;
    case mrn::kThenAddScale:
        err = mrn::launch_then_add_scale(bf16, g, a, c.rows, stream, &launched);
        break;
    case mrn::kRmsnormQ8:
        err = mrn::launch_rmsnorm_q8_1(bf16, g, a, c.rows, stream, &launched);
        break;
    default:
        err = mrn::op_seam_bf16(c.op)
                  ? mrn::launch_seam_bf16(c.op, bf16, g, a, c.rows, stream, &launched)
                  : mrn::launch_seam_f16(c.op, bf16, g, a, c.rows, stream, &launched);
        break;
    }
    g_launch_count.fetch_add(launched, std::memory_order_relaxed);
    if (err != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(err);
        (void)cudaGetLastError();   // clear the non-sticky launch error
        return MRN_ERR_CUDA;
    }
    return MRN_OK;
}

// The seam norms: the fused form (weighted) and the split route's weightless
// first operation.  x is f32 or bf16; the output (and gamma) hold 16-bit
// values of `seam`.  The output may be x itself only when x also holds 16-bit
// elements, so that element (r, j) of both sits at the same address.
mrn_status seam_norm(bool weighted, const void *x, const void *gamma, void *y, int64_t rows,
                     int64_t n, float eps, mrn_dtype dtype, mrn_dtype seam, cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK) return st;
    if (seam != MRN_F16 && seam != MRN_BF16) return MRN_ERR_UNSUPPORTED_DTYPE;
    if (rows == 0) return MRN_OK;
    if (!x || !y || (weighted && !gamma)) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(x, e) || !aligned_to(y, 2) || (weighted && !aligned_to(gamma, 2)))
        return MRN_ERR_MISALIGNED;
    const Span sx = span_of(x, rows * n * e), sy = span_of(y, rows * n * 2);
    if (e == 2 ? !output_vs_row_input_ok(sy, sx) : overlaps(sy, sx)) return MRN_ERR_ALIASING;
    if (weighted && overlaps(sy, span_of(gamma, n * 2))) return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(x, 16) && aligned_to(y, 16) &&
                     (!weighted || aligned_to(gamma, 16));
    const bool bf = seam == MRN_BF16;
    const mrn::Op op = weighted ? (bf ? mrn::kSeamBF16 : mrn::kSeamF16)
                                : (bf ? mrn::kUnweightedBF16 : mrn::kUnweightedF16);
    Call c{op, dtype, rows, n, KernelArgs{}, false};
    c.args.x = x;
    c.args.g1 = gamma;
    c.args.y = y;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

}  // namespace

extern "C" {

mrn_status mrn_rmsnorm(const void *x, const void *gamma, void *y, int64_t rows, int64_t n,
                       float eps, mrn_dtype dtype, cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK || rows == 0) return st;
    if (!x || !gamma || !y) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(x, e) || !aligned_to(gamma, e) || !aligned_to(y, e))
        return MRN_ERR_MISALIGNED;
    const int64_t row_bytes = rows * n * e;
    const Span sx = span_of(x, row_bytes), sg = span_of(gamma, n * e), sy = span_of(y, row_bytes);
    if (!output_vs_row_input_ok(sy, sx) || overlaps(sy, sg)) return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(x, 16) && aligned_to(gamma, 16) &&
                     aligned_to(y, 16);
    Call c{mrn::kRmsnorm, dtype, rows, n, KernelArgs{}, same_offset16({x, y})};
    c.args.x = x;
    c.args.g1 = gamma;
    c.args.y = y;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

mrn_status mrn_rmsnorm_then_add(const void *x, const void *gamma, const void *residual, void *out,
                                int64_t rows, int64_t n, float eps, mrn_dtype dtype,
                                cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK || rows == 0) return st;
    if (!x || !gamma || !residual || !out) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(x, e) || !aligned_to(gamma, e) || !aligned_to(residual, e) ||
        !aligned_to(out, e))
        return MRN_ERR_MISALIGNED;
    const int64_t row_bytes = rows * n * e;
    const Span sx = span_of(x, row_bytes), sr = span_of(residual, row_bytes);
    const Span sg = span_of(gamma, n * e), so = span_of(out, row_bytes);
    if (!output_vs_row_input_ok(so, sx) || !output_vs_row_input_ok(so, sr) || overlaps(so, sg))
        return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(x, 16) && aligned_to(gamma, 16) &&
                     aligned_to(residual, 16) && aligned_to(out, 16);
    Call c{mrn::kThenAdd, dtype, rows, n, KernelArgs{}, same_offset16({x, residual, out})};
    c.args.x = x;
    c.args.res = residual;
    c.args.g1 = gamma;
    c.args.y = out;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

mrn_status mrn_norm_residual_norm(const void *block_out, const void *residual,
                                  const void *gamma_post, const void *gamma_pre,
                                  void *out_stream, void *normed, int64_t rows, int64_t n,
                                  float eps_post, float eps_pre, mrn_dtype dtype,
                                  cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps_post, eps_pre);
    if (st != MRN_OK || rows == 0) return st;
    if (!block_out || !residual || !gamma_post || !gamma_pre || !out_stream || !normed)
        return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(block_out, e) || !aligned_to(residual, e) || !aligned_to(gamma_post, e) ||
        !aligned_to(gamma_pre, e) || !aligned_to(out_stream, e) || !aligned_to(normed, e))
        return MRN_ERR_MISALIGNED;
    const int64_t row_bytes = rows * n * e;
    const Span sb = span_of(block_out, row_bytes), sr = span_of(residual, row_bytes);
    const Span sgp = span_of(gamma_post, n * e), sgq = span_of(gamma_pre, n * e);
    const Span ss = span_of(out_stream, row_bytes), sn = span_of(normed, row_bytes);
    if (!output_vs_row_input_ok(ss, sb) || !output_vs_row_input_ok(ss, sr) ||
        !output_vs_row_input_ok(sn, sb) || !output_vs_row_input_ok(sn, sr) || overlaps(ss, sn) ||
        overlaps(ss, sgp) || overlaps(ss, sgq) || overlaps(sn, sgp) || overlaps(sn, sgq))
        return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(block_out, 16) && aligned_to(residual, 16) &&
                     aligned_to(gamma_post, 16) && aligned_to(gamma_pre, 16) &&
                     aligned_to(out_stream, 16) && aligned_to(normed, 16);
    Call c{mrn::kSandwich, dtype, rows, n, KernelArgs{},
           same_offset16({block_out, residual, out_stream, normed})};
    c.args.x = block_out;
    c.args.res = residual;
    c.args.g1 = gamma_post;
    c.args.g2 = gamma_pre;
    c.args.y = out_stream;
    c.args.y2 = normed;
    c.args.eps1 = eps_post;
    c.args.eps2 = eps_pre;
    return launch(c, a16, stream);
}

mrn_status mrn_add_rmsnorm(const void *a, const void *b, const void *gamma, void *residual_out,
                           void *normed, int64_t rows, int64_t n, float eps, mrn_dtype dtype,
                           cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK || rows == 0) return st;
    if (!a || !b || !gamma || !residual_out || !normed) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(a, e) || !aligned_to(b, e) || !aligned_to(gamma, e) ||
        !aligned_to(residual_out, e) || !aligned_to(normed, e))
        return MRN_ERR_MISALIGNED;
    const int64_t row_bytes = rows * n * e;
    const Span sa = span_of(a, row_bytes), sb = span_of(b, row_bytes);
    const Span sg = span_of(gamma, n * e);
    const Span ss = span_of(residual_out, row_bytes), sn = span_of(normed, row_bytes);
    if (!output_vs_row_input_ok(ss, sa) || !output_vs_row_input_ok(ss, sb) ||
        !output_vs_row_input_ok(sn, sa) || !output_vs_row_input_ok(sn, sb) || overlaps(ss, sn) ||
        overlaps(ss, sg) || overlaps(sn, sg))
        return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(a, 16) && aligned_to(b, 16) &&
                     aligned_to(gamma, 16) && aligned_to(residual_out, 16) &&
                     aligned_to(normed, 16);
    Call c{mrn::kAddRmsnorm, dtype, rows, n, KernelArgs{}, false};
    c.args.x = a;
    c.args.res = b;
    c.args.g1 = gamma;
    c.args.y = residual_out;
    c.args.y2 = normed;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

mrn_status mrn_rmsnorm_then_add_scale(const void *x, const void *gamma, const void *residual,
                                      const void *out_scale, void *out, int64_t rows, int64_t n,
                                      float eps, mrn_dtype dtype, cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK || rows == 0) return st;
    if (!x || !gamma || !residual || !out_scale || !out) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(x, e) || !aligned_to(gamma, e) || !aligned_to(residual, e) ||
        !aligned_to(out_scale, e) || !aligned_to(out, e))
        return MRN_ERR_MISALIGNED;
    const int64_t row_bytes = rows * n * e;
    const Span sx = span_of(x, row_bytes), sr = span_of(residual, row_bytes);
    const Span sg = span_of(gamma, n * e), sc = span_of(out_scale, e);
    const Span so = span_of(out, row_bytes);
    if (!output_vs_row_input_ok(so, sx) || !output_vs_row_input_ok(so, sr) || overlaps(so, sg) ||
        overlaps(so, sc))
        return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(x, 16) && aligned_to(gamma, 16) &&
                     aligned_to(residual, 16) && aligned_to(out, 16);
    Call c{mrn::kThenAddScale, dtype, rows, n, KernelArgs{}, same_offset16({x, residual, out})};
    c.args.x = x;
    c.args.res = residual;
    c.args.g1 = gamma;
    c.args.scale = out_scale;
    c.args.y = out;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

mrn_status mrn_rmsnorm_q8_1(const void *x, const void *gamma, void *blocks, int64_t rows,
                            int64_t n, float eps, mrn_dtype dtype, cudaStream_t stream) {
    mrn_status st = check_common(rows, n, dtype, eps, eps);
    if (st != MRN_OK) return st;
    if (n % mrn::kQ8Block != 0) return MRN_ERR_INVALID_SIZE;
    if (rows > 0 && rows > INT64_MAX / ((n / mrn::kQ8Block) * mrn::kQ8BlockBytes))
        return MRN_ERR_INVALID_SIZE;
    if (rows == 0) return MRN_OK;
    if (!x || !gamma || !blocks) return MRN_ERR_NULL_POINTER;
    const int64_t e = elem_bytes(dtype);
    if (!aligned_to(x, e) || !aligned_to(gamma, e) || !aligned_to(blocks, 4))
        return MRN_ERR_MISALIGNED;
    const Span sx = span_of(x, rows * n * e), sg = span_of(gamma, n * e);
    const Span so = span_of(blocks, rows * (n / mrn::kQ8Block) * mrn::kQ8BlockBytes);
    if (overlaps(so, sx) || overlaps(so, sg)) return MRN_ERR_ALIASING;
    const bool a16 = (n * e) % 16 == 0 && aligned_to(x, 16) && aligned_to(gamma, 16);
    Call c{mrn::kRmsnormQ8, dtype, rows, n, KernelArgs{}, false};
    c.args.x = x;
    c.args.g1 = gamma;
    c.args.y = blocks;
    c.args.eps1 = eps;
    c.args.eps2 = eps;
    return launch(c, a16, stream);
}

mrn_status mrn_rmsnorm_seam(const void *x, const void *gamma, void *y, int64_t rows, int64_t n,
                            float eps, mrn_dtype dtype, mrn_dtype seam, cudaStream_t stream) {
    return seam_norm(true, x, gamma, y, rows, n, eps, dtype, seam, stream);
}

mrn_status mrn_rmsnorm_unweighted(const void *x, void *u, int64_t rows, int64_t n, float eps,
                                  mrn_dtype dtype, mrn_dtype seam, cudaStream_t stream) {
    return seam_norm(false, x, nullptr, u, rows, n, eps, dtype, seam, stream);
}

mrn_status mrn_seam_scale(const void *u, const void *gamma, void *y, int64_t rows, int64_t n,
                          mrn_dtype seam, cudaStream_t stream) {
    if (seam != MRN_F16 && seam != MRN_BF16) return MRN_ERR_UNSUPPORTED_DTYPE;
    if (n < 1 || rows < 0) return MRN_ERR_INVALID_SIZE;
    if (n > INT64_MAX / 2 || (rows > 0 && rows > INT64_MAX / (n * 2))) return MRN_ERR_INVALID_SIZE;
    if (rows == 0) return MRN_OK;
    if (!u || !gamma || !y) return MRN_ERR_NULL_POINTER;
    if (!aligned_to(u, 2) || !aligned_to(gamma, 2) || !aligned_to(y, 2)) return MRN_ERR_MISALIGNED;
    const Span su = span_of(u, rows * n * 2), sg = span_of(gamma, n * 2);
    const Span sy = span_of(y, rows * n * 2);
    if (!output_vs_row_input_ok(sy, su) || overlaps(sy, sg)) return MRN_ERR_ALIASING;
    const bool a16 = (n * 2) % 16 == 0 && aligned_to(u, 16) && aligned_to(gamma, 16) &&
                     aligned_to(y, 16);
    uint64_t launched = 0;
    const cudaError_t err = mrn::launch_seam_scale(
        seam == MRN_BF16, u, gamma, y, rows, n, a16 ? 8 : 1, sm_count_of_current_device(),
        (t_launch_options & MRN_LAUNCH_PDL) != 0, stream, &launched);
    g_launch_count.fetch_add(launched, std::memory_order_relaxed);
    if (err != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(err);
        (void)cudaGetLastError();
        return MRN_ERR_CUDA;
    }
    return MRN_OK;
}

const char *mrn_status_string(mrn_status status) {
    switch (status) {
    case MRN_OK: return "ok";
    case MRN_ERR_NULL_POINTER: return "a required pointer is NULL";
    case MRN_ERR_INVALID_SIZE: return "invalid size (n < 1, rows < 0 or byte size overflow)";
    case MRN_ERR_INVALID_EPS: return "eps must be finite and > 0";
    case MRN_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case MRN_ERR_ALIASING: return "forbidden overlap between buffers";
    case MRN_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case MRN_ERR_CUDA: return "CUDA launch failed (see mrn_last_cuda_error)";
    case MRN_ERR_INVALID_GEOMETRY: return "forced geometry cannot cover this call";
    }
    return "unknown status";
}

int mrn_last_cuda_error(void) { return t_last_cuda_error; }

mrn_status mrn_query_geometry(mrn_op op, int64_t rows, int64_t n, mrn_dtype dtype,
                              int32_t aligned16, int32_t sm_count, mrn_geometry *out) {
    if (!out) return MRN_ERR_NULL_POINTER;
    if (op < MRN_OP_RMSNORM || op > MRN_OP_RMSNORM_UNWEIGHTED) return MRN_ERR_INVALID_GEOMETRY;
    mrn_status st = check_common(rows, n, dtype, 1.0f, 1.0f);
    if (st != MRN_OK) return st;
    // aligned16: 1 = every pointer 16-byte aligned; 2 = the row operands at
    // one offset within 16 bytes (not all aligned); 0 = neither
    const bool a16 = aligned16 == 1 && (n * elem_bytes(dtype)) % 16 == 0;
    const bool same = aligned16 == 2 || (aligned16 == 1 && !a16);
    // (the seam's geometry does not depend on its 16-bit format)
    const mrn::Op iop = op == MRN_OP_RMSNORM_SEAM         ? mrn::kSeamF16
                        : op == MRN_OP_RMSNORM_UNWEIGHTED ? mrn::kUnweightedF16
                                                          : static_cast<mrn::Op>(op);
    Geometry g;
    if (t_forced) {
        if (!resolve_forced(t_forced_geometry, iop, n, dtype, a16, &g, same))
            return MRN_ERR_INVALID_GEOMETRY;
    } else {
        g = choose_geometry(iop, rows, n, dtype, a16,
                            sm_count > 0 ? sm_count : sm_count_of_current_device(), same);
    }
    out->kind = g.kind;
    out->vec = g.vec;
    out->k = g.k;
    out->threads = g.threads;
    out->cluster = g.cluster;
    out->lanes_per_row = g.lanes;
    out->rows_per_cta = g.rows_per_cta;
    const bool staged = g.kind == mrn::kTma || (g.kind == mrn::kQ8Blocks && g.stages > 0);
    out->stages = staged ? g.stages : 0;
    out->ctas = staged ? g.ctas : 0;
    out->groups = staged ? g.groups : 0;
    out->edge = g.edge;
    return MRN_OK;
}

mrn_status mrn_force_geometry(const mrn_geometry *geometry) {
    if (!geometry || geometry->kind == MRN_GEOM_AUTO) {
        t_forced = false;
        return MRN_OK;
    }
    Geometry g = {};
    g.kind = geometry->kind;
    g.vec = geometry->vec;
    g.k = geometry->k;
    g.threads = geometry->threads;
    g.cluster = geometry->cluster;
    g.lanes = geometry->lanes_per_row;
    g.stages = geometry->stages;
    g.ctas = geometry->ctas;
    g.groups = geometry->groups;
    g.edge = geometry->edge != 0 ? 1 : 0;
    if ((g.kind == mrn::kTma || (g.kind == mrn::kQ8Blocks && g.stages > 0)) && g.groups == 0)
        g.groups = 1;
    if (g.kind == mrn::kRowsPerWarp && g.threads == 0) g.threads = mrn::kWarpKernelThreads;
    if (g.kind == mrn::kStream) g.k = 1;
    if ((g.kind == mrn::kTma || g.kind == mrn::kStream) && g.cluster == 0) g.cluster = 1;
    if (g.kind != mrn::kCta && g.kind != mrn::kTma && g.kind != mrn::kStream) g.cluster = 1;
    if (!geometry_is_consistent(g) || g.vec < 0) return MRN_ERR_INVALID_GEOMETRY;
    t_forced_geometry = g;
    t_forced = true;
    return MRN_OK;
}

uint64_t mrn_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

mrn_status mrn_set_launch_options(uint32_t options) {
    if (options & ~static_cast<uint32_t>(MRN_LAUNCH_PDL | MRN_LAUNCH_TEST_WAIT_TIMEOUT))
        return MRN_ERR_INVALID_GEOMETRY;
    t_launch_options = options;
    return MRN_OK;
}

uint32_t mrn_launch_options(void) { return t_launch_options; }

int mrn_wait_timeouts(void) {
    const int counts[] = {mrn::take_wait_timeouts_rmsnorm(), mrn::take_wait_timeouts_then_add(),
                          mrn::take_wait_timeouts_sandwich(),
                          mrn::take_wait_timeouts_add_rmsnorm(),
                          mrn::take_wait_timeouts_then_add_scale(),
                          mrn::take_wait_timeouts_rmsnorm_q8_1(),
                          mrn::take_wait_timeouts_seam_f16(),
                          mrn::take_wait_timeouts_seam_bf16()};
    int total = 0;
    for (int v : counts) {
        if (v < 0) {
            (void)cudaGetLastError();
            return -1;
        }
        total += v;
    }
    return total;
}

}  // extern "C"
