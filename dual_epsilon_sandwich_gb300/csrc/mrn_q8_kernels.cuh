// mrn_q8_kernels.cuh -- RMSNorm fused with Q8_1 block quantisation, whole
// 32-element blocks per thread: one row per CTA, and the persistent staged
// form.  (The lane-layout Q8_1 output of the generic kernels, q8_1_output,
// stays in mrn_kernels.cuh.)
#pragma once

#include "mrn_kernels.cuh"

namespace mrn {

// ---------------------------------------------------------------------------
// RMSNorm + Q8_1 with whole blocks per thread (Hesper fusedRMSNormQ8_1Kernel;
// the same arithmetic as q8_1_output).  One row per CTA; thread t owns the
// 32-element blocks t, t + blockDim.x, ... (KB of them) and holds each as
// 16-byte chunks (4 for bf16, 8 for f32), so a block's amax, reciprocal and
// header cost no shuffles and are paid once per 32 elements.  The products
// run two lanes at a time (mul.rn.f32x2 / fma.rn.f32x2: each half rounded as
// the scalar instruction would).  Each thread writes its 36-byte blocks into
// shared memory (stride 9 words: no bank conflicts), and the CTA then copies
// the row's blocks to global memory with coalesced 16-byte stores.  Needs
// 16-byte aligned rows; n = 32 * (number of blocks).
// ---------------------------------------------------------------------------
// Low bytes of four codes (each in the low byte of a word) packed in order.
__device__ __forceinline__ uint32_t pack4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
    return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

// Code word of four normed values (two f32 pairs) by IEEE division and
// clamps: the path for a block whose amax is zero, tiny or huge.  Kept out of
// line so that the common path's loop body stays small.
static __device__ __noinline__ uint32_t q8_word_exact(uint64_t p0, uint64_t p1, float d) {
    float v[4];
    f2_unpack(p0, v[0], v[1]);
    f2_unpack(p1, v[2], v[3]);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = static_cast<uint32_t>(d > 0.0f ? min(127, max(-128, __float2int_rn(v[i] / d))) : 0);
    return pack4(c[0], c[1], c[2], c[3]);
}

// Code words of one chunk slot (VEC elements = VEC / 2 f32 pairs), four codes
// to a word: by the block reciprocal (fast) or by IEEE division and clamps.
template <int VEC>
__device__ __forceinline__ void q8_chunk_words(const uint64_t *xn, bool fast, uint64_t id2,
                                               float d, uint32_t *w) {
    constexpr float kRoundShift = 12582912.0f;   // 1.5 * 2^23
    const uint64_t sh2 = f2_pack(kRoundShift, kRoundShift);
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) {
        if (fast) {
            float c0, c1, c2, c3;
            f2_unpack(f2_fma(xn[2 * q], id2, sh2), c0, c1);
            f2_unpack(f2_fma(xn[2 * q + 1], id2, sh2), c2, c3);
            w[q] = pack4(__float_as_uint(c0), __float_as_uint(c1), __float_as_uint(c2),
                         __float_as_uint(c3));
        } else {
            w[q] = q8_word_exact(xn[2 * q], xn[2 * q + 1], d);
        }
    }
}

// Sum of squares of a thread's KB blocks (CH 16-byte chunks each): four
// independent accumulators per half (short dependency chains), added in one
// fixed order.  bf16 squares by the mixed-precision fma (the same sums in
// fewer instructions: measured on GB300, 16384 x 4096 bf16, with the product
// below, 5.38 -> 5.82 TB/s); f32 two lanes at a time.
template <class T, int KB, int CH>
__device__ __forceinline__ float q8_sum_sq(const Frag<T, 16 / T::kBytes> (&xv)[KB][CH]) {
    constexpr int VEC = 16 / T::kBytes;
    float acc_lo[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc_hi[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if constexpr (T::kBytes == 2) {
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int i = 0; i < CH; ++i)
#pragma unroll
                for (int p = 0; p < VEC / 2; ++p) {
                    const uint32_t w = xv[kb][i].w[p];
                    const int j = (i * (VEC / 2) + p) & 3;
                    acc_lo[j] = fma_bf16_lo(w, w, acc_lo[j]);
                    acc_hi[j] = fma_bf16_hi(w, w, acc_hi[j]);
                }
    } else {
        uint64_t acc[4] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f),
                           f2_pack(0.0f, 0.0f)};
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int i = 0; i < CH; ++i)
#pragma unroll
                for (int p = 0; p < VEC / 2; ++p) {
                    const uint64_t xp = frag_pair(xv[kb][i], p);
                    const int j = (i * (VEC / 2) + p) & 3;
                    acc[j] = f2_fma(xp, xp, acc[j]);
                }
#pragma unroll
        for (int j = 0; j < 4; ++j) f2_unpack(acc[j], acc_lo[j], acc_hi[j]);
    }
    return ((acc_lo[0] + acc_hi[0]) + (acc_lo[1] + acc_hi[1])) +
           ((acc_lo[2] + acc_hi[2]) + (acc_lo[3] + acc_hi[3]));
}

// x * gamma of elements 2p and 2p + 1 of two chunks as an f32 pair, exact
// (bf16: the mixed-precision fma with -0 keeps the sign of a zero product).
template <class T>
__device__ __forceinline__ uint64_t q8_x_gamma(const Frag<T, 16 / T::kBytes> &x,
                                               const Frag<T, 16 / T::kBytes> &g, int p) {
    if constexpr (T::kBytes == 2) {
        return f2_pack(fma_bf16_lo(x.w[p], g.w[p], -0.0f), fma_bf16_hi(x.w[p], g.w[p], -0.0f));
    } else {
        return f2_mul(frag_pair(x, p), frag_pair(g, p));
    }
}

template <class T, int KB>
__global__ void __launch_bounds__(kQ8BlockMaxThreads)
mrn_q8_block_kernel(const KernelArgs a) {
    constexpr int VEC = 16 / T::kBytes;       // elements per 16-byte chunk
    constexpr int CH = kQ8Block / VEC;        // chunks per block
    constexpr int NP = kQ8Block / 2;          // f32 pairs per block
    extern __shared__ __align__(16) unsigned char q8_row[];   // the row's blocks
    __shared__ ReduceSlots slots;
    pdl_enter();
    const int64_t row = a.row0 + blockIdx.x;
    const int nb = static_cast<int>(a.n / kQ8Block);
    const int tid = threadIdx.x;
    const char *xr = static_cast<const char *>(a.x) + row * a.n * T::kBytes;
    const char *gr = static_cast<const char *>(a.g1);

    Frag<T, VEC> xv[KB][CH];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        const int b = tid + k * static_cast<int>(blockDim.x);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            if (b < nb) {
                ld_ro(xv[k][c], xr + (static_cast<int64_t>(b) * CH + c) * 16);
            } else {
                xv[k][c].zero();
            }
        }
    }
    const float part = q8_sum_sq<T, KB, CH>(xv);
    const float inv = inv_rms(cta_allsum(part, slots, 1, 0, false), a.n, a.eps1);
    const uint64_t inv2 = f2_pack(inv, inv);

#pragma unroll
    for (int k = 0; k < KB; ++k) {
        const int b = tid + k * static_cast<int>(blockDim.x);
        if (b >= nb) continue;
        uint64_t xn[NP];
        float m[NP];   // per-pair maxima, then a max tree (short chains)
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            Frag<T, VEC> g;
            ld_ro(g, gr + (static_cast<int64_t>(b) * CH + c) * 16);
#pragma unroll
            for (int p = 0; p < VEC / 2; ++p) {
                // x_normed = (x * gamma) * inv, the page's product order
                const uint64_t v = f2_mul(q8_x_gamma<T>(xv[k][c], g, p), inv2);
                xn[c * (VEC / 2) + p] = v;
                float lo, hi;
                f2_unpack(v, lo, hi);
                m[c * (VEC / 2) + p] = fmaxf(fabsf(lo), fabsf(hi));
            }
        }
#pragma unroll
        for (int w = NP / 2; w > 0; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
        const float amax = m[0];
        const bool fast = amax >= 0x1p-100f && amax <= 0x1p100f;
        const float d = amax / 127.0f;
        const float id = fast ? __fdividef(127.0f, amax) : 0.0f;
        const uint64_t id2 = f2_pack(id, id);
        uint32_t *dst = reinterpret_cast<uint32_t *>(q8_row + b * kQ8BlockBytes);
        dst[0] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(d)));
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            uint32_t w[VEC / 4];
            q8_chunk_words<VEC>(xn + c * (VEC / 2), fast, id2, d, w);
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) dst[1 + c * (VEC / 4) + q] = w[q];
        }
    }
    __syncthreads();
    // The row's blocks, shared -> global: 16-byte stores where the row allows.
    const int64_t bytes = static_cast<int64_t>(nb) * kQ8BlockBytes;
    char *out = static_cast<char *>(a.y) + row * bytes;
    if ((bytes & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
        for (int64_t i = tid; i < bytes / 16; i += blockDim.x) {
            const uint4 v = *reinterpret_cast<const uint4 *>(q8_row + i * 16);
            asm volatile(MRN_ST_OP ".v4.u32 [%0], {%1,%2,%3,%4};"
                         :: "l"(out + i * 16), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
        }
    } else {
        for (int64_t i = tid; i < bytes / 4; i += blockDim.x) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(q8_row + i * 4);
            asm volatile(MRN_ST_OP ".u32 [%0], %1;" :: "l"(out + i * 4), "r"(v) : "memory");
        }
    }
}

template <class T>
cudaError_t launch_q8_blocks(const Geometry &g, KernelArgs a, int64_t rows, cudaStream_t stream,
                             uint64_t *launches) {
    using Fn = void (*)(KernelArgs);
    const Fn fn = g.k == 1 ? mrn_q8_block_kernel<T, 1> : mrn_q8_block_kernel<T, 2>;
    const size_t shared = static_cast<size_t>(a.n / kQ8Block) * kQ8BlockBytes;
    for (int64_t r0 = 0; r0 < rows; r0 += kRowsPerLaunch) {
        const int64_t nrows = rows - r0 < kRowsPerLaunch ? rows - r0 : kRowsPerLaunch;
        a.row0 = r0;
        a.rows_end = r0 + nrows;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(static_cast<unsigned>(nrows), 1, 1);
        cfg.blockDim = dim3(g.threads, 1, 1);
        cfg.dynamicSmemBytes = shared;
        cfg.stream = stream;
        if (g.pdl) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        const cudaError_t err = cudaLaunchKernelEx(&cfg, fn, a);
        if (err != cudaSuccess) return err;
        ++*launches;
    }
    return cudaSuccess;
}

// Staged form of the same: persistent CTAs of G warp groups; each row's x is
// copied into a shared-memory stage by cp.async.bulk (the stage ring, waits,
// refill and abort of mrn_tma_kernel) and gamma once per CTA.  A thread reads
// its blocks' 16-byte chunks from the stage in an order rotated by its lane,
// so that the eight lanes of a 16-byte shared load touch eight different
// bank groups; register slot i then holds chunk (i + rot) % CH, and its codes
// are written at that chunk's offset.  Each group assembles its row's blocks
// in its own shared-memory buffer; one thread then copies the row out with a
// single bulk copy (cp.async.bulk shared -> global) when the row's bytes and
// address are 16-byte multiples, else the group copies it word by word.

template <class T, int KB, int G>
__global__ void __launch_bounds__(G * kQ8TmaGroupThreads, 1)
mrn_q8_tma_kernel(const KernelArgs a, const int stages) {
    constexpr int VEC = 16 / T::kBytes;   // elements per chunk
    constexpr int CH = kQ8Block / VEC;    // chunks per block: 4 or 8
    constexpr int NP = kQ8Block / 2;      // f32 pairs per block
    using Fr = Frag<T, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ ReduceSlots slots[G];
    __shared__ __align__(8) uint64_t bars[kTmaMaxStages + 1];   // [stages] = gamma
    __shared__ int issued[kTmaMaxStages];
    __shared__ int consumed[kTmaMaxStages];
    __shared__ volatile int abort_flag;

    const uint32_t rb = static_cast<uint32_t>(a.n * T::kBytes);
    const int nb = static_cast<int>(a.n / kQ8Block);
    const int64_t outb = q8_out_stride(nb);
    unsigned char *const gsm = smem;
    unsigned char *const stage0 = smem + rb;
    unsigned char *const outs = stage0 + static_cast<int64_t>(stages) * rb;
    const int tid = threadIdx.x;
    const int gsize = blockDim.x / G;
    const int grp = tid / gsize;
    const int gtid = tid - grp * gsize;
    const int bar_id = 1 + grp;
    const int rot = static_cast<int>(threadIdx.x & 7) / (8 / CH);
    const int64_t first = a.row0 + blockIdx.x;
    const int64_t step = gridDim.x;
    const int64_t my_rows = first < a.rows_end ? (a.rows_end - first + step - 1) / step : 0;
    const int64_t row_bytes = a.n * T::kBytes;
    const char *const xg = static_cast<const char *>(a.x);
    if (stages < G || stages > kTmaMaxStages || stages % G != 0) {
        // The host never launches this; refuse rather than start any copy.
        if (tid == 0) atomicAdd(&g_wait_timeouts, 1u);
        return;
    }

    if (tid == 0) {
        for (int s = 0; s <= stages; ++s) mbar_init(&bars[s], 1);
        for (int s = 0; s < kTmaMaxStages; ++s) issued[s] = consumed[s] = 0;
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_enter();   // (the shared-memory set-up above overlapped the previous grid)
    if (tid == 0 && my_rows > 0) {
        mbar_arrive_expect_tx(&bars[stages], rb + a.stall_bytes);   // (test hook: 0)
        bulk_to_shared(gsm, a.g1, rb, &bars[stages]);
        for (int s = 0; s < stages && s < my_rows; ++s) {
            stage_row<1>(stage0 + s * rb, xg, nullptr, (first + s * step) * row_bytes, rb, rb,
                         &bars[s]);
            issued[s] = 1;
        }
    }
    int failed = (my_rows > 0 && !mbar_wait_bounded(&bars[stages], 0)) ? 1 : 0;

    for (int64_t it = grp; it < my_rows; it += G) {
        const int s = static_cast<int>(it % stages);
        const uint32_t parity = static_cast<uint32_t>((it / stages) & 1);
        const int64_t row = first + it * step;
        if (!failed && !mbar_wait_bounded(&bars[s], parity)) failed = 1;

        const unsigned char *sp = stage0 + static_cast<int64_t>(s) * rb;
        Fr xv[KB][CH];
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const int b = gtid + kb * gsize;
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int cc = (i + rot) & (CH - 1);
                if (b < nb) {
                    ld_shared(xv[kb][i], sp + (static_cast<int64_t>(b) * CH + cc) * 16);
                } else {
                    xv[kb][i].zero();
                }
            }
        }
        const float part = q8_sum_sq<T, KB, CH>(xv);
        // the previous row's bulk copy has read the group's block buffer
        if (gtid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        int any_failed;
        const float tot = wg_allsum<true>(part, slots[grp], bar_id, gsize, gtid,
                                          failed | abort_flag, &any_failed);
        if (any_failed) {
            if (gtid == 0) abort_flag = 1;
            break;
        }
        // Every thread of the group holds its part of the stage now: refill it.
        if (gtid == 0) {
            consumed[s] += 1;
            if (it + stages < my_rows) {
                fence_proxy_async_smem();
                stage_row<1>(stage0 + s * rb, xg, nullptr,
                             (first + (it + stages) * step) * row_bytes, rb, rb, &bars[s]);
                issued[s] += 1;
            }
        }
        const float inv = inv_rms(tot, a.n, a.eps1);
        const uint64_t inv2 = f2_pack(inv, inv);
        unsigned char *const ob = outs + grp * outb;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const int b = gtid + kb * gsize;
            if (b >= nb) continue;
            uint64_t xn[NP];
            float m[NP];   // per-pair maxima, then a max tree (short chains)
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int cc = (i + rot) & (CH - 1);
                Fr g;
                ld_shared(g, gsm + (static_cast<int64_t>(b) * CH + cc) * 16);
#pragma unroll
                for (int p = 0; p < VEC / 2; ++p) {
                    // x_normed = (x * gamma) * inv, the page's product order
                    const uint64_t v = f2_mul(q8_x_gamma<T>(xv[kb][i], g, p), inv2);
                    xn[i * (VEC / 2) + p] = v;
                    float lo, hi;
                    f2_unpack(v, lo, hi);
                    m[i * (VEC / 2) + p] = fmaxf(fabsf(lo), fabsf(hi));
                }
            }
#pragma unroll
            for (int w = NP / 2; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
            const float amax = m[0];
            const bool fast = amax >= 0x1p-100f && amax <= 0x1p100f;
            const float d = amax / 127.0f;
            const float id = fast ? __fdividef(127.0f, amax) : 0.0f;
            const uint64_t id2 = f2_pack(id, id);
            unsigned char *const blk = ob + b * kQ8BlockBytes;
            *reinterpret_cast<uint32_t *>(blk) =
                static_cast<uint32_t>(__half_as_ushort(__float2half_rn(d)));
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int cc = (i + rot) & (CH - 1);
                uint32_t w[VEC / 4];
                q8_chunk_words<VEC>(xn + i * (VEC / 2), fast, id2, d, w);
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q)
                    *reinterpret_cast<uint32_t *>(blk + 4 + cc * VEC + 4 * q) = w[q];
            }
        }
        const int64_t bytes = static_cast<int64_t>(nb) * kQ8BlockBytes;
        char *const out = static_cast<char *>(a.y) + row * bytes;
        const bool bulk = (bytes & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
        if (bulk) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        group_sync(bar_id, gsize);   // the group's blocks of this row are complete
        if (bulk) {
            if (gtid == 0) {
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
                             "cp.async.bulk.commit_group;"
                             :: "l"(out), "r"(smem_addr(ob)), "r"(static_cast<uint32_t>(bytes))
                             : "memory");
            }
        } else {
            for (int64_t i = gtid; i < bytes / 4; i += gsize) {
                const uint32_t v = *reinterpret_cast<const uint32_t *>(ob + i * 4);
                asm volatile(MRN_ST_OP ".u32 [%0], %1;" :: "l"(out + i * 4), "r"(v) : "memory");
            }
        }
        // (the next row writes this buffer only after its first reduction's
        // barrier, which every thread of the group reaches after this copy, and
        // which the issuing thread enters only once the bulk copy has read it)
    }

    // Exit: as mrn_tma_kernel -- after a failure, wait (bounded) for the
    // copies still in flight before the CTA leaves its shared memory.
    if (gtid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncthreads();
    if (tid == 0 && my_rows > 0 && abort_flag) {
        atomicAdd(&g_wait_timeouts, 1u);
        (void)mbar_wait_bounded(&bars[stages], 0);
        for (int s = 0; s < stages; ++s) {
            if (issued[s] > consumed[s])
                (void)mbar_wait_bounded(&bars[s], static_cast<uint32_t>(consumed[s] & 1));
        }
    }
}


template <class T>
cudaError_t launch_q8_tma(const Geometry &g, KernelArgs a, int64_t rows, cudaStream_t stream,
                          uint64_t *launches) {
    static TmaLaunchCache cache[kMaxCachedDevices][2][2];   // [groups - 1][k - 1]
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    TmaLaunchCache uncached;
    TmaLaunchCache &c =
        (dev >= 0 && dev < kMaxCachedDevices) ? cache[dev][g.groups - 1][g.k - 1] : uncached;
    using Fn = void (*)(KernelArgs, int);
    Fn fn;
    if (g.groups == 1) {
        fn = g.k == 1 ? mrn_q8_tma_kernel<T, 1, 1> : mrn_q8_tma_kernel<T, 2, 1>;
    } else {
        fn = g.k == 1 ? mrn_q8_tma_kernel<T, 1, 2> : mrn_q8_tma_kernel<T, 2, 2>;
    }
    const int64_t shared = q8_tma_shared_bytes(a.n, T::kBytes, g.stages, g.groups);
    cudaError_t err;
    if (c.shared_opened.load(std::memory_order_relaxed) < shared) {
        err = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(shared));
        if (err != cudaSuccess) return err;
        c.shared_opened.store(shared, std::memory_order_relaxed);
    }
    int64_t ctas = g.ctas;
    if (ctas <= 0) {
        const int64_t key = shared * 2048 + g.threads;
        int per_sm = c.occ_key.load(std::memory_order_relaxed) == key
                         ? c.occ_per_sm.load(std::memory_order_relaxed) : 0;
        if (per_sm == 0) {
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, g.threads,
                                                                static_cast<size_t>(shared));
            if (err != cudaSuccess) return err;
            if (per_sm < 1) return cudaErrorInvalidConfiguration;
            c.occ_per_sm.store(per_sm, std::memory_order_relaxed);
            c.occ_key.store(key, std::memory_order_relaxed);
        }
        ctas = static_cast<int64_t>(device_sm_count()) * per_sm;
        if (ctas < 1) return cudaErrorInvalidDevice;
    }
    for (int64_t r0 = 0; r0 < rows; r0 += kRowsPerLaunch) {
        const int64_t nrows = rows - r0 < kRowsPerLaunch ? rows - r0 : kRowsPerLaunch;
        a.row0 = r0;
        a.rows_end = r0 + nrows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas < nrows ? ctas : nrows), 1, 1);
        cfg.blockDim = dim3(g.threads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(shared);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        if (g.pdl) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        err = cudaLaunchKernelEx(&cfg, fn, a, g.stages);
        if (err != cudaSuccess) return err;
        ++*launches;
    }
    return cudaSuccess;
}

}  // namespace mrn
