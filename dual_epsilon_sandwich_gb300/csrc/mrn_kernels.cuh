// mrn_kernels.cuh -- sm_103a kernels for RMSNorm, post-norm-then-add, the
// dual-epsilon sandwich tail and the operations built on the same row
// reduction (residual add + norm, then-add-scale, RMSNorm + Q8_1, the
// split-norm seam).
//
// The computation ("Chapter 12 -- RMSNorm and the dual-epsilon sandwich",
// sections 12.1, 12.4.3 and 12.7; Hesper "RMSNorm Layer", rmsNormThenAddKernel
// and the kernels named at each operation below):
//   inv = 1 / sqrt(sum_j v_j^2 / n + eps)            (f32, IEEE sqrt and divide)
//   rmsnorm   y = (x * inv) * gamma
//   then-add  out = fma(x * inv, gamma, residual)
//   sandwich  s = fma(b * inv(b; eps_post), gamma_post, residual)   -> stored
//             normed = (s * inv(s; eps_pre)) * gamma_pre           (s as stored)
//
// Design for a bandwidth-bound row reduction on GB300:
//  * every operand element is read from HBM once and every output written
//    once: the row (and the residual) stay in registers (or a shared-memory
//    stage) between the reduction and the output pass;
//  * 16-byte vector loads/stores (4 x f32 or 8 x bf16), consecutive lanes on
//    consecutive vectors, so a warp moves 512 contiguous bytes per access;
//    streaming operands bypass L1 (L1::no_allocate) and ask L2 for 256-byte
//    prefetch; gamma goes through the read-only path and stays cached;
//  * reductions: butterfly shuffles (every lane ends with the same bits),
//    then one shared-memory slot per warp, then -- for rows split over a
//    thread-block cluster -- one DSMEM slot per CTA written into every peer
//    and a release/acquire cluster barrier.  Every CTA sums the same partials
//    in the same order, so all CTAs of a row use bit-identical inv;
//  * geometries: several rows per warp (small n), one row per CTA or per
//    cluster (register resident), a looped fallback for rows too wide for
//    registers, persistent CTAs whose rows are bulk-copied (cp.async.bulk)
//    into shared-memory stages ahead of use (the RMSNorm + Q8_1 kernels with
//    whole 32-element blocks per thread are in mrn_q8_kernels.cuh);
//  * every kernel starts with griddepcontrol.wait / launch_dependents, so a
//    launch with programmatic stream serialisation changes no result.
// The only waits are the hardware cluster barrier (reached unconditionally by
// every thread of the cluster) and, in the staged kernels, mbarrier waits on
// their own bulk copies, each bounded in time (see mbar_wait_bounded).
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mrn_internal.h"

// Compile-time cache-policy switches (defaults are the measured best):
//   MRN_STORE_STREAMING  1: outputs stored with .cs (evict-first in L2)
//   MRN_BULK_EVICT_FIRST 1: staged row copies carry an L2 evict-first policy
#ifndef MRN_STORE_STREAMING
#define MRN_STORE_STREAMING 0
#endif
#ifndef MRN_BULK_EVICT_FIRST
#define MRN_BULK_EVICT_FIRST 1
#endif
#if MRN_STORE_STREAMING
#define MRN_ST_OP "st.global.cs"
#else
#define MRN_ST_OP "st.global"
#endif

namespace mrn {

struct F32 { static constexpr int kBytes = 4; };
struct BF16 { static constexpr int kBytes = 2; };

// ---------------------------------------------------------------------------
// Register fragments: VEC elements of one operand, kept as raw bits.
// ---------------------------------------------------------------------------
template <class T, int VEC> struct Frag;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t *>(&v);
}

template <> struct Frag<F32, 4> {
    uint32_t w[4];
    __device__ __forceinline__ void zero() { w[0] = w[1] = w[2] = w[3] = 0u; }
    __device__ __forceinline__ float get(int i) const { return __uint_as_float(w[i]); }
    __device__ __forceinline__ void put(const float (&f)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __float_as_uint(f[i]);
    }
    __device__ __forceinline__ void clear(int i) { w[i] = 0u; }
    // element i stored alone at p
    __device__ __forceinline__ void st_elem(char *p, int i) const {
        asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(w[i]) : "memory");
    }
};

template <> struct Frag<BF16, 8> {
    uint32_t w[4];
    __device__ __forceinline__ void zero() { w[0] = w[1] = w[2] = w[3] = 0u; }
    __device__ __forceinline__ float get(int i) const {
        const uint32_t u = w[i >> 1];
        return (i & 1) ? __uint_as_float(u & 0xFFFF0000u) : __uint_as_float(u << 16);
    }
    __device__ __forceinline__ void put(const float (&f)[8]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
    }
    __device__ __forceinline__ void clear(int i) { w[i >> 1] &= (i & 1) ? 0x0000FFFFu : 0xFFFF0000u; }
    __device__ __forceinline__ void st_elem(char *p, int i) const {
        const unsigned short h = static_cast<unsigned short>((i & 1) ? (w[i >> 1] >> 16)
                                                                     : (w[i >> 1] & 0xFFFFu));
        asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(h) : "memory");
    }
};

template <> struct Frag<F32, 1> {
    uint32_t w;
    __device__ __forceinline__ void zero() { w = 0u; }
    __device__ __forceinline__ float get(int) const { return __uint_as_float(w); }
    __device__ __forceinline__ void put(const float (&f)[1]) { w = __float_as_uint(f[0]); }
};

template <> struct Frag<BF16, 1> {
    unsigned short h;
    __device__ __forceinline__ void zero() { h = 0; }
    __device__ __forceinline__ float get(int) const {
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ __forceinline__ void put(const float (&f)[1]) {
        h = __bfloat16_as_ushort(__float2bfloat16_rn(f[0]));
    }
};

// Two f32 lanes per instruction (mul.rn.f32x2 / fma.rn.f32x2: each half
// rounded exactly as the scalar instruction would), on register pairs.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// Mixed-precision fma of the bf16 halves of two words into an f32 accumulator:
// d = a * b + c with the bf16 operands taken exactly (their product is exact
// in f32; one rounding with c), i.e. fmaf(float(a), float(b), c) without
// widening the halves first.  lo: the low halves, hi: the high halves.
__device__ __forceinline__ float fma_bf16_lo(uint32_t wa, uint32_t wb, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}" : "=f"(d) : "r"(wa), "r"(wb), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t wa, uint32_t wb, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}" : "=f"(d) : "r"(wa), "r"(wb), "f"(c));
    return d;
}
// Elements 2p and 2p + 1 of a 16-byte fragment as an f32 pair.
__device__ __forceinline__ uint64_t frag_pair(const Frag<BF16, 8> &f, int p) {
    const uint32_t w = f.w[p];
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint64_t frag_pair(const Frag<F32, 4> &f, int p) {
    return f2_pack(__uint_as_float(f.w[2 * p]), __uint_as_float(f.w[2 * p + 1]));
}
// ---------------------------------------------------------------------------
// Global memory access.  `stream` = operand read once (bypass L1, 256-byte L2
// prefetch); `ro` = read-only, cached (gamma); `st` = plain store; `ld` =
// plain coherent load (re-reading data this thread stored earlier).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_stream(Frag<F32, 4> &f, const void *p) {
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_stream(Frag<BF16, 8> &f, const void *p) {
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_stream(Frag<F32, 1> &f, const void *p) {
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(f.w) : "l"(p));
}
__device__ __forceinline__ void ld_stream(Frag<BF16, 1> &f, const void *p) {
    asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(f.h) : "l"(p));
}

// Streaming loads and stores with an L2 eviction-priority policy (the looped
// kernel: a slice read twice is kept in L2 by its first read and released by
// its last).  The policy is a createpolicy descriptor.
__device__ __forceinline__ uint64_t l2_policy_keep() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_drop() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void ld_hint(Frag<F32, 4> &f, const void *p, uint64_t pol) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void ld_hint(Frag<BF16, 8> &f, const void *p, uint64_t pol) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void ld_hint(Frag<F32, 1> &f, const void *p, uint64_t pol) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                 : "=r"(f.w) : "l"(p), "l"(pol) : "memory");
}
__device__ __forceinline__ void ld_hint(Frag<BF16, 1> &f, const void *p, uint64_t pol) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;"
                 : "=h"(f.h) : "l"(p), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(void *p, const Frag<F32, 4> &f, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(f.w[0]), "r"(f.w[1]), "r"(f.w[2]), "r"(f.w[3]), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(void *p, const Frag<BF16, 8> &f, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(f.w[0]), "r"(f.w[1]), "r"(f.w[2]), "r"(f.w[3]), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(void *p, const Frag<F32, 1> &f, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" :: "l"(p), "r"(f.w), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(void *p, const Frag<BF16, 1> &f, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u16 [%0], %1, %2;" :: "l"(p), "h"(f.h), "l"(pol) : "memory");
}

__device__ __forceinline__ void ld_ro(Frag<F32, 4> &f, const void *p) {
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_ro(Frag<BF16, 8> &f, const void *p) {
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_ro(Frag<F32, 1> &f, const void *p) {
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(f.w) : "l"(p));
}
__device__ __forceinline__ void ld_ro(Frag<BF16, 1> &f, const void *p) {
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(f.h) : "l"(p));
}

__device__ __forceinline__ void ld_plain(Frag<F32, 4> &f, const void *p) {
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p) : "memory");
}
__device__ __forceinline__ void ld_plain(Frag<BF16, 8> &f, const void *p) {
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p) : "memory");
}
__device__ __forceinline__ void ld_plain(Frag<F32, 1> &f, const void *p) {
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(f.w) : "l"(p) : "memory");
}
__device__ __forceinline__ void ld_plain(Frag<BF16, 1> &f, const void *p) {
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(f.h) : "l"(p) : "memory");
}

__device__ __forceinline__ void st_global(void *p, const Frag<F32, 4> &f) {
    asm volatile(MRN_ST_OP ".v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(f.w[0]), "r"(f.w[1]), "r"(f.w[2]), "r"(f.w[3]) : "memory");
}
__device__ __forceinline__ void st_global(void *p, const Frag<BF16, 8> &f) {
    asm volatile(MRN_ST_OP ".v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(f.w[0]), "r"(f.w[1]), "r"(f.w[2]), "r"(f.w[3]) : "memory");
}
__device__ __forceinline__ void st_global(void *p, const Frag<F32, 1> &f) {
    asm volatile(MRN_ST_OP ".u32 [%0], %1;" :: "l"(p), "r"(f.w) : "memory");
}
__device__ __forceinline__ void st_global(void *p, const Frag<BF16, 1> &f) {
    asm volatile(MRN_ST_OP ".u16 [%0], %1;" :: "l"(p), "h"(f.h) : "memory");
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
// Butterfly sum over `width` lanes (a power of two <= 32).  Both operands of
// every addition are the same on the two partner lanes and f32 addition is
// commutative, so all lanes of a group end with bit-identical sums.
__device__ __forceinline__ float group_allsum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ unsigned cluster_nctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_index_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_count_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store v into the shared-memory word `local` of CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_f32(float *local, unsigned rank, float v) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(local));
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(remote), "f"(v) : "memory");
}

// Store v into the shared-memory word `local` of CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_u32(int *local, unsigned rank, int v) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(local));
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(remote), "r"(v) : "memory");
}

struct ReduceSlots {
    float warp[32];
    float cta[kMaxCluster];
};

// Sum of v over all threads of the CTA and, when cl > 1, over all CTAs of
// the cluster.  Every thread of every CTA must call it (it contains
// __syncthreads and cluster barriers).  `first` marks the first cluster
// reduction of the kernel: it completes the arrive issued at kernel start,
// which guarantees every peer CTA is running before its shared memory is
// written.
__device__ __forceinline__ float cta_allsum(float v, ReduceSlots &s, unsigned cl, unsigned crank,
                                            bool first) {
    v = warp_allsum(v);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (lane == 0) s.warp[warp] = v;
    __syncthreads();
    float t = warp_allsum(lane < nwarps ? s.warp[lane] : 0.0f);
    if (cl > 1) {
        if (first) cluster_wait_acquire();
        if (threadIdx.x < cl) st_cluster_f32(&s.cta[crank], threadIdx.x, t);
        cluster_arrive_release();
        cluster_wait_acquire();
        t = warp_allsum(lane < static_cast<int>(cl) ? s.cta[lane] : 0.0f);
    }
    return t;
}

// Programmatic dependent launch.  Every kernel waits for the grid it depends
// on (the previous kernel on the stream) to complete and publish its memory --
// a no-op unless the launch allowed programmatic serialisation -- before its
// first global memory access, and then lets its own dependent grid be
// scheduled, so that the next launch's set-up overlaps this kernel instead of
// following it.  The staged kernels initialise their shared memory and
// mbarriers before the wait.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float inv_rms(float sum_sq, int64_t n, float eps) {
    return 1.0f / sqrtf(sum_sq / static_cast<float>(n) + eps);
}

template <class T, int VEC>
__device__ __forceinline__ float frag_sum_sq(const Frag<T, VEC> &f) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) s = fmaf(f.get(i), f.get(i), s);
    return s;
}

template <class T> __device__ __forceinline__ const char *elem_ptr(const void *base, int64_t e) {
    return static_cast<const char *>(base) + e * T::kBytes;
}
template <class T> __device__ __forceinline__ char *elem_ptr(void *base, int64_t e) {
    return static_cast<char *>(base) + e * T::kBytes;
}

// y = (x * inv) * g
template <class T, int VEC>
__device__ __forceinline__ Frag<T, VEC> apply_norm(const Frag<T, VEC> &x, float inv,
                                                    const Frag<T, VEC> &g) {
    float o[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] = (x.get(i) * inv) * g.get(i);
    Frag<T, VEC> r;
    r.put(o);
    return r;
}

// out = fma(x * inv, g, r)
template <class T, int VEC>
__device__ __forceinline__ Frag<T, VEC> apply_norm_add(const Frag<T, VEC> &x, float inv,
                                                        const Frag<T, VEC> &g,
                                                        const Frag<T, VEC> &r) {
    float o[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] = fmaf(x.get(i) * inv, g.get(i), r.get(i));
    Frag<T, VEC> out;
    out.put(o);
    return out;
}

// out = fma(x * inv, g, r) * scale   (then-add-then-broadcast-scale)
template <class T, int VEC>
__device__ __forceinline__ Frag<T, VEC> apply_norm_add_scale(const Frag<T, VEC> &x, float inv,
                                                              const Frag<T, VEC> &g,
                                                              const Frag<T, VEC> &r, float sc) {
    float o[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] = fmaf(x.get(i) * inv, g.get(i), r.get(i)) * sc;
    Frag<T, VEC> out;
    out.put(o);
    return out;
}

// s = a + b, rounded once to T   (the residual add of add+norm)
template <class T, int VEC>
__device__ __forceinline__ Frag<T, VEC> add_frags(const Frag<T, VEC> &a, const Frag<T, VEC> &b) {
    float o[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] = a.get(i) + b.get(i);
    Frag<T, VEC> out;
    out.put(o);
    return out;
}

// The broadcast scale of then-add-scale (one element of type T), as f32.
template <int OP, class T>
__device__ __forceinline__ float load_out_scale(const void *p) {
    if (OP != kThenAddScale) return 1.0f;
    Frag<T, 1> f;
    ld_ro(f, p);
    return f.get(0);
}

// The output of the single-norm operations for one fragment.
template <int OP, class T, int VEC>
__device__ __forceinline__ Frag<T, VEC> single_norm_output(const Frag<T, VEC> &x, float inv,
                                                           const Frag<T, VEC> &g,
                                                           const Frag<T, VEC> &r, float sc) {
    if (OP == kRmsnorm) return apply_norm(x, inv, g);
    if (OP == kThenAdd) return apply_norm_add(x, inv, g, r);
    return apply_norm_add_scale(x, inv, g, r, sc);
}

// RMSNorm + Q8_1 output of one fragment (Hesper fusedRMSNormQ8_1Kernel):
// x_normed = (x * gamma) * inv; a 32-element block is held by VPB = 32/VEC
// consecutive lanes (one register slot each), which agree on the block's
// amax by a butterfly max; d = amax / 127; q = x_normed / d rounded to
// nearest, ties to even, clamped to int8 (0 when d == 0).
//
// The quotient is formed as x_normed * (127 / amax), the reciprocal taken
// once per block by the approximate divide: it can differ from x_normed / d
// only within a few f32 ulps of a rounding tie.  Rounding to the nearest integer,
// ties to even, is one fused multiply-add: fma(x_normed, 127/amax, 1.5 * 2^23)
// lands in [2^23, 2^24), where the f32 spacing is exactly 1, so the single
// rounding of the fma is the integer rounding and the low byte of the
// result's bits is the two's-complement code (|x_normed * 127/amax| <= 127.5
// by construction, so no clamp is needed on this path).  For an amax outside
// [2^-100, 2^100] (zero, tiny or huge) the codes fall back to per-element
// IEEE division and an explicit clamp.  Lane 0 of the block writes the header (f16 d,
// f16 s = 0), every lane its VEC codes.  Every lane of the warp must call
// this (it shuffles); `valid` only gates the stores.  v is the fragment's
// index within the row.
template <class T, int VEC>
__device__ __forceinline__ void q8_1_output(const Frag<T, VEC> &x, const Frag<T, VEC> &g,
                                            float inv, bool valid, char *row_blocks,
                                            int64_t v) {
    static_assert(VEC == 1 || VEC % 4 == 0, "codes are stored one byte or whole words at a time");
    constexpr int VPB = kQ8Block / VEC;
    constexpr float kRoundShift = 12582912.0f;   // 1.5 * 2^23
    float xn[VEC];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        xn[i] = (x.get(i) * g.get(i)) * inv;
        amax = fmaxf(amax, fabsf(xn[i]));
    }
#pragma unroll
    for (int o = VPB / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (!valid) return;
    uint32_t code[VEC];   // the code in the low byte
    if (amax >= 0x1p-100f && amax <= 0x1p100f) {
        // 127/amax by the approximate divide (within 2 ulp for a divisor in
        // [2^-126, 2^126]); the quotient moves by a few ulps at most.
        const float id = __fdividef(127.0f, amax);
#pragma unroll
        for (int i = 0; i < VEC; ++i) code[i] = __float_as_uint(fmaf(xn[i], id, kRoundShift));
    } else {
        const float d = amax / 127.0f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int q = d > 0.0f ? min(127, max(-128, __float2int_rn(xn[i] / d))) : 0;
            code[i] = static_cast<uint32_t>(q);
        }
    }
    uint32_t packed[(VEC + 3) / 4];
    if (VEC >= 4) {
#pragma unroll
        for (int w = 0; w < VEC / 4; ++w) {
            const uint32_t lo = __byte_perm(code[4 * w], code[4 * w + 1], 0x0040);
            const uint32_t hi = __byte_perm(code[4 * w + 2], code[4 * w + 3], 0x0040);
            packed[w] = __byte_perm(lo, hi, 0x5410);
        }
    } else {
        packed[0] = code[0] & 0xFFu;
    }
    const uint64_t uv = static_cast<uint64_t>(v);   // v >= 0
    char *block = row_blocks + (uv / VPB) * kQ8BlockBytes;
    const int j = static_cast<int>(uv % VPB);
    if (j == 0) {
        const float d = amax / 127.0f;
        const uint32_t header = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(d)));
        asm volatile("st.global.u32 [%0], %1;" :: "l"(block), "r"(header) : "memory");
    }
    char *codes = block + 4 + j * VEC;
    if (VEC >= 4) {
#pragma unroll
        for (int w = 0; w < VEC / 4; ++w)
            asm volatile("st.global.u32 [%0], %1;" :: "l"(codes + 4 * w), "r"(packed[w])
                         : "memory");
    } else {
        const unsigned short b = static_cast<unsigned short>(packed[0] & 0xFFu);
        asm volatile("st.global.u8 [%0], %1;" :: "l"(codes), "h"(b) : "memory");
    }
}

// First byte of a row's Q8_1 blocks.
__device__ __forceinline__ char *q8_row_blocks(const KernelArgs &a, int64_t row) {
    return static_cast<char *>(a.y) + row * (a.n / kQ8Block) * kQ8BlockBytes;
}

// ---------------------------------------------------------------------------
// Split-norm seam ("Chapter 12 -- RMSNorm and the dual-epsilon sandwich",
// section 12.7, the cross-vendor seam): the weightless norm is published in a
// 16-bit format S (binary16 or bf16), u = S(x * inv), and the weighted forms
// apply the weight as a second S operation, y = S(u * gamma) with gamma given
// in S: the S multiply (mul.rn.f16x2 / mul.rn.bf16x2, subnormals kept)
// rounds the exact product of the two S values once.
// ---------------------------------------------------------------------------
template <int VEC> struct H16 {   // VEC 16-bit values, two per word (low first)
    uint32_t w[(VEC + 1) / 2];
};

template <bool BF> __device__ __forceinline__ uint32_t seam_pack2(float lo, float hi) {
    if (BF) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <bool BF> __device__ __forceinline__ uint32_t seam_pack1(float v) {
    if (BF) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return __half_as_ushort(__float2half_rn(v));
}
// Exact f32 value of the low / high S value of a word.
template <bool BF> __device__ __forceinline__ float seam_lo(uint32_t w) {
    if (BF) return __uint_as_float(w << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
template <bool BF> __device__ __forceinline__ float seam_hi(uint32_t w) {
    if (BF) return __uint_as_float(w & 0xFFFF0000u);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// gamma of the seam (read-only, cached), the split route's u (streamed), and
// the 16-bit output.
__device__ __forceinline__ void ld_h16(H16<8> &f, const void *p) {
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_h16(H16<4> &f, const void *p) {
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(f.w[0]), "=r"(f.w[1]) : "l"(p));
}
__device__ __forceinline__ void ld_h16(H16<1> &f, const void *p) {
    unsigned short h;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(h) : "l"(p));
    f.w[0] = h;
}
__device__ __forceinline__ void ld_stream_h16(H16<8> &f, const void *p) {
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "l"(p));
}
__device__ __forceinline__ void ld_stream_h16(H16<1> &f, const void *p) {
    unsigned short h;
    asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(h) : "l"(p));
    f.w[0] = h;
}
__device__ __forceinline__ void st_h16(void *p, const H16<8> &f) {
    asm volatile(MRN_ST_OP ".v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(f.w[0]), "r"(f.w[1]), "r"(f.w[2]), "r"(f.w[3]) : "memory");
}
__device__ __forceinline__ void st_h16(void *p, const H16<4> &f) {
    asm volatile(MRN_ST_OP ".v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(f.w[0]), "r"(f.w[1])
                 : "memory");
}
__device__ __forceinline__ void st_h16(void *p, const H16<1> &f) {
    const unsigned short h = static_cast<unsigned short>(f.w[0] & 0xFFFFu);
    asm volatile(MRN_ST_OP ".u16 [%0], %1;" :: "l"(p), "h"(h) : "memory");
}

// Two S products in one instruction: the IEEE multiply of the format,
// round to nearest even.
template <bool BF> __device__ __forceinline__ uint32_t seam_mul2(uint32_t u, uint32_t g) {
    uint32_t r;
    if (BF) {
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(u), "r"(g));
    } else {
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(u), "r"(g));
    }
    return r;
}

// S(u * gamma) of VEC values of S held two per word (VEC == 1: the low half;
// the high halves are zero and their product is discarded).
template <bool BF, int VEC>
__device__ __forceinline__ H16<VEC> seam_scale_frag(const H16<VEC> &u, const H16<VEC> &g) {
    H16<VEC> out;
#pragma unroll
    for (int i = 0; i < (VEC + 1) / 2; ++i) out.w[i] = seam_mul2<BF>(u.w[i], g.w[i]);
    if (VEC == 1) out.w[0] &= 0xFFFFu;
    return out;
}

// Seam output of one fragment of x at row-element offset e: u = S(x * inv),
// and for the weighted forms y = S(u * gamma); 16-bit values stored at y.
template <int OP, class T, int VEC>
__device__ __forceinline__ void seam_output(const Frag<T, VEC> &x, float inv, const H16<VEC> &g,
                                            void *y, int64_t e) {
    constexpr bool BF = op_seam_bf16(OP);
    H16<VEC> u;
    if constexpr (VEC == 1) {
        u.w[0] = seam_pack1<BF>(x.get(0) * inv);
    } else {
        const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) {
            float lo, hi;
            f2_unpack(f2_mul(frag_pair(x, i), inv2), lo, hi);   // x * inv, two lanes at once
            u.w[i] = seam_pack2<BF>(lo, hi);
        }
    }
    void *p = static_cast<char *>(y) + e * 2;
    if (op_seam_weighted(OP)) {
        st_h16(p, seam_scale_frag<BF, VEC>(u, g));
    } else {
        st_h16(p, u);
    }
}

// ---------------------------------------------------------------------------
// Row body shared by the register-resident kernels.  A "slot" k of this
// thread holds load index v = first + k * stride of the row (masked when
// v >= nvec).  `Reduce` sums a float over all threads of the row.
// ---------------------------------------------------------------------------
template <int OP, class T, int VEC, int K, class Reduce1, class Reduce2>
__device__ __forceinline__ void row_body(const KernelArgs &a, int64_t row, bool row_ok,
                                         int64_t first, int64_t stride, Reduce1 reduce1,
                                         Reduce2 reduce2) {
    using Fr = Frag<T, VEC>;
    const int64_t row_elem = row * a.n;
    Fr xv[K];
    Fr rv[K];
    Fr gv[K];
    bool ok[K];
    // All loads of the row are issued before the first reduction: the row, the
    // residual and the first gamma are in flight together.
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t v = first + k * stride;
        ok[k] = row_ok && v < a.nvec;
        const int64_t e = row_elem + v * VEC;
        if (ok[k]) {
            ld_stream(xv[k], elem_ptr<T>(a.x, e));
            if (op_row_inputs(OP) == 2) ld_stream(rv[k], elem_ptr<T>(a.res, e));
        } else {
            xv[k].zero();
            rv[k].zero();
        }
    }
    H16<VEC> hg[K];   // the seam's 16-bit gamma
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!ok[k]) continue;
        const int64_t ge = (first + k * stride) * VEC;
        if (op_seam_weighted(OP)) {
            ld_h16(hg[k], static_cast<const char *>(a.g1) + ge * 2);
        } else if (!op_is_seam(OP)) {
            ld_ro(gv[k], elem_ptr<T>(a.g1, ge));
        }
    }

    const float sc = load_out_scale<OP, T>(a.scale);

    float ss = 0.0f;
    if (OP == kAddRmsnorm) {
        // residual_out = a + b (rounded to T), stored; its stored value is normed
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (!ok[k]) continue;
            rv[k] = add_frags(xv[k], rv[k]);
            st_global(elem_ptr<T>(a.y, row_elem + (first + k * stride) * VEC), rv[k]);
            ss += frag_sum_sq(rv[k]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) ss += frag_sum_sq(xv[k]);
    }
    const float inv1 = inv_rms(reduce1(ss), a.n, a.eps1);

    if (OP == kAddRmsnorm) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (!ok[k]) continue;
            const int64_t v = first + k * stride;
            st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(rv[k], inv1, gv[k]));
        }
        return;
    }
    if (OP == kRmsnormQ8) {
        char *blocks = q8_row_blocks(a, row);
#pragma unroll
        for (int k = 0; k < K; ++k) {   // no early exit: every lane shuffles
            if (!ok[k]) gv[k].zero();
            q8_1_output(xv[k], gv[k], inv1, ok[k], blocks, first + k * stride);
        }
        return;
    }
    if (op_is_seam(OP)) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (!ok[k]) continue;
            const int64_t v = first + k * stride;
            seam_output<OP, T, VEC>(xv[k], inv1, hg[k], a.y, row_elem + v * VEC);
        }
        return;
    }
    if (OP != kSandwich) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (!ok[k]) continue;
            const int64_t v = first + k * stride;
            st_global(elem_ptr<T>(a.y, row_elem + v * VEC),
                      single_norm_output<OP>(xv[k], inv1, gv[k], rv[k], sc));
        }
        return;
    }

    // Sandwich: stream = fma(b * inv_post, gamma_post, residual), stored, and its
    // stored (rounded) value feeds the second reduction and the pre norm.
    float ss2 = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!ok[k]) continue;
        const int64_t v = first + k * stride;
        rv[k] = apply_norm_add(xv[k], inv1, gv[k], rv[k]);
        st_global(elem_ptr<T>(a.y, row_elem + v * VEC), rv[k]);
        ss2 += frag_sum_sq(rv[k]);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (ok[k]) ld_ro(gv[k], elem_ptr<T>(a.g2, (first + k * stride) * VEC));
    }
    const float inv2 = inv_rms(reduce2(ss2), a.n, a.eps2);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!ok[k]) continue;
        const int64_t v = first + k * stride;
        st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(rv[k], inv2, gv[k]));
    }
}

// Several rows per warp: `lanes` (power of two <= 32) threads per row, K
// register slots each; up to 256 threads per CTA (128 by the automatic choice).
template <int OP, class T, int VEC, int K>
__global__ void __launch_bounds__(kWarpKernelThreads)
mrn_rows_per_warp_kernel(const KernelArgs a, const int lanes) {
    pdl_enter();
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = a.row0 + gtid / lanes;
    const int lane_in_row = threadIdx.x & (lanes - 1);
    auto reduce = [lanes](float v) { return group_allsum(v, lanes); };
    row_body<OP, T, VEC, K>(a, row, row < a.rows_end, lane_in_row, lanes, reduce, reduce);
}

constexpr int kStreamUnroll = 4;   // loads per operand in flight per thread (looped kernel)

// ---------------------------------------------------------------------------
// Persistent, TMA-staged kernel.  Each CTA owns rows blockIdx.x, +gridDim.x,
// ...  and keeps `stages` of them in flight in shared memory: the row (and
// the residual) of a future row arrive by cp.async.bulk while the current
// row is reduced and written, so HBM reads never wait for the reductions.
// The gammas are copied into shared memory once per CTA.  A stage is
// refilled right after the first reduction of the row it held: that
// reduction's barrier is the point after which every thread has moved the
// stage into registers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// One arrival (release at CTA scope: this thread's shared-memory writes are
// visible to threads whose wait completes the phase).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}
// Raise the barrier's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// 4 bytes global -> shared without staging them in registers (cp.async; the
// thread does not wait for them).
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
// Arrive on the barrier once this thread's cp.async copies so far have landed
// (one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_to_shared(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar) {
#if MRN_BULK_EVICT_FIRST
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                 "[%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
                 : "memory");
#else
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
#endif
}

// Every wait on an mbarrier is bounded: about one second of wall time (and
// an iteration cap) after which the wait reports failure.  A failed wait is
// counted in g_wait_timeouts, the CTA agrees on it at its next barrier,
// drains the copies it has in flight (again bounded) and returns without
// writing the row.  With the copies issued here a wait never runs out.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
static __device__ unsigned int g_wait_timeouts;   // one per translation unit

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 28); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}

// Shared-memory loads of staged rows; the memory clobber keeps them ahead of
// the barrier after which the stage is refilled.
__device__ __forceinline__ void ld_shared(Frag<F32, 4> &f, const void *p) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "r"(smem_addr(p))
                 : "memory");
}
__device__ __forceinline__ void ld_shared(Frag<BF16, 8> &f, const void *p) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(f.w[0]), "=r"(f.w[1]), "=r"(f.w[2]), "=r"(f.w[3]) : "r"(smem_addr(p))
                 : "memory");
}

// Copy `bytes` of one row of x (and of the residual when NS == 2, into the
// slot `stride` bytes further on) into a stage.
template <int NS>
__device__ __forceinline__ void stage_row(unsigned char *dst, const char *x, const char *res,
                                          int64_t offset, uint32_t bytes, uint32_t stride,
                                          uint64_t *bar) {
    mbar_arrive_expect_tx(bar, NS * bytes);
    bulk_to_shared(dst, x + offset, bytes, bar);
    if (NS == 2) bulk_to_shared(dst + stride, res + offset, bytes, bar);
}

// Rows that are not 16-byte aligned, in the staged kernel.  A row that starts
// `mis` bytes past a 16-byte boundary is staged as the 16-byte granules that
// cover it: granule v holds the row's bytes [16 v - mis, 16 v - mis + 16).
// Bytes of a granule outside the row (the start of the first granule, the
// end of the last) belong to the neighbouring rows or lie past the operand;
// they are zeroed in registers before any arithmetic and never stored.  Every
// granule lies in the same 16-byte-aligned memory as a byte of the operand,
// so reading it cannot leave the operand's pages.
// Byte range [lo, hi) of granule v that lies inside the row (span = granules).
__device__ __forceinline__ void granule_bounds(int64_t v, int64_t ngran, uint32_t mis,
                                               uint32_t rb, uint32_t *lo, uint32_t *hi) {
    *lo = v == 0 ? mis : 0u;
    *hi = v == ngran - 1 ? mis + rb - 16u * static_cast<uint32_t>(v) : 16u;
}
// Zero the elements of a granule outside [lo, hi).
template <class T, int VEC>
__device__ __forceinline__ void mask_granule(Frag<T, VEC> &f, uint32_t lo, uint32_t hi) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const uint32_t b = static_cast<uint32_t>(i * T::kBytes);
        if (b < lo || b >= hi) f.clear(i);
    }
}
// Store the elements of granule f that lie in [lo, hi) at the 16-byte-aligned
// address p: one vector store for a whole granule, else element by element.
template <class T, int VEC>
__device__ __forceinline__ void st_granule(char *p, const Frag<T, VEC> &f, uint32_t lo,
                                           uint32_t hi) {
    if (lo == 0u && hi == 16u) {
        st_global(p, f);
        return;
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const uint32_t b = static_cast<uint32_t>(i * T::kBytes);
        if (b >= lo && b < hi) f.st_elem(p + b, i);
    }
}

// Named barrier `id` over `count` threads (a multiple of 32).
__device__ __forceinline__ void group_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the OR of `flag` over the participants.
__device__ __forceinline__ int group_sync_or(int id, int count, int flag) {
    int any;
    asm volatile("{\n\t.reg .pred q, p;\n\t"
                 "setp.ne.s32 q, %1, 0;\n\t"
                 "bar.red.or.pred p, %2, %3, q;\n\t"
                 "selp.s32 %0, 1, 0, p;\n\t}"
                 : "=r"(any) : "r"(flag), "r"(id), "r"(count) : "memory");
    return any;
}

// Four sums reduced together (the one-exchange sandwich): butterflies over
// the warp (all lanes get the same bits), then one slot per warp.
struct Sums4 {
    float v[4];
};
__device__ __forceinline__ Sums4 warp_allsum4(Sums4 s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) s.v[i] += __shfl_xor_sync(0xFFFFFFFFu, s.v[i], o);
    return s;
}
// The same over one warp group (named barrier `id`), ORing a failure flag
// across the group in the same barrier.
__device__ __forceinline__ Sums4 wg_allsum4(Sums4 v, float4 *slots, int id, int count, int gtid,
                                            int flag, int *any) {
    v = warp_allsum4(v);
    const int lane = gtid & 31;
    const int warp = gtid >> 5;
    if (lane == 0) slots[warp] = make_float4(v.v[0], v.v[1], v.v[2], v.v[3]);
    *any = group_sync_or(id, count, flag);
    Sums4 t = {{0.0f, 0.0f, 0.0f, 0.0f}};
    if (lane < (count >> 5)) {
        const float4 w = slots[lane];
        t = Sums4{{w.x, w.y, w.z, w.w}};
    }
    return warp_allsum4(t);
}

// Sum of v over the `count` threads of one warp group (named barrier `id`),
// optionally ORing a failure flag across the group in the same barrier.
template <bool VOTE>
__device__ __forceinline__ float wg_allsum(float v, ReduceSlots &s, int id, int count,
                                              int gtid, int flag, int *any) {
    v = warp_allsum(v);
    const int lane = gtid & 31;
    const int warp = gtid >> 5;
    if (lane == 0) s.warp[warp] = v;
    if (VOTE) {
        *any = group_sync_or(id, count, flag);
    } else {
        group_sync(id, count);
    }
    return warp_allsum(lane < (count >> 5) ? s.warp[lane] : 0.0f);
}

// G warp groups share the stage ring and the gammas; group g handles the
// CTA's rows it = g, g+G, ...  so that G rows are reduced and written at the
// same time while the other stages are being filled.  Each group reduces
// over its own named barrier (ids 1..G).  `stages` must be a multiple of G:
// stage s then only ever holds rows of group s % G, so every wait on a stage
// barrier comes after the previous use of that stage has completed (a parity
// wait cannot tell a phase from the one two steps earlier), and every refill
// follows the consumption of the row it replaces.  If any wait runs out, the group
// that sees it raises `abort`; every group stops at its next vote, all meet
// at a CTA barrier, and thread 0 drains (bounded) every stage copy still in
// flight before the CTA exits.
//
// EDGE: rows that are not 16-byte aligned (a row pitch n * s that is not a
// multiple of 16, or operands offset from a 16-byte boundary), for the plain,
// then-add, then-add-scale and sandwich operations.  Every row operand and
// output must sit at the same offset `mis` from a 16-byte boundary in a row,
// and the host makes the persistent grid a multiple of 8 CTAs, so that all the
// rows of one CTA share that offset (a CTA's rows are gridDim.x rows apart,
// and 8 rows advance the offset by a multiple of 16 bytes for any n).  Each
// row is staged as the granules that cover it (granule_bounds); the gammas are
// copied element by element into shared memory at offset `mis` of zeroed
// slots, so that granule v of a staged row and of a gamma slot hold the same
// elements; edge granules are masked and stored element by element.  Stage
// slots are a.stage_bytes apart (at least the row's bytes rounded up to 16,
// plus 16).
template <int OP, class T, int K, int G, bool EDGE>
__global__ void __launch_bounds__(tma_max_threads(K, G), 1)
mrn_tma_kernel(const KernelArgs a, const int stages) {
    constexpr int VEC = 16 / T::kBytes;
    using Fr = Frag<T, VEC>;
    constexpr int NS = op_row_inputs(OP);   // row operands staged per row
    constexpr int NG = op_staged_gammas(OP);   // gammas kept in shared memory
    static_assert(!EDGE || op_has_edge_staging(OP), "edge staging: plain, then-add(-scale), sandwich");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ ReduceSlots slots1[G];
    __shared__ ReduceSlots slots2[G];
    // The f32 sandwich after a group's first row (gammas in shared memory): its
    // stream's sum of squares from three first-pass sums, one reduction per row
    // (as in the register kernel; the stored stream reduced again where those
    // sums cancel).  Slot sets alternate by row as for single-reduction operations.
    constexpr bool kOneExchange = OP == kSandwich && T::kBytes == 4;
    __shared__ __align__(16) float4 slots4[kOneExchange ? 2 : 1][G][32];
    __shared__ __align__(8) uint64_t bars[kTmaMaxStages + 1];   // [stages] = the gammas
    __shared__ int issued[kTmaMaxStages];
    __shared__ int consumed[kTmaMaxStages];
    __shared__ volatile int abort_flag;

    const uint32_t rb = static_cast<uint32_t>(a.n * T::kBytes);
    const uint32_t sb = EDGE ? a.stage_bytes : rb;        // bytes between shared-memory slots
    unsigned char *const gsm = smem;
    unsigned char *const stage0 = smem + NG * sb;
    const int tid = threadIdx.x;
    const int gsize = blockDim.x / G;
    const int grp = tid / gsize;
    const int gtid = tid - grp * gsize;
    const int bar_id = 1 + grp;
    const int64_t first = a.row0 + blockIdx.x;
    const int64_t step = gridDim.x;
    const int64_t my_rows = first < a.rows_end ? (a.rows_end - first + step - 1) / step : 0;
    const int64_t row_bytes = a.n * T::kBytes;
    const char *const xg = static_cast<const char *>(a.x);
    const char *const rg = static_cast<const char *>(a.res);
    if (stages < G || stages > kTmaMaxStages || stages % G != 0) {
        // The host never launches this; refuse rather than start any copy.
        if (tid == 0) atomicAdd(&g_wait_timeouts, 1u);
        return;
    }
    // This CTA's rows: `mis` bytes past a 16-byte boundary, `span` bytes of
    // granules per operand, `ngran` granules (EDGE); else whole 16-byte loads.
    uint32_t mis = 0;
    if (EDGE && my_rows > 0)
        mis = static_cast<uint32_t>((reinterpret_cast<uintptr_t>(xg) + first * row_bytes) & 15u);
    const uint32_t span = EDGE ? ((mis + rb + 15u) & ~15u) : rb;
    const int64_t ngran = EDGE ? static_cast<int64_t>(span >> 4) : a.nvec;
    if (EDGE && my_rows > 0) {
        // Refuse what the host never launches: a span beyond a slot, rows of
        // this CTA at different offsets, an operand at another offset (its
        // bulk copy or vector stores would be misaligned).
        const uintptr_t off = static_cast<uintptr_t>(first * row_bytes);
        bool ok = span <= sb &&
                  (my_rows == 1 || ((step * row_bytes) & 15) == 0) &&
                  ((reinterpret_cast<uintptr_t>(a.y) + off) & 15u) == mis;
        if (NS == 2) ok = ok && ((reinterpret_cast<uintptr_t>(rg) + off) & 15u) == mis;
        if (OP == kSandwich) ok = ok && ((reinterpret_cast<uintptr_t>(a.y2) + off) & 15u) == mis;
        if (!ok) {
            if (tid == 0) atomicAdd(&g_wait_timeouts, 1u);
            return;
        }
    }

    // EDGE: every thread places part of the gammas and arrives on the gamma
    // barrier once, so the gammas complete that barrier as a bulk copy does and
    // are awaited at the same point.  f32: each element by a 4-byte cp.async,
    // the thread's arrival made when its copies have landed (the threads go on
    // to their first rows at once); bf16: loaded and stored by the threads.
    const bool gamma_by_threads = EDGE && NG > 0;
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
        mbar_init(&bars[stages], gamma_by_threads ? blockDim.x : 1u);
        for (int s = 0; s < kTmaMaxStages; ++s) issued[s] = consumed[s] = 0;
        abort_flag = 0;
        fence_mbar_init();
    }
    if (gamma_by_threads && my_rows > 0) {
        // the bytes of each gamma slot's first and last granule outside gamma
        // must read as zero (the masked edge elements multiply them)
        const uint32_t last = span - 16u;
        for (uint32_t i = tid; i < NG * 8u; i += blockDim.x) {
            const uint32_t q = i >> 3, w = i & 7u;
            reinterpret_cast<uint32_t *>(gsm + q * sb + (w < 4u ? 0u : last))[w & 3u] = 0u;
        }
    }
    __syncthreads();
    pdl_enter();   // (the shared-memory set-up above overlapped the previous grid)
    if (tid == 0 && my_rows > 0) {
        // The first rows' copies go out before the gammas', and the gammas are
        // awaited only after a group's first reduction: their arrival overlaps
        // that row's load and reduction instead of preceding it (measured on
        // GB300: 4096 x 6656 sandwich 70.8 -> 70.2 us per call).
        for (int s = 0; s < stages && s < my_rows; ++s) {
            stage_row<NS>(stage0 + s * NS * sb, xg, rg, (first + s * step) * row_bytes - mis,
                          span, sb, &bars[s]);
            issued[s] = 1;
        }
        if (!gamma_by_threads) {
            // (NG == 0: completes at once; stall_bytes is a test hook, 0 in use)
            mbar_arrive_expect_tx(&bars[stages], NG * rb + a.stall_bytes);
            if (NG >= 1) bulk_to_shared(gsm, a.g1, rb, &bars[stages]);
            if (NG == 2) bulk_to_shared(gsm + rb, a.g2, rb, &bars[stages]);
        }
    }
    if (T::kBytes == 4 && gamma_by_threads && my_rows > 0) {
        // gamma element j to byte mis + 4 j of its slot
        if (tid == 0) mbar_expect_tx(&bars[stages], a.stall_bytes);   // (test hook: 0 in use)
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const char *src = static_cast<const char *>(q == 0 ? a.g1 : a.g2);
            unsigned char *dst = gsm + q * sb + mis;
            for (int64_t j = tid; j < a.n; j += blockDim.x) cp_async_4(dst + 4 * j, src + 4 * j);
        }
        cp_async_arrive(&bars[stages]);
    } else if (gamma_by_threads && my_rows > 0) {
        // gamma element j to byte mis + j * s of its slot, while the
        // first rows' copies are in flight: each thread reads whole 16-byte
        // granules of gamma (the same over-read as for the rows), all its
        // loads first, and places the elements that belong to gamma
        constexpr int GL = 4;   // granule loads per gamma and thread in flight
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const uintptr_t g0 = reinterpret_cast<uintptr_t>(q == 0 ? a.g1 : a.g2);
            const uint32_t gm = static_cast<uint32_t>(g0 & 15u);
            const char *gbase = reinterpret_cast<const char *>(g0 - gm);
            const int64_t gspan = (gm + rb + 15u) >> 4;
            unsigned char *dst = gsm + q * sb + mis;   // gamma's byte b - gm goes to dst + b - gm
            for (int64_t v0 = tid; v0 < gspan; v0 += GL * blockDim.x) {
                Fr w[GL];
#pragma unroll
                for (int u = 0; u < GL; ++u) {
                    const int64_t v = v0 + u * static_cast<int64_t>(blockDim.x);
                    if (v < gspan) ld_ro(w[u], gbase + v * 16);
                }
#pragma unroll
                for (int u = 0; u < GL; ++u) {
                    const int64_t v = v0 + u * static_cast<int64_t>(blockDim.x);
                    if (v >= gspan) continue;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        const int64_t b = v * 16 + i * T::kBytes;   // byte within gamma's granules
                        if (b < gm || b >= gm + rb) continue;
                        if (T::kBytes == 4) {
                            *reinterpret_cast<uint32_t *>(dst + (b - gm)) = w[u].w[i & 3];
                        } else {
                            *reinterpret_cast<unsigned short *>(dst + (b - gm)) =
                                static_cast<unsigned short>((i & 1) ? (w[u].w[i >> 1] >> 16)
                                                                    : (w[u].w[i >> 1] & 0xFFFFu));
                        }
                    }
                }
            }
        }
        if (tid == 0) {
            mbar_arrive_expect_tx(&bars[stages], a.stall_bytes);   // (test hook: 0 in use)
        } else {
            mbar_arrive(&bars[stages]);
        }
    }
    int failed = 0;
    bool gammas_in = my_rows == 0;   // the gamma copy awaited (by this thread)
    if (OP == kAddRmsnorm && my_rows > 0) {
        // (its sums are stored before the first reduction: wait up front, so a
        // timed-out copy still means nothing is written)
        failed = mbar_wait_bounded(&bars[stages], 0) ? 0 : 1;
        gammas_in = true;
    }
    const float sc = load_out_scale<OP, T>(a.scale);

    // EDGE: the register slots of this thread that hold a partial granule (at
    // most the row's first and last); the same for every row of the CTA.
    uint32_t edge_slots = 0;
    if (EDGE) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
            uint32_t lo, hi;
            granule_bounds(v, ngran, mis, rb, &lo, &hi);
            if (v < ngran && (lo != 0u || hi != 16u)) edge_slots |= 1u << k;
        }
    }
    // Store slot k (granule v) of an output row (out_base + row_byte0 is the
    // row's first granule): whole vectors, element-wise for a partial granule.
    auto store = [&](void *out_base, int64_t row_byte0, int64_t v, int k, const Fr &f) {
        char *p = static_cast<char *>(out_base) + row_byte0 + v * 16;
        if (EDGE && ((edge_slots >> k) & 1u)) {
            uint32_t lo, hi;
            granule_bounds(v, ngran, mis, rb, &lo, &hi);
            st_granule(p, f, lo, hi);
        } else {
            st_global(p, f);
        }
    };

    for (int64_t it = grp; it < my_rows; it += G) {
        const int s = static_cast<int>(it % stages);
        const uint32_t parity = static_cast<uint32_t>((it / stages) & 1);
        const int64_t row = first + it * step;
        if (!failed && !mbar_wait_bounded(&bars[s], parity)) failed = 1;

        Fr xv[K];
        Fr rv[K];
        const unsigned char *sp = stage0 + s * NS * sb;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
            if (v < ngran) {
                ld_shared(xv[k], sp + v * 16);
                if (NS == 2) ld_shared(rv[k], sp + sb + v * 16);
                if (EDGE && ((edge_slots >> k) & 1u)) {
                    uint32_t lo, hi;
                    granule_bounds(v, ngran, mis, rb, &lo, &hi);
                    mask_granule(xv[k], lo, hi);
                    if (NS == 2) mask_granule(rv[k], lo, hi);
                }
            } else {
                xv[k].zero();
                rv[k].zero();
            }
        }
        H16<VEC> hg[K];   // the seam's 16-bit gamma, through L1, in flight over the reduction
        if (op_seam_weighted(OP)) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v < a.nvec) ld_h16(hg[k], static_cast<const char *>(a.g1) + v * VEC * 2);
            }
        }
        const int64_t row_elem = row * a.n;
        const int64_t row_byte0 = row * row_bytes - mis;   // the row's first granule
        float ss = 0.0f;
        const bool fused = kOneExchange && gammas_in;       // (uniform over the group)
        Sums4 part = {{0.0f, 0.0f, 0.0f, 0.0f}};            // sum b^2, (b g1)^2, (b g1) r, r^2
        if (kOneExchange && fused) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v >= ngran) continue;
                Fr g;
                ld_shared(g, gsm + v * 16);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const float bx = xv[k].get(i), r = rv[k].get(i);
                    const float q = bx * g.get(i);
                    part.v[0] = fmaf(bx, bx, part.v[0]);
                    part.v[1] = fmaf(q, q, part.v[1]);
                    part.v[2] = fmaf(q, r, part.v[2]);
                    part.v[3] = fmaf(r, r, part.v[3]);
                }
            }
        } else if (OP == kAddRmsnorm) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v >= a.nvec || failed) continue;
                rv[k] = add_frags(xv[k], rv[k]);
                st_global(elem_ptr<T>(a.y, row_elem + v * VEC), rv[k]);
                ss += frag_sum_sq(rv[k]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k) ss += frag_sum_sq(xv[k]);
        }
        // One barrier per reduction: a warp may start the next row's reduction
        // while another still reads this one's warp sums.  Single-reduction
        // operations therefore alternate the two slot sets by row (a set is
        // rewritten only after the next row's barrier, which every reader
        // passes after its read); the sandwich's second reduction separates
        // the uses of each set.
        ReduceSlots &rs1 = (OP != kSandwich && ((it / G) & 1)) ? slots2[grp] : slots1[grp];
        int any_failed;
        Sums4 tot4 = {{0.0f, 0.0f, 0.0f, 0.0f}};
        float tot;
        if (kOneExchange && fused) {
            tot4 = wg_allsum4(part, slots4[kOneExchange ? ((it / G) & 1) : 0][grp], bar_id, gsize,
                              gtid, failed | abort_flag, &any_failed);
            tot = tot4.v[0];
        } else {
            tot = wg_allsum<true>(ss, rs1, bar_id, gsize, gtid, failed | abort_flag, &any_failed);
        }
        if (any_failed) {
            if (gtid == 0) abort_flag = 1;
            break;
        }
        // Every thread of the group holds its part of the stage now: refill it.
        if (gtid == 0) {
            consumed[s] += 1;
            if (it + stages < my_rows) {
                fence_proxy_async_smem();
                stage_row<NS>(stage0 + s * NS * sb, xg, rg,
                              (first + (it + stages) * step) * row_bytes - mis, span, sb,
                              &bars[s]);
                issued[s] += 1;
            }
        }
        if (!gammas_in) {
            // First row of this group: the gammas must have landed before any
            // output; the group agrees on a timed-out wait in one vote and stops
            // before writing anything.
            gammas_in = true;
            const int late = (!failed && !mbar_wait_bounded(&bars[stages], 0)) ? 1 : failed;
            if (group_sync_or(bar_id, gsize, late)) {
                if (gtid == 0) abort_flag = 1;
                break;
            }
        }
        const float inv1 = inv_rms(tot, a.n, a.eps1);

        if (OP == kAddRmsnorm) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v >= a.nvec) continue;
                Fr g;
                ld_shared(g, gsm + v * 16);
                st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(rv[k], inv1, g));
            }
            continue;
        }
        if (op_is_seam(OP)) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v < a.nvec) seam_output<OP, T, VEC>(xv[k], inv1, hg[k], a.y, row_elem + v * VEC);
            }
            continue;
        }
        if (OP == kRmsnormQ8) {
            char *blocks = q8_row_blocks(a, row);
#pragma unroll
            for (int k = 0; k < K; ++k) {   // no early exit: every lane shuffles
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                Fr g;
                if (v < a.nvec) {
                    ld_shared(g, gsm + v * 16);
                } else {
                    g.zero();
                }
                q8_1_output(xv[k], g, inv1, v < a.nvec, blocks, v);
            }
            continue;
        }
        if (OP != kSandwich) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
                if (v >= ngran) continue;
                Fr g;
                ld_shared(g, gsm + v * 16);
                store(a.y, row_byte0, v, k, single_norm_output<OP>(xv[k], inv1, g, rv[k], sc));
            }
            continue;
        }
        // (one exchange: sum s^2 = inv1^2 A + 2 inv1 B + C where those terms do not
        // cancel -- their magnitudes sum to at most twice the result)
        bool direct = true;
        float est = 0.0f;
        if (kOneExchange && fused) {
            const float i2 = inv1 * inv1;
            est = fmaf(i2, tot4.v[1], fmaf(2.0f * inv1, tot4.v[2], tot4.v[3]));
            const float mag = fmaf(i2, tot4.v[1], fmaf(2.0f * inv1, fabsf(tot4.v[2]), tot4.v[3]));
            direct = !(est >= 0.5f * mag);
        }
        float ss2 = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
            if (v >= ngran) continue;
            Fr g;
            ld_shared(g, gsm + v * 16);
            rv[k] = apply_norm_add(xv[k], inv1, g, rv[k]);
            store(a.y, row_byte0, v, k, rv[k]);
            if (direct) ss2 += frag_sum_sq(rv[k]);
        }
        const float inv2 = inv_rms(direct ? wg_allsum<false>(ss2, slots2[grp], bar_id, gsize, gtid,
                                                              0, nullptr)
                                          : est,
                                   a.n, a.eps2);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = gtid + static_cast<int64_t>(k) * gsize;
            if (v >= ngran) continue;
            Fr g;
            ld_shared(g, gsm + sb + v * 16);
            store(a.y2, row_byte0, v, k, apply_norm(rv[k], inv2, g));
        }
    }

    // Exit: with no failure every issued copy was consumed.  After a failure,
    // wait (bounded) for the copies still in flight so that none lands after
    // the CTA has left its shared memory (each thread its own cp.async first).
    if (EDGE && T::kBytes == 4) cp_async_wait_all();
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

// ---------------------------------------------------------------------------
// Staged kernel for rows too wide for one CTA's registers: a thread-block
// cluster of C CTAs handles one row at a time, CTA `crank` owning slice
// [crank * S, (crank + 1) * S) of it (S = n / C elements, a multiple of 16
// bytes).  Persistent: cluster c takes rows c, c + (number of clusters), ...
// Each CTA bulk-copies its slice of a future row (and of the residual) into
// a shared-memory stage, `stages` rows ahead, and its slice of the gammas
// once.  A row's sum is the CTA sums exchanged as messages: each CTA sends
// {partial, stop vote} to every peer with st.async, which lands in the
// peer's mailbox [row parity][sender rank] and completes the peer's
// mailbox mbarrier for that parity (armed by the peer for (C - 1) * 8
// bytes); a CTA waits (bounded) on its own mbarrier, then every CTA adds the
// C partials in rank order, its own from registers (all CTAs get the same
// bits).  No cluster-wide barrier per row, so no row waits for the previous
// row's output stores to drain.  Mailboxes alternate with the row's parity:
// a CTA sends row j + 2's message only after it has received every peer's
// row j + 1 message, and a peer sends that only after it has read its row j
// mailbox, so a mailbox is never overwritten while it may still be read and
// no message lands in a later phase of the mbarrier than the one awaited.
// All CTAs of a cluster walk the same rows; a failed (bounded) stage wait is
// the stop vote, so the whole cluster stops at one row, then each CTA
// drains its own copies.  A cluster barrier at start (after the mbarriers
// are initialised) and one at exit (no CTA leaves while a message may still
// be addressed to it) are the only cluster-wide barriers.  Operations:
// plain, then-add, then-add-scale and the sandwich.
// ---------------------------------------------------------------------------
struct ClusterMail {
    float warp[32];
    uint2 box[2][kMaxCluster];   // [row parity][sender rank] = {partial bits, stop vote}
    uint64_t bar[2];             // [row parity]: every peer's message for that row landed
};

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}
// Bounded like mbar_wait_bounded, for mbarriers completed by peers' messages.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 28); ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}
// Store {x, y} into `box` of CTA `rank` of this cluster, completing 8 bytes
// of the transaction count of that CTA's `bar`.
__device__ __forceinline__ void send_pair(uint2 *box, uint64_t *bar, unsigned rank, uint32_t x,
                                          uint32_t y) {
    uint32_t rbox, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbox) : "r"(smem_addr(box)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
                 :: "r"(rbox), "r"(x), "r"(y), "r"(rbar) : "memory");
}

// Sum of v over the cluster for row `it` of this CTA (every thread of every
// CTA calls it).  *stop is set (uniformly over the CTA) when any CTA voted
// `flag` or a message did not arrive in time; *timed_out when the latter
// happened to this thread.  `first` completes the cluster arrive issued at
// start, after which every peer's mailboxes are initialised.
__device__ __forceinline__ float cluster_row_sum(float v, ClusterMail &m, unsigned cl,
                                                 unsigned crank, int64_t it, int flag, int *stop,
                                                 int *timed_out, bool first) {
    v = warp_allsum(v);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (lane == 0) m.warp[warp] = v;
    __syncthreads();
    const float t = warp_allsum(lane < nwarps ? m.warp[lane] : 0.0f);
    const int f = __syncthreads_or(flag);   // (also: every thread has read m.warp)
    const int p = static_cast<int>(it & 1);
    if (first) cluster_wait_acquire();
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&m.bar[p], (cl - 1) * 8u);
    if (threadIdx.x < cl && threadIdx.x != crank)
        send_pair(&m.box[p][crank], &m.bar[p], threadIdx.x, __float_as_uint(t),
                  static_cast<uint32_t>(f));
    const bool ok = mbar_wait_bounded_cluster(&m.bar[p], static_cast<uint32_t>((it >> 1) & 1));
    if (!ok) *timed_out = 1;
    const bool mine = lane < static_cast<int>(cl);
    uint2 got = make_uint2(0u, 0u);
    if (mine) got = lane == static_cast<int>(crank)
                        ? make_uint2(__float_as_uint(t), static_cast<uint32_t>(f))
                        : m.box[p][lane];
    *stop = __syncthreads_or(!ok || (mine && got.y != 0u));
    return warp_allsum(mine ? __uint_as_float(got.x) : 0.0f);
}

// ---------------------------------------------------------------------------
// Register kernel: one row per CTA, or per cluster of cl CTAs (launched with
// a cluster dimension); CTA `rank` covers loads [rank*threads*K,
// (rank+1)*threads*K).  In a cluster each reduction is one exchange of
// messages: every CTA sends its partial to every peer with st.async into the
// peer's mailbox for that reduction, completing the peer's mailbox mbarrier
// (armed for (cl - 1) * 4 bytes), and adds the cl partials in rank order, its
// own from registers (all CTAs get the same bits).  A cluster barrier at
// start, after the mailboxes are initialised, is the only cluster-wide
// barrier: nothing ties a reduction to the stores before it (the sandwich's
// second reduction does not wait for the stream's stores), and every message
// a CTA receives is one it waits for before it leaves.
// ---------------------------------------------------------------------------
struct RowMail {
    float warp[32];
    float box[kMaxCluster];   // [sender rank]
    uint64_t bar;             // every peer's partial landed
};

// Store v into `box` of CTA `rank` of this cluster, completing 4 bytes of the
// transaction count of that CTA's `bar`.
__device__ __forceinline__ void send_f32(float *box, uint64_t *bar, unsigned rank, float v) {
    uint32_t rbox, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbox) : "r"(smem_addr(box)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(rbox), "r"(__float_as_uint(v)), "r"(rbar) : "memory");
}

// Sum of v over the CTA and its cluster (cl > 1); every thread of every CTA
// calls it once per mailbox.  `first` completes the cluster arrive issued at
// start.  A message wait that runs out (bounded, about one second) sets
// *timed_out: the row's outputs are then unspecified and the kernel counts it.
__device__ __forceinline__ float cluster_mail_sum(float v, RowMail &m, unsigned cl,
                                                  unsigned crank, bool first, uint32_t stall,
                                                  int *timed_out) {
    v = warp_allsum(v);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (lane == 0) m.warp[warp] = v;
    __syncthreads();
    const float t = warp_allsum(lane < nwarps ? m.warp[lane] : 0.0f);
    if (first) cluster_wait_acquire();
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&m.bar, (cl - 1) * 4u + stall);   // (test hook: 0)
    if (threadIdx.x < cl && threadIdx.x != crank) send_f32(&m.box[crank], &m.bar, threadIdx.x, t);
    if (!mbar_wait_bounded_cluster(&m.bar, 0)) *timed_out = 1;
    const bool mine = lane < static_cast<int>(cl);
    return warp_allsum(mine ? (lane == static_cast<int>(crank) ? t : m.box[lane]) : 0.0f);
}

// ---------------------------------------------------------------------------
// Looped kernel for rows wider than the register-resident and staged
// geometries hold: one row per CTA, or per thread-block cluster of cl CTAs
// (launched with a cluster dimension), CTA `crank` looping over its slice
// [vlo, vhi) of the row's loads (a multiple of 32 loads, so a Q8_1 block
// never straddles two CTAs).  The slice is read once for the sum and once more
// for the output; the sandwich reads the stream it stored once more for the
// second norm.  The second read comes from L2 while the rows in flight fit in
// it: over a cluster of 16, a row's slices are 1/16 of it and only one row per
// resident cluster is in flight (256 rows of 1 MB: tens of MB), where one row
// per CTA put every row in flight at once and read DRAM twice.  A reduction
// over the cluster is one exchange of st.async messages (cluster_mail_sum),
// as in the register kernel.  Each iteration handles kStreamUnroll loads per
// operand so that several are in flight.
// ---------------------------------------------------------------------------
template <int OP, class T, int VEC>
__global__ void __launch_bounds__(kStreamMaxThreads)
mrn_stream_kernel(const KernelArgs a) {
    using Fr = Frag<T, VEC>;
    constexpr int U = kStreamUnroll;
    __shared__ ReduceSlots slots1;
    __shared__ ReduceSlots slots2;
    __shared__ __align__(8) RowMail mail1;
    __shared__ __align__(8) RowMail mail2;
    const unsigned cl = cluster_nctarank();
    const unsigned crank = cluster_ctarank();
    if (cl > 1) {
        if (threadIdx.x == 0) {
            mbar_init(&mail1.bar, 1);
            mbar_init(&mail2.bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        cluster_arrive_relaxed();   // (thread 0: after its initialisation and fence)
    }
    pdl_enter();
    const int64_t row = a.row0 + cluster_index_x();
    const int64_t row_elem = row * a.n;
    const int64_t nt = blockDim.x;
    const int64_t per = ((a.nvec + cl - 1) / cl + 31) / 32 * 32;
    const int64_t vlo = min(a.nvec, static_cast<int64_t>(crank) * per);
    const int64_t vhi = min(a.nvec, vlo + per);
    int timed_out = 0;
    auto reduce1 = [&](float v) {
        return cl > 1 ? cluster_mail_sum(v, mail1, cl, crank, true, a.stall_bytes, &timed_out)
                      : cta_allsum(v, slots1, 1, 0, false);
    };
    auto reduce2 = [&](float v) {
        return cl > 1 ? cluster_mail_sum(v, mail2, cl, crank, false, 0u, &timed_out)
                      : cta_allsum(v, slots2, 1, 0, false);
    };

    // A slice read twice stays in L2 between its reads: its first read marks
    // the lines evict-last, its last read evict-first (as does the re-read of
    // the sandwich's stream and of add + norm's sum, which are stored evict-last).
    const uint64_t keep = l2_policy_keep();
    const uint64_t drop = l2_policy_drop();
    const float sc = load_out_scale<OP, T>(a.scale);
    float ss = 0.0f;
    for (int64_t v0 = vlo + threadIdx.x; v0 < vhi; v0 += nt * U) {
        Fr x[U], r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * nt;
            if (v < vhi) {
                if (OP == kAddRmsnorm) {
                    ld_hint(x[u], elem_ptr<T>(a.x, row_elem + v * VEC), drop);
                    ld_stream(r[u], elem_ptr<T>(a.res, row_elem + v * VEC));
                } else {
                    ld_hint(x[u], elem_ptr<T>(a.x, row_elem + v * VEC), keep);
                }
            } else {
                x[u].zero();
                r[u].zero();
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (OP == kAddRmsnorm) {
                const int64_t v = v0 + u * nt;
                if (v >= vhi) continue;
                x[u] = add_frags(x[u], r[u]);       // residual_out, stored and normed below
                st_hint(elem_ptr<T>(a.y, row_elem + v * VEC), x[u], keep);
            }
            ss += frag_sum_sq(x[u]);
        }
    }
    const float inv1 = inv_rms(reduce1(ss), a.n, a.eps1);

    if (OP == kAddRmsnorm) {
        // re-read the sums this same thread stored
        for (int64_t v0 = vlo + threadIdx.x; v0 < vhi; v0 += nt * U) {
            Fr sm[U], g[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi) {
                    ld_hint(sm[u], elem_ptr<T>(a.y, row_elem + v * VEC), drop);
                    ld_ro(g[u], elem_ptr<T>(a.g1, v * VEC));
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi)
                    st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(sm[u], inv1, g[u]));
            }
        }
    } else if (OP == kRmsnormQ8) {
        // The trip count is uniform across each warp (the q8 output shuffles):
        // the slice starts at a multiple of 32 loads.
        char *blocks = q8_row_blocks(a, row);
        const int64_t lane = threadIdx.x & 31;
        for (int64_t v0 = vlo + threadIdx.x; v0 - lane < vhi; v0 += nt * U) {
            Fr x[U], g[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi) {
                    ld_hint(x[u], elem_ptr<T>(a.x, row_elem + v * VEC), drop);
                    ld_ro(g[u], elem_ptr<T>(a.g1, v * VEC));
                } else {
                    x[u].zero();
                    g[u].zero();
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                q8_1_output(x[u], g[u], inv1, v < vhi, blocks, v);
            }
        }
    } else if (op_is_seam(OP)) {
        for (int64_t v0 = vlo + threadIdx.x; v0 < vhi; v0 += nt * U) {
            Fr x[U];
            H16<VEC> g[U] = {};
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi) {
                    ld_hint(x[u], elem_ptr<T>(a.x, row_elem + v * VEC), drop);
                    if (op_seam_weighted(OP))
                        ld_h16(g[u], static_cast<const char *>(a.g1) + v * VEC * 2);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi) seam_output<OP, T, VEC>(x[u], inv1, g[u], a.y, row_elem + v * VEC);
            }
        }
    } else {
        float ss2 = 0.0f;
        for (int64_t v0 = vlo + threadIdx.x; v0 < vhi; v0 += nt * U) {
            Fr x[U], g[U], r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v < vhi) {
                    ld_hint(x[u], elem_ptr<T>(a.x, row_elem + v * VEC), drop);
                    ld_ro(g[u], elem_ptr<T>(a.g1, v * VEC));
                    if (OP != kRmsnorm) ld_stream(r[u], elem_ptr<T>(a.res, row_elem + v * VEC));
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * nt;
                if (v >= vhi) continue;
                const int64_t e = row_elem + v * VEC;
                if (OP == kSandwich) {
                    const Fr o = apply_norm_add(x[u], inv1, g[u], r[u]);
                    st_hint(elem_ptr<T>(a.y, e), o, keep);
                    ss2 += frag_sum_sq(o);
                } else {
                    st_global(elem_ptr<T>(a.y, e), single_norm_output<OP>(x[u], inv1, g[u], r[u], sc));
                }
            }
        }
        if (OP == kSandwich) {
            // the stream as stored, read back by the thread that stored it
            const float inv2 = inv_rms(reduce2(ss2), a.n, a.eps2);
            for (int64_t v0 = vlo + threadIdx.x; v0 < vhi; v0 += nt * U) {
                Fr sv[U], g[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + u * nt;
                    if (v < vhi) {
                        ld_hint(sv[u], elem_ptr<T>(a.y, row_elem + v * VEC), drop);
                        ld_ro(g[u], elem_ptr<T>(a.g2, v * VEC));
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + u * nt;
                    if (v < vhi)
                        st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(sv[u], inv2, g[u]));
                }
            }
        }
    }
    if (timed_out) {
        // A late message may still be landing in this CTA: wait once more
        // (bounded) before leaving; count the timeout once per warp.
        (void)mbar_wait_bounded_cluster(&mail1.bar, 0);
        if (OP == kSandwich) (void)mbar_wait_bounded_cluster(&mail2.bar, 0);
        const unsigned lanes = __activemask();
        if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(lanes) - 1))
            atomicAdd(&g_wait_timeouts, 1u);
    }
}

// Four sums at once (the one-exchange sandwich below): each CTA's four
// partials travel as one 16-byte st.async message per peer.
struct RowMail4 {
    float4 warp[32];
    float4 box[kMaxCluster];   // [sender rank]
    uint64_t bar;              // every peer's partials landed
};
template <bool USED> struct RowMail4Slot {   // present only where the kernel uses it
    RowMail4 m;
};
template <> struct RowMail4Slot<false> {};
__device__ __forceinline__ void send_f32x4(float4 *box, uint64_t *bar, unsigned rank,
                                           const Sums4 &t) {
    uint32_t rbox, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbox) : "r"(smem_addr(box)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(rbox), "r"(__float_as_uint(t.v[0])), "r"(__float_as_uint(t.v[1])),
                    "r"(__float_as_uint(t.v[2])), "r"(__float_as_uint(t.v[3])), "r"(rbar)
                 : "memory");
}
// Sums of four values over the CTA and, when cl > 1, over the cluster (every
// thread of every CTA calls it, as the kernel's first cluster operation: it
// completes the arrive issued at start).  Every CTA adds the cl partials in
// rank order, so all get the same bits.  A timed-out message wait sets
// *timed_out (the row's outputs are then unspecified).
__device__ __forceinline__ Sums4 cluster_mail_sum4(Sums4 v, RowMail4 &m, unsigned cl,
                                                   unsigned crank, uint32_t stall,
                                                   int *timed_out) {
    v = warp_allsum4(v);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (lane == 0) m.warp[warp] = make_float4(v.v[0], v.v[1], v.v[2], v.v[3]);
    __syncthreads();
    Sums4 t = {{0.0f, 0.0f, 0.0f, 0.0f}};
    if (lane < nwarps) {
        const float4 w = m.warp[lane];
        t = Sums4{{w.x, w.y, w.z, w.w}};
    }
    t = warp_allsum4(t);
    if (cl == 1) return t;
    cluster_wait_acquire();
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&m.bar, (cl - 1) * 16u + stall);   // (test hook: 0)
    if (threadIdx.x < cl && threadIdx.x != crank) send_f32x4(&m.box[crank], &m.bar, threadIdx.x, t);
    if (!mbar_wait_bounded_cluster(&m.bar, 0)) *timed_out = 1;
    Sums4 got = {{0.0f, 0.0f, 0.0f, 0.0f}};
    if (lane < static_cast<int>(cl)) {
        if (lane == static_cast<int>(crank)) {
            got = t;
        } else {
            const float4 w = m.box[lane];
            got = Sums4{{w.x, w.y, w.z, w.w}};
        }
    }
    return warp_allsum4(got);
}

// The f32 sandwich with one reduction on the critical path (the register
// kernel, for decode).  The stream s = (b * inv1) * g1 + r of the fused tail
// ("Chapter 12", section 12.4.3) has, in exact arithmetic,
//   sum s^2 = inv1^2 * sum (b g1)^2 + 2 inv1 * sum (b g1) r + sum r^2,
// and the three sums on the right need no inv1: they are taken in the first
// pass, beside sum b^2, and reduced together in one exchange.  Where the
// terms do not cancel (their magnitudes sum to at most twice the result) the
// f32 error of the result stays within a few units of 2^-24 per reduction
// level, as for the direct sum of the stored stream; where they do, the row
// takes the second reduction of the stored stream, as the general path does.
// The decision depends only on the reduced sums, so every CTA of the cluster
// takes the same one.
template <class T, int VEC, int K, class Reduce4, class Reduce2>
__device__ __forceinline__ void sandwich_one_exchange(const KernelArgs &a, int64_t row,
                                                      int64_t first, int64_t stride,
                                                      Reduce4 reduce4, Reduce2 reduce2,
                                                      bool *second) {
    using Fr = Frag<T, VEC>;
    // With few slots per thread (decode) gamma_pre is loaded with everything
    // else, so that no load waits behind the exchange; with many (batches)
    // it reuses gamma_post's registers after the stream is formed.
    constexpr bool kEarlyG2 = K <= 2;
    const int64_t row_elem = row * a.n;
    Fr xv[K];
    Fr rv[K];
    Fr gv[K];
    Fr g2v[kEarlyG2 ? K : 1];
    bool ok[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t v = first + k * stride;
        ok[k] = v < a.nvec;
        const int64_t e = row_elem + v * VEC;
        if (ok[k]) {
            ld_stream(xv[k], elem_ptr<T>(a.x, e));
            ld_stream(rv[k], elem_ptr<T>(a.res, e));
        } else {
            xv[k].zero();
            rv[k].zero();
        }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (ok[k]) {
            ld_ro(gv[k], elem_ptr<T>(a.g1, (first + k * stride) * VEC));
            if constexpr (kEarlyG2) ld_ro(g2v[k], elem_ptr<T>(a.g2, (first + k * stride) * VEC));
        } else {
            gv[k].zero();
        }
    }
    Sums4 part = {{0.0f, 0.0f, 0.0f, 0.0f}};   // sum b^2, sum (b g1)^2, sum (b g1) r, sum r^2
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float b = xv[k].get(i), r = rv[k].get(i);
            const float q = b * gv[k].get(i);
            part.v[0] = fmaf(b, b, part.v[0]);
            part.v[1] = fmaf(q, q, part.v[1]);
            part.v[2] = fmaf(q, r, part.v[2]);
            part.v[3] = fmaf(r, r, part.v[3]);
        }
    const Sums4 tot = reduce4(part);
    const float inv1 = inv_rms(tot.v[0], a.n, a.eps1);
    const float i2 = inv1 * inv1;
    const float est = fmaf(i2, tot.v[1], fmaf(2.0f * inv1, tot.v[2], tot.v[3]));
    const float mag = fmaf(i2, tot.v[1], fmaf(2.0f * inv1, fabsf(tot.v[2]), tot.v[3]));
    const bool direct = !(est >= 0.5f * mag);   // (a NaN takes the direct sum too)
    float ss2 = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!ok[k]) continue;
        const int64_t v = first + k * stride;
        rv[k] = apply_norm_add(xv[k], inv1, gv[k], rv[k]);
        st_global(elem_ptr<T>(a.y, row_elem + v * VEC), rv[k]);
        if (direct) ss2 += frag_sum_sq(rv[k]);
    }
    if constexpr (!kEarlyG2) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (ok[k]) ld_ro(gv[k], elem_ptr<T>(a.g2, (first + k * stride) * VEC));
        }
    }
    *second = direct;
    const float inv2 = inv_rms(direct ? reduce2(ss2) : est, a.n, a.eps2);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!ok[k]) continue;
        const int64_t v = first + k * stride;
        st_global(elem_ptr<T>(a.y2, row_elem + v * VEC),
                  apply_norm(rv[k], inv2, kEarlyG2 ? g2v[kEarlyG2 ? k : 0] : gv[k]));
    }
}

template <int OP, class T, int VEC, int K>
__device__ __forceinline__ void cta_kernel_body(const KernelArgs &a) {
    __shared__ ReduceSlots slots1;
    __shared__ ReduceSlots slots2;
    __shared__ __align__(8) RowMail mail1;
    __shared__ __align__(8) RowMail mail2;
    constexpr bool kOneExchange = OP == kSandwich && T::kBytes == 4;   // f32 sandwich
    __shared__ __align__(16) RowMail4Slot<kOneExchange> mail4;
    const unsigned cl = cluster_nctarank();
    const unsigned crank = cluster_ctarank();
    if (cl > 1) {
        if (threadIdx.x == 0) {
            mbar_init(&mail1.bar, 1);
            mbar_init(&mail2.bar, 1);
            if constexpr (kOneExchange) mbar_init(&mail4.m.bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        cluster_arrive_relaxed();   // (thread 0: after its initialisation and fence)
    }
    pdl_enter();
    const int64_t row = a.row0 + cluster_index_x();
    const int64_t first = static_cast<int64_t>(crank) * blockDim.x * K + threadIdx.x;
    int timed_out = 0;
    if constexpr (kOneExchange) {
        auto reduce4 = [&](Sums4 v) {
            return cluster_mail_sum4(v, mail4.m, cl, crank, a.stall_bytes, &timed_out);
        };
        auto reduce2 = [&](float v) {
            return cl > 1 ? cluster_mail_sum(v, mail2, cl, crank, false, 0u, &timed_out)
                          : cta_allsum(v, slots2, 1, 0, false);
        };
        bool second = false;
        sandwich_one_exchange<T, VEC, K>(a, row, first, blockDim.x, reduce4, reduce2, &second);
        if (timed_out) {
            // A late message may still be landing in this CTA: wait once more
            // (bounded) before leaving; count the timeout once per warp.
            (void)mbar_wait_bounded_cluster(&mail4.m.bar, 0);
            if (second) (void)mbar_wait_bounded_cluster(&mail2.bar, 0);
            const unsigned lanes = __activemask();
            if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(lanes) - 1))
                atomicAdd(&g_wait_timeouts, 1u);
        }
        return;
    }
    auto reduce1 = [&](float v) {
        return cl > 1 ? cluster_mail_sum(v, mail1, cl, crank, true, a.stall_bytes, &timed_out)
                      : cta_allsum(v, slots1, 1, 0, false);
    };
    auto reduce2 = [&](float v) {
        return cl > 1 ? cluster_mail_sum(v, mail2, cl, crank, false, 0u, &timed_out)
                      : cta_allsum(v, slots2, 1, 0, false);
    };
    row_body<OP, T, VEC, K>(a, row, true, first, blockDim.x, reduce1, reduce2);
    if (timed_out) {
        // A late message may still be landing in this CTA: wait once more
        // (bounded) before leaving; count the timeout once per warp.
        (void)mbar_wait_bounded_cluster(&mail1.bar, 0);
        if (OP == kSandwich) (void)mbar_wait_bounded_cluster(&mail2.bar, 0);
        const unsigned lanes = __activemask();
        if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(lanes) - 1))
            atomicAdd(&g_wait_timeouts, 1u);
    }
}

template <int OP, class T, int VEC, int K>
__global__ void __launch_bounds__(cta_max_threads(K)) mrn_cta_kernel(const KernelArgs a) {
    cta_kernel_body<OP, T, VEC, K>(a);
}

// Plain f32 RMSNorm at 8 slots per thread, asking for three CTAs per SM (80
// registers): one row per CTA then keeps three rows' loads in flight per SM
// (measured on GB300: 4096 x 6656 in CTAs of 224 threads 34.0 us, against
// 37.4 us for the staged kernel; with the default register budget two CTAs
// fit).  A kernel of its own: a minimum-blocks bound on the shared template
// changes every other instantiation's register allocation too.
template <int OP, class T, int VEC>
__global__ void __launch_bounds__(cta_max_threads(8), 3) mrn_cta_kernel_k8x3(const KernelArgs a) {
    cta_kernel_body<OP, T, VEC, 8>(a);
}

template <int OP, class T, int K>
__global__ void __launch_bounds__(cta_max_threads(K), 1)
mrn_tma_cluster_kernel(const KernelArgs a, const int stages) {
    constexpr int VEC = 16 / T::kBytes;
    using Fr = Frag<T, VEC>;
    constexpr int NS = op_row_inputs(OP);   // row operands staged per row
    constexpr int NG = op_gammas(OP);       // gamma slices kept in shared memory
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) ClusterMail mail1;
    __shared__ __align__(8) ClusterMail mail2;
    __shared__ __align__(8) uint64_t bars[kTmaMaxStages + 1];   // [stages] = the gammas
    __shared__ int issued[kTmaMaxStages];
    __shared__ int consumed[kTmaMaxStages];
    const unsigned cl = cluster_nctarank();
    const unsigned crank = cluster_ctarank();
    const int64_t slice = a.n / cl;                    // elements of a row per CTA
    const uint32_t sb = static_cast<uint32_t>(slice * T::kBytes);
    const int64_t svec = slice / VEC;
    unsigned char *const gsm = smem;
    unsigned char *const stage0 = smem + NG * sb;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int64_t first = a.row0 + cluster_index_x();
    const int64_t step = cluster_count_x();
    const int64_t my_rows = first < a.rows_end ? (a.rows_end - first + step - 1) / step : 0;
    const int64_t row_bytes = a.n * T::kBytes;
    const int64_t soff = static_cast<int64_t>(crank) * sb;   // this CTA's slice in a row
    const char *const xg = static_cast<const char *>(a.x) + soff;
    const char *const rg = static_cast<const char *>(a.res) + soff;
    const bool bad_stages = stages < 1 || stages > kTmaMaxStages;

    if (tid == 0) {
        for (int st = 0; st <= stages && st <= kTmaMaxStages; ++st) mbar_init(&bars[st], 1);
        for (int st = 0; st < kTmaMaxStages; ++st) issued[st] = consumed[st] = 0;
        for (int q = 0; q < 2; ++q) {
            mbar_init(&mail1.bar[q], 1);
            mbar_init(&mail2.bar[q], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();   // (thread 0: after its initialisation and fence)
    pdl_enter();   // (the shared-memory set-up above overlapped the previous grid)
    if (tid == 0 && my_rows > 0 && !bad_stages) {
        mbar_arrive_expect_tx(&bars[stages], NG * sb + a.stall_bytes);   // (test hook: 0)
        bulk_to_shared(gsm, static_cast<const char *>(a.g1) + soff, sb, &bars[stages]);
        if (NG == 2) bulk_to_shared(gsm + sb, static_cast<const char *>(a.g2) + soff, sb,
                                    &bars[stages]);
        for (int st = 0; st < stages && st < my_rows; ++st) {
            stage_row<NS>(stage0 + st * NS * sb, xg, rg, (first + st * step) * row_bytes, sb, sb,
                          &bars[st]);
            issued[st] = 1;
        }
    }
    // (the host never launches bad_stages; the kernel then only votes to stop)
    int failed = bad_stages ? 1 : ((my_rows > 0 && !mbar_wait_bounded(&bars[stages], 0)) ? 1 : 0);
    const float sc = load_out_scale<OP, T>(a.scale);
    bool first_sum = true;
    int stopped = 0;           // 1 / 2: stopped at the first / second exchange of row stop_it
    int64_t stop_it = 0;

    for (int64_t it = 0; it < my_rows; ++it) {
        const int s = bad_stages ? 0 : static_cast<int>(it % stages);
        const uint32_t parity = bad_stages ? 0u : static_cast<uint32_t>((it / stages) & 1);
        const int64_t row = first + it * step;
        if (!failed && !mbar_wait_bounded(&bars[s], parity)) failed = 1;

        Fr xv[K];
        Fr rv[K];
        const unsigned char *sp = stage0 + s * NS * sb;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = tid + static_cast<int64_t>(k) * nt;
            if (v < svec && !failed) {
                ld_shared(xv[k], sp + v * 16);
                if (NS == 2) ld_shared(rv[k], sp + sb + v * 16);
            } else {
                xv[k].zero();
                rv[k].zero();
            }
        }
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) ss += frag_sum_sq(xv[k]);
        int stop;
        const float tot = cluster_row_sum(ss, mail1, cl, crank, it, failed, &stop, &failed,
                                          first_sum);
        first_sum = false;
        if (stop) {
            stopped = 1;
            stop_it = it;
            break;
        }
        // Every thread holds its part of the stage now (the barrier above): refill it.
        if (tid == 0) {
            consumed[s] += 1;
            if (it + stages < my_rows) {
                fence_proxy_async_smem();
                stage_row<NS>(stage0 + s * NS * sb, xg, rg,
                              (first + (it + stages) * step) * row_bytes, sb, sb, &bars[s]);
                issued[s] += 1;
            }
        }
        const float inv1 = inv_rms(tot, a.n, a.eps1);
        const int64_t row_elem = row * a.n + static_cast<int64_t>(crank) * slice;
        if (OP != kSandwich) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t v = tid + static_cast<int64_t>(k) * nt;
                if (v >= svec) continue;
                Fr g;
                ld_shared(g, gsm + v * 16);
                st_global(elem_ptr<T>(a.y, row_elem + v * VEC),
                          single_norm_output<OP>(xv[k], inv1, g, rv[k], sc));
            }
            continue;
        }
        float ss2 = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = tid + static_cast<int64_t>(k) * nt;
            if (v >= svec) continue;
            Fr g;
            ld_shared(g, gsm + v * 16);
            rv[k] = apply_norm_add(xv[k], inv1, g, rv[k]);
            st_global(elem_ptr<T>(a.y, row_elem + v * VEC), rv[k]);
            ss2 += frag_sum_sq(rv[k]);
        }
        int stop2;
        const float tot2 = cluster_row_sum(ss2, mail2, cl, crank, it, 0, &stop2, &failed, false);
        if (stop2) {
            stopped = 2;
            stop_it = it;
            break;
        }
        const float inv2 = inv_rms(tot2, a.n, a.eps2);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t v = tid + static_cast<int64_t>(k) * nt;
            if (v >= svec) continue;
            Fr g;
            ld_shared(g, gsm + sb + v * 16);
            st_global(elem_ptr<T>(a.y2, row_elem + v * VEC), apply_norm(rv[k], inv2, g));
        }
    }
    if (first_sum) cluster_wait_acquire();   // (no row: complete the start-up arrive)

    // Exit: after a stop, wait (bounded) for this CTA's copies still in flight
    // before it leaves its shared memory.  Then one cluster barrier: every
    // peer has issued all its messages once it is past it.  After a timed-out
    // message wait, the late message may still be landing: wait (bounded) for
    // that mailbox phase once more before leaving.
    const int any_timeout = __syncthreads_or(failed);
    if (tid == 0 && my_rows > 0 && stopped) {
        if (any_timeout) atomicAdd(&g_wait_timeouts, 1u);
        if (!bad_stages) {
            (void)mbar_wait_bounded(&bars[stages], 0);
            for (int st = 0; st < stages; ++st) {
                if (issued[st] > consumed[st])
                    (void)mbar_wait_bounded(&bars[st], static_cast<uint32_t>(consumed[st] & 1));
            }
        }
    }
    cluster_arrive_relaxed();
    cluster_wait_acquire();
    if (tid == 0 && stopped && any_timeout) {
        ClusterMail &m = stopped == 1 ? mail1 : mail2;
        (void)mbar_wait_bounded_cluster(&m.bar[stop_it & 1],
                                        static_cast<uint32_t>((stop_it >> 1) & 1));
    }
}

// Persistent grid of the staged kernel: as many CTAs as fit on the device
// (SM count x CTAs per SM), at most one per row.  Occupancy answers are
// cached per (kernel, threads, shared bytes); the SM count per device.
inline int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int count = 0;
    if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < 64) cached[dev] = count;
    return count;
}

// Per-kernel, per-device launch facts of the staged kernel, cached after the
// first launch: the dynamic shared memory it was opened up to, and the CTAs
// per SM at the last (threads, shared bytes) asked for.  Races between
// threads only repeat an idempotent runtime call.
constexpr int kMaxCachedDevices = 64;
struct TmaLaunchCache {
    std::atomic<int64_t> shared_opened{0};
    std::atomic<int64_t> occ_key{-1};
    std::atomic<int> occ_per_sm{0};
};

// Rows per launch, so that grid.x stays far below 2^31 - 1 for any cluster.
constexpr int64_t kRowsPerLaunch = int64_t(1) << 26;

// ---------------------------------------------------------------------------
// Host-side launch of one operation (instantiated once per .cu file).
// ---------------------------------------------------------------------------

using WarpKernelFn = void (*)(KernelArgs, int);
using CtaKernelFn = void (*)(KernelArgs);

template <int OP, class T, int VEC> struct KernelTable {
    static constexpr WarpKernelFn warp[kMaxK] = {
        mrn_rows_per_warp_kernel<OP, T, VEC, 1>, mrn_rows_per_warp_kernel<OP, T, VEC, 2>,
        mrn_rows_per_warp_kernel<OP, T, VEC, 3>, mrn_rows_per_warp_kernel<OP, T, VEC, 4>,
        mrn_rows_per_warp_kernel<OP, T, VEC, 5>, mrn_rows_per_warp_kernel<OP, T, VEC, 6>,
        mrn_rows_per_warp_kernel<OP, T, VEC, 7>, mrn_rows_per_warp_kernel<OP, T, VEC, 8>};
    static constexpr CtaKernelFn cta8() {
        if constexpr (OP == kRmsnorm && T::kBytes == 4) {
            return mrn_cta_kernel_k8x3<OP, T, VEC>;
        } else {
            return mrn_cta_kernel<OP, T, VEC, 8>;
        }
    }
    static constexpr CtaKernelFn cta[kMaxK] = {
        mrn_cta_kernel<OP, T, VEC, 1>, mrn_cta_kernel<OP, T, VEC, 2>,
        mrn_cta_kernel<OP, T, VEC, 3>, mrn_cta_kernel<OP, T, VEC, 4>,
        mrn_cta_kernel<OP, T, VEC, 5>, mrn_cta_kernel<OP, T, VEC, 6>,
        mrn_cta_kernel<OP, T, VEC, 7>, cta8()};
    static constexpr CtaKernelFn stream = mrn_stream_kernel<OP, T, VEC>;
};

template <int OP, class T> struct TmaTable {
    static constexpr WarpKernelFn fn[2][kMaxK] = {
        {mrn_tma_kernel<OP, T, 1, 1, false>, mrn_tma_kernel<OP, T, 2, 1, false>,
         mrn_tma_kernel<OP, T, 3, 1, false>, mrn_tma_kernel<OP, T, 4, 1, false>,
         mrn_tma_kernel<OP, T, 5, 1, false>, mrn_tma_kernel<OP, T, 6, 1, false>,
         mrn_tma_kernel<OP, T, 7, 1, false>, mrn_tma_kernel<OP, T, 8, 1, false>},
        {mrn_tma_kernel<OP, T, 1, 2, false>, mrn_tma_kernel<OP, T, 2, 2, false>,
         mrn_tma_kernel<OP, T, 3, 2, false>, mrn_tma_kernel<OP, T, 4, 2, false>,
         mrn_tma_kernel<OP, T, 5, 2, false>, mrn_tma_kernel<OP, T, 6, 2, false>,
         mrn_tma_kernel<OP, T, 7, 2, false>, mrn_tma_kernel<OP, T, 8, 2, false>}};
};
// Rows that are not 16-byte aligned: two warp groups only.
template <int OP, class T> struct TmaEdgeTable {
    static constexpr WarpKernelFn fn[kMaxK] = {
        mrn_tma_kernel<OP, T, 1, 2, true>, mrn_tma_kernel<OP, T, 2, 2, true>,
        mrn_tma_kernel<OP, T, 3, 2, true>, mrn_tma_kernel<OP, T, 4, 2, true>,
        mrn_tma_kernel<OP, T, 5, 2, true>, mrn_tma_kernel<OP, T, 6, 2, true>,
        mrn_tma_kernel<OP, T, 7, 2, true>, mrn_tma_kernel<OP, T, 8, 2, true>};
};

template <int OP, class T>
cudaError_t launch_tma(const Geometry &g, KernelArgs a, int64_t rows, cudaStream_t stream,
                       uint64_t *launches) {
    static TmaLaunchCache cache[kMaxCachedDevices][3][kMaxK];   // [groups - 1 | edge][k - 1]
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    TmaLaunchCache uncached;
    const bool edge = g.edge != 0;
    if (edge && (!op_has_edge_staging(OP) || g.groups != 2)) return cudaErrorInvalidConfiguration;
    const int gi = edge ? 2 : g.groups - 1;
    TmaLaunchCache &c =
        (dev >= 0 && dev < kMaxCachedDevices) ? cache[dev][gi][g.k - 1] : uncached;
    WarpKernelFn fn = nullptr;
    if constexpr (op_has_edge_staging(OP)) {
        fn = edge ? TmaEdgeTable<OP, T>::fn[g.k - 1] : TmaTable<OP, T>::fn[gi][g.k - 1];
    } else {
        fn = TmaTable<OP, T>::fn[gi][g.k - 1];
    }
    a.stage_bytes = edge ? static_cast<uint32_t>(edge_stage_bytes(a.n * T::kBytes)) : 0u;
    const int64_t shared =
        tma_shared_bytes(OP, edge ? edge_stage_bytes(a.n * T::kBytes) : a.n * T::kBytes, g.stages);
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
    if (edge) {
        // a CTA's rows all start at one offset within 16 bytes (see mrn_tma_kernel)
        ctas = ctas / kEdgeGridMultiple * kEdgeGridMultiple;
        if (ctas < kEdgeGridMultiple) ctas = kEdgeGridMultiple;
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

template <int OP, class T> struct TmaClusterTable {
    static constexpr WarpKernelFn fn[kMaxK] = {
        mrn_tma_cluster_kernel<OP, T, 1>, mrn_tma_cluster_kernel<OP, T, 2>,
        mrn_tma_cluster_kernel<OP, T, 3>, mrn_tma_cluster_kernel<OP, T, 4>,
        mrn_tma_cluster_kernel<OP, T, 5>, mrn_tma_cluster_kernel<OP, T, 6>,
        mrn_tma_cluster_kernel<OP, T, 7>, mrn_tma_cluster_kernel<OP, T, 8>};
};

// Persistent grid of clusters: as many clusters as can be resident at once
// (cudaOccupancyMaxActiveClusters), at most one per row.
template <int OP, class T>
cudaError_t launch_tma_cluster(const Geometry &g, KernelArgs a, int64_t rows, cudaStream_t stream,
                               uint64_t *launches) {
    static TmaLaunchCache cache[kMaxCachedDevices][kMaxK];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    TmaLaunchCache uncached;
    TmaLaunchCache &c = (dev >= 0 && dev < kMaxCachedDevices) ? cache[dev][g.k - 1] : uncached;
    const WarpKernelFn fn = TmaClusterTable<OP, T>::fn[g.k - 1];
    const int64_t slice_bytes = a.n / g.cluster * T::kBytes;
    const int64_t shared = slice_bytes * (op_gammas(OP) + g.stages * op_row_inputs(OP));
    cudaError_t err;
    if (c.shared_opened.load(std::memory_order_relaxed) < shared) {
        err = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(shared));
        if (err != cudaSuccess) return err;
        c.shared_opened.store(shared, std::memory_order_relaxed);
    }
    if (g.cluster > 8) {   // (independent of the shared-memory size opened above)
        err = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(g.threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(shared);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(g.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int64_t clusters = g.ctas > 0 ? g.ctas / g.cluster : 0;
    if (clusters <= 0) {
        const int64_t key = shared * 4096 + g.threads * 16 + g.cluster;
        int resident = c.occ_key.load(std::memory_order_relaxed) == key
                           ? c.occ_per_sm.load(std::memory_order_relaxed) : 0;
        if (resident == 0) {
            cfg.gridDim = dim3(static_cast<unsigned>(g.cluster), 1, 1);
            err = cudaOccupancyMaxActiveClusters(&resident, fn, &cfg);
            if (err != cudaSuccess) return err;
            if (resident < 1) return cudaErrorInvalidConfiguration;
            c.occ_per_sm.store(resident, std::memory_order_relaxed);
            c.occ_key.store(key, std::memory_order_relaxed);
        }
        clusters = resident;
    }
    if (g.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    for (int64_t r0 = 0; r0 < rows; r0 += kRowsPerLaunch) {
        const int64_t nrows = rows - r0 < kRowsPerLaunch ? rows - r0 : kRowsPerLaunch;
        a.row0 = r0;
        a.rows_end = r0 + nrows;
        const int64_t nclusters = clusters < nrows ? clusters : nrows;
        cfg.gridDim = dim3(static_cast<unsigned>(nclusters * g.cluster), 1, 1);
        err = cudaLaunchKernelEx(&cfg, fn, a, g.stages);
        if (err != cudaSuccess) return err;
        ++*launches;
    }
    return cudaSuccess;
}

// Timeouts counted by this translation unit's kernels on the current device
// since the previous call.  The device counter is never reset (a reset
// racing with a kernel's atomicAdd could lose a count); the last value
// reported per device is kept on the host under a lock and the difference
// (modulo 2^32) is returned.
template <int OP> int take_wait_timeouts() {
    static std::mutex lock;
    static unsigned int reported[kMaxCachedDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxCachedDevices) return -1;
    std::lock_guard<std::mutex> guard(lock);
    unsigned int count = 0;
    if (cudaMemcpyFromSymbol(&count, g_wait_timeouts, sizeof(count)) != cudaSuccess) return -1;
    const unsigned int fresh = count - reported[dev];
    reported[dev] = count;
    return static_cast<int>(fresh & 0x7FFFFFFFu);
}


template <int OP, class T, int VEC>
cudaError_t launch_typed(const Geometry &g, KernelArgs a, int64_t rows, cudaStream_t stream,
                         uint64_t *launches) {
    using Tab = KernelTable<OP, T, VEC>;
    for (int64_t r0 = 0; r0 < rows; r0 += kRowsPerLaunch) {
        const int64_t nrows = rows - r0 < kRowsPerLaunch ? rows - r0 : kRowsPerLaunch;
        a.row0 = r0;
        a.rows_end = r0 + nrows;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        cfg.blockDim = dim3(g.threads, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 0;
        if (g.pdl) {
            attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
            ++cfg.numAttrs;
        }
        cudaError_t err;
        if (g.kind == kRowsPerWarp) {
            const int64_t rpc = g.threads / g.lanes;
            cfg.gridDim = dim3(static_cast<unsigned>((nrows + rpc - 1) / rpc), 1, 1);
            err = cudaLaunchKernelEx(&cfg, Tab::warp[g.k - 1], a, g.lanes);
        } else if (g.kind == kCta) {
            const CtaKernelFn fn = Tab::cta[g.k - 1];
            cfg.gridDim = dim3(static_cast<unsigned>(nrows * g.cluster), 1, 1);
            if (g.cluster > 1) {
                if (g.cluster > 8) {
                    err = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (err != cudaSuccess) return err;
                }
                cudaLaunchAttribute &c = attr[cfg.numAttrs++];
                c.id = cudaLaunchAttributeClusterDimension;
                c.val.clusterDim.x = static_cast<unsigned>(g.cluster);
                c.val.clusterDim.y = 1;
                c.val.clusterDim.z = 1;
            }
            err = cudaLaunchKernelEx(&cfg, fn, a);
        } else {
            cfg.gridDim = dim3(static_cast<unsigned>(nrows * g.cluster), 1, 1);
            if (g.cluster > 1) {
                if (g.cluster > 8) {
                    err = cudaFuncSetAttribute(reinterpret_cast<const void *>(Tab::stream),
                                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (err != cudaSuccess) return err;
                }
                cudaLaunchAttribute &c = attr[cfg.numAttrs++];
                c.id = cudaLaunchAttributeClusterDimension;
                c.val.clusterDim.x = static_cast<unsigned>(g.cluster);
                c.val.clusterDim.y = 1;
                c.val.clusterDim.z = 1;
            }
            err = cudaLaunchKernelEx(&cfg, Tab::stream, a);
        }
        if (err != cudaSuccess) return err;
        ++*launches;
    }
    return cudaSuccess;
}

template <int OP>
cudaError_t launch_op(bool bf16, const Geometry &g, const KernelArgs &a, int64_t rows,
                      cudaStream_t stream, uint64_t *launches) {
    if (g.kind == kTma && g.cluster > 1) {
        if constexpr (op_has_cluster_staging(OP)) {
            return bf16 ? launch_tma_cluster<OP, BF16>(g, a, rows, stream, launches)
                        : launch_tma_cluster<OP, F32>(g, a, rows, stream, launches);
        }
        return cudaErrorInvalidConfiguration;
    }
    if (g.kind == kTma) {
        return bf16 ? launch_tma<OP, BF16>(g, a, rows, stream, launches)
                    : launch_tma<OP, F32>(g, a, rows, stream, launches);
    }
    if (bf16) {
        return g.vec == 1 ? launch_typed<OP, BF16, 1>(g, a, rows, stream, launches)
                          : launch_typed<OP, BF16, 8>(g, a, rows, stream, launches);
    }
    return g.vec == 1 ? launch_typed<OP, F32, 1>(g, a, rows, stream, launches)
                      : launch_typed<OP, F32, 4>(g, a, rows, stream, launches);
}

}  // namespace mrn
