// ct_device.cuh -- small device helpers: FP8 conversion, mbarrier and TMA
// wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ct {
namespace dev {

// ---- FP8 conversion --------------------------------------------------------
// Two fp32 values to two FP8 codes with round-to-nearest-even and saturation
// to the largest finite value (the .satfinite form of the PTX cvt).  The
// result packs `lo` in bits 0-7 and `hi` in bits 8-15.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == 0) {
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// bf16 pair packed in a 32-bit word -> its two fp32 values (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two IEEE fp32 products a*s, b*s (round to nearest even, no flush to
// zero) with one packed f32x2 multiply of the sm_100 family.
__device__ __forceinline__ void mul2_rn(float a, float b, float s, float& ra, float& rb) {
    asm("{\n\t.reg .b64 ta, ts, td;\n\t"
        "mov.b64 ta, {%2, %3};\n\t"
        "mov.b64 ts, {%4, %4};\n\t"
        "mul.rn.f32x2 td, ta, ts;\n\t"
        "mov.b64 {%0, %1}, td;\n\t}"
        : "=f"(ra), "=f"(rb)
        : "f"(a), "f"(b), "f"(s));
}

// Cast 8 bf16 (one 16-byte vector) to 8 FP8 codes (two 32-bit words, byte i
// = element i).
template <int FMT>
__device__ __forceinline__ uint2 cast8(const uint4& v, float scale) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float a, b;
        mul2_rn(bf16_lo(w[e]), bf16_hi(w[e]), scale, a, b);
        h[e] = cvt_fp8x2<FMT>(a, b);
    }
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// ---- programmatic dependent launch ----------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation allowed.  It first lets the next kernel in the stream be
// scheduled (that kernel will itself wait below), then waits until every
// kernel it depends on has completed and its memory is visible, before it
// reads anything.  With an ordinary predecessor both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- shared-memory addresses, timers ----------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// about two seconds (returns false then).  A correct launch never gets
// near the limit; the bound only keeps a broken one from hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The same, but also gives up as soon as *abort becomes nonzero.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && (*abort || globaltimer_ns() - t0 > kWaitLimitNs)) return false;
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among the `count` threads of the consumer warps only (named
// barrier 1; barrier 0 is __syncthreads).
__device__ __forceinline__ void consumer_sync(int count) {
    asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory");
}

// Barrier among the 256 threads of thread group g of a CTA that runs several
// independent groups (named barrier 1 + g).
__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, 256;" ::"r"(1 + g) : "memory");
}

// ---- compensated summation -----------------------------------------------------
// Kahan sum in fp32 (error within a few fp32 ulps of the sum of magnitudes
// for any number of terms, without fp64, which runs at a small fraction of
// the fp32 rate on this GPU).  Once the running sum is not finite (an Inf or
// NaN among the terms) the correction is dropped, so the sum keeps the plain
// IEEE result (Inf, or NaN for Inf - Inf and NaN terms) instead of the
// Inf - Inf of the correction term.
struct Kahan {
    float sum = 0.0f, comp = 0.0f;
    __device__ __forceinline__ void add(float v) {
        const float y = __fsub_rn(v, comp);
        const float t = __fadd_rn(sum, y);
        comp = isfinite(t) ? __fsub_rn(__fsub_rn(t, sum), y) : 0.0f;
        sum = t;
    }
};

// ---- TMA ---------------------------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled bulk tensor load into shared memory; completion is signalled on
// `bar` as transaction bytes.  x is the innermost (column) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled bulk tensor prefetch into L2: no shared memory and no completion
// signal, only a hint.  L2 is where every write of the GPU lands, so a line
// prefetched before its last write is simply updated by it: a prefetch can
// never make a later read see stale data.  Same coordinate rules as the load.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global
// address into L2: a hint with no completion signal; a later write to the
// same lines updates them in L2, so it cannot make a read stale.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- 4x4 byte transpose ------------------------------------------------------
// r0..r3 hold rows 0..3 of a 4x4 byte block (byte k = column k); on return
// c0..c3 hold its columns (byte i = row i).
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                             uint32_t& c0, uint32_t& c1, uint32_t& c2,
                                             uint32_t& c3) {
    const uint32_t t0 = __byte_perm(r0, r1, 0x5140);  // r0.b0 r1.b0 r0.b1 r1.b1
    const uint32_t t1 = __byte_perm(r2, r3, 0x5140);  // r2.b0 r3.b0 r2.b1 r3.b1
    const uint32_t t2 = __byte_perm(r0, r1, 0x7362);  // r0.b2 r1.b2 r0.b3 r1.b3
    const uint32_t t3 = __byte_perm(r2, r3, 0x7362);  // r2.b2 r3.b2 r2.b3 r3.b3
    c0 = __byte_perm(t0, t1, 0x5410);
    c1 = __byte_perm(t0, t1, 0x7632);
    c2 = __byte_perm(t2, t3, 0x5410);
    c3 = __byte_perm(t2, t3, 0x7632);
}

// Shared-memory layout of the FP8 copy of a 128x128 tile used for the
// transposed write: 128 rows of 32 words (4 FP8 codes each); word wd of row r
// lives at wd ^ swz(r).  The XOR spreads the 8 row blocks that the transpose
// pass reads at once over all 32 banks, and keeps the two words of every
// 8-byte row store adjacent (swz is even).
__device__ __forceinline__ int swz(int r) { return 2 * ((r >> 3) & 15); }

// Column-sum scratch of one tile: the 8 warps' sums of 128 columns.  Warp
// w's 16 active lanes (chunk c) store columns 8c .. 8c+3 as one float4 at
// w * kColsumStride + 4c and columns 8c+4 .. 8c+7 at w * kColsumStride + 80 +
// 4c, so each store instruction covers 256 contiguous bytes (no bank
// conflict) and the reads of 32 consecutive columns fall in 32 banks.
constexpr int kColsumStride = 160;
__device__ __forceinline__ int colsum_index(int w, int col) {
    return w * kColsumStride + ((col & 7) >> 2) * 80 + 4 * (col >> 3) + (col & 3);
}
__device__ __forceinline__ void colsum_store(float* colsum, int warp, int c, const float (&cs)[8]) {
    float* base = colsum + warp * kColsumStride + 4 * c;
    *reinterpret_cast<float4*>(base) = make_float4(cs[0], cs[1], cs[2], cs[3]);
    *reinterpret_cast<float4*>(base + 80) = make_float4(cs[4], cs[5], cs[6], cs[7]);
}

// ---- asynchronous copies into shared memory ----------------------------------
// 16-byte copy from global (16-byte aligned) to shared memory, bypassing L1;
// only the first src_bytes (1..16) are read, the rest of the 16 is zero.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Max of the two bf16 magnitudes (sign cleared) of a packed pair, kept as a
// pair: one AND and one native 16x2 unsigned max per word.
__device__ __forceinline__ uint32_t absmax_pair(uint32_t acc, uint32_t w) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w & 0x7FFF7FFFu));
    return r;
}

// Collapse a pair accumulator into the fp32 bit pattern of the larger
// magnitude (bf16 widened to fp32).
__device__ __forceinline__ uint32_t pair_to_f32_bits(uint32_t acc) {
    const uint32_t a = acc & 0xFFFFu, b = acc >> 16;
    return (a > b ? a : b) << 16;
}

}  // namespace dev
}  // namespace ct
