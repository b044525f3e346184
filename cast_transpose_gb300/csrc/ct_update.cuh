// ct_update.cuh -- the delayed-scaling update of one amax-history column
// ("[PyTorch] Refactor FP8 workspaces in linear modules", Motivations: the
// scale update kernel and the too-tiny-amax / infinite-scale case), shared
// by the update kernels.
//
// For column i of a history H[L][stride] (row 0 = the amax of the step that
// just ran):
//   a = max over the L rows (NaN propagates, the first NaN is kept; among
//       equal values the earliest row is kept),
//   s = (fp8_max / a) / 2^margin in fp32, kept only when a > 0, a finite and
//       s finite -- otherwise the old scale stays,
//   scale_inv = 1 / scale,
//   then the window slides: row r takes row r-1 (r = L-1 .. 1), row 0 := 0.
// The "most recent" rule takes a = row 0 alone instead of the maximum.
// Loads go through L2 (ld.global.cg): the amaxes were merged there by the
// cast kernels' atomics.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ct {
namespace dev {

__device__ __forceinline__ void finish_scale(float a, float s_old, float fp8_max,
                                             float two_pow_margin, float* scale,
                                             float* scale_inv) {
    float s = s_old;
    if (a > 0.0f && isfinite(a)) {
        const float cand = __fdiv_rn(__fdiv_rn(fp8_max, a), two_pow_margin);
        if (isfinite(cand)) s = cand;
    }
    *scale = s;
    *scale_inv = __fdiv_rn(1.0f, s);
}

// (value, row) candidate order of the history maximum: a NaN beats any
// number and an earlier NaN beats a later one; otherwise the larger value
// wins and equal values go to the earlier row.  This is exactly the result
// of scanning the rows in order, keeping the first NaN or a strictly larger
// value, so any reduction tree gives the same bits.
__device__ __forceinline__ bool better(float va, int ra, float vb, int rb) {
    const bool na = isnan(va), nb = isnan(vb);
    if (na || nb) return na && (!nb || ra < rb);
    if (va != vb) return va > vb;
    return ra < rb;
}

// Warp-cooperative update of one column, L <= 32 * kUpdateRowsPerLane.  Lane l
// holds rows l, l+32, ...; every read happens before any write, so the update
// costs one round trip to memory.  All 32 lanes must call it.
constexpr int kUpdateRowsPerLane = 32;

// most_recent != 0: a is row 0 alone (the "most recent" rule); the window
// still slides.
__device__ __forceinline__ void update_column_warp(float* hist, int64_t stride, int L, float* scale,
                                                   float* scale_inv, float fp8_max,
                                                   float two_pow_margin, int lane,
                                                   int most_recent = 0) {
    float v[kUpdateRowsPerLane];
    float best = __int_as_float(0x7FFFFFFF);
    int best_r = -1;
    const float s_old = lane == 0 ? __ldcg(scale) : 0.0f;   // same round trip as the history
#pragma unroll
    for (int j = 0; j < kUpdateRowsPerLane; ++j) {
        const int r = lane + 32 * j;
        if (r < L) {
            v[j] = __ldcg(hist + int64_t(r) * stride);
            if (best_r < 0 || better(v[j], r, best, best_r)) {
                best = v[j];
                best_r = r;
            }
        }
    }
    if (most_recent) {
        best = v[0];   // lane 0 holds row 0; only lane 0 uses `best` below
    } else {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, best, off);
            const int orr = __shfl_xor_sync(0xFFFFFFFFu, best_r, off);
            if (orr >= 0 && (best_r < 0 || better(ov, orr, best, best_r))) {
                best = ov;
                best_r = orr;
            }
        }
    }
    if (lane == 0) finish_scale(best, s_old, fp8_max, two_pow_margin, scale, scale_inv);
#pragma unroll
    for (int j = 0; j < kUpdateRowsPerLane; ++j) {
        const int r = lane + 32 * j;
        if (r + 1 < L) hist[int64_t(r + 1) * stride] = v[j];
    }
    if (lane == 0) hist[0] = 0.0f;
}

// Any L, one thread, sequential scan.
__device__ __forceinline__ void update_column_serial(float* hist, int64_t stride, int L,
                                                     float* scale, float* scale_inv,
                                                     float fp8_max, float two_pow_margin,
                                                     int most_recent = 0) {
    float a = __ldcg(hist);
    for (int r = 1; r < L && !most_recent; ++r) {
        if (isnan(a)) break;
        const float v = __ldcg(hist + int64_t(r) * stride);
        if (isnan(v) || v > a) a = v;
    }
    finish_scale(a, __ldcg(scale), fp8_max, two_pow_margin, scale, scale_inv);
    for (int r = L - 1; r >= 1; --r) hist[int64_t(r) * stride] = __ldcg(hist + int64_t(r - 1) * stride);
    hist[0] = 0.0f;
}

}  // namespace dev
}  // namespace ct
