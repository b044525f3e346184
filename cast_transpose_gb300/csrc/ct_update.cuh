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

#include "ct_internal.h"

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

// ---- deferred updates -------------------------------------------------------
// A run of K casts that share history column i, each of which would be
// followed by the update above, can defer the K updates to one pass after the
// run.  Cast j of the run max-merges its amax into pending row j instead of
// history row 0.  Write c_j for the amax that update j would have seen in
// row 0: pending row j, and for j = 0 also history row 0 (the slot cast 0
// would have merged into), merged the way the casts merge (the larger bit
// pattern).  With H the history before the run, update j sees the window
//   c_j, c_{j-1}, ..., c_0, H[1], ..., H[L-1-j]     (j < L),
// so its maximum is the larger of max(c_0 .. c_j) and max(H[1 .. L-1-j]);
// it replaces the scale by cand_j = (fp8_max / a_j) / 2^margin when the guard
// passes and keeps the previous one otherwise.  The scale after k updates is
// therefore cand_j of the latest j < k whose guard passes, or the scale before
// the run when none does.  (Which NaN a window keeps does not matter: any
// NaN fails the guard.)  The run's columns and positions: ct::PendingScale.

// NaN-propagating maximum (identity: -inf).
__device__ __forceinline__ float max_nan(float a, float b) {
    return (isnan(a) || isnan(b)) ? __int_as_float(0x7FFFFFFF) : fmaxf(a, b);
}

// The scale after ps.k deferred updates, in every lane.  All 32 lanes of the
// warp must call it.  Every load is issued before any result is used (one
// round trip for histories of up to 32 + k rows): lane j holds c_j, lane i
// history row L - k + i (the rows that leave the windows one per update),
// and the lanes share the rows 1 .. L - k - 1 that every window keeps.
__device__ __forceinline__ float pending_scale_warp(const PendingScale& ps, int lane) {
    constexpr unsigned kAll = 0xFFFFFFFFu;
    const int k = ps.k;
    const float s0 = __ldcg(ps.scale0);
    if (k == 0) return s0;
    float c = -INFINITY, t = -INFINITY, h = -INFINITY;
    const int m0 = ps.L - k;   // first row that leaves the window (update k - 1 sees rows 1 .. m0)
    if (lane < k) {
        c = __ldcg(ps.pending + int64_t(lane) * ps.stride);
        if (lane == 0) c = __uint_as_float(max(__float_as_uint(c), __float_as_uint(__ldcg(ps.hist))));
        if (m0 + lane >= 1) t = __ldcg(ps.hist + int64_t(m0 + lane) * ps.stride);
    }
#pragma unroll 8
    for (int r = 1 + lane; r < m0; r += 32) h = max_nan(h, __ldcg(ps.hist + int64_t(r) * ps.stride));
    const float c_own = c;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h = max_nan(h, __shfl_xor_sync(kAll, h, off));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {   // inclusive prefix maxima over the lanes
        const float cu = __shfl_up_sync(kAll, c, off), tu = __shfl_up_sync(kAll, t, off);
        if (lane >= off) {
            c = max_nan(c, cu);
            t = max_nan(t, tu);
        }
    }
    // update j = lane: rows 1 .. L-1-j of H are the shared rows and tail rows 0 .. k-1-j
    const float tj = __shfl_sync(kAll, t, (k - 1 - lane) & 31);
    const float a = ps.most_recent ? c_own : max_nan(max_nan(c, h), tj);
    float cand = 0.0f;
    bool ok = false;
    if (lane < k && a > 0.0f && isfinite(a)) {
        cand = __fdiv_rn(__fdiv_rn(ps.fp8_max, a), ps.two_pow_margin);
        ok = isfinite(cand);
    }
    const unsigned valid = __ballot_sync(kAll, ok);
    if (valid == 0) return s0;
    return __shfl_sync(kAll, cand, 31 - __clz(valid));
}

// The scale a cast kernel casts with: *scale, or the deferred-update scale
// (uniform branch; with ps.hist set all 32 lanes must call it).
__device__ __forceinline__ float cast_scale(const float* scale, const PendingScale& ps, int lane) {
    return ps.hist != nullptr ? pending_scale_warp(ps, lane) : *scale;
}

// The K deferred updates of column i applied at once (one warp): scale and
// scale_inv as after update K - 1, the window slid by K rows (row 0 := 0,
// rows 1 .. K := c_{K-1} .. c_0, rows K+1 .. L-1 := H[1 .. L-1-K]) and the
// pending rows cleared.  Every read happens before any write.
__device__ __forceinline__ void apply_pending_warp(float* hist, float* pending, float* scale,
                                                   float* scale_inv, const PendingScale& ps,
                                                   int lane) {
    const float s = pending_scale_warp(ps, lane);
    const int K = ps.k, L = ps.L;
    float c = 0.0f;
    if (lane < K) {
        c = __ldcg(pending + int64_t(lane) * ps.stride);
        if (lane == 0) c = __uint_as_float(max(__float_as_uint(c), __float_as_uint(__ldcg(hist))));
    }
    float v[kUpdateRowsPerLane];
#pragma unroll
    for (int j = 0; j < kUpdateRowsPerLane; ++j) {
        const int r = lane + 32 * j;   // row r of H moves to row r + K
        v[j] = (r >= 1 && r + K < L) ? __ldcg(hist + int64_t(r) * ps.stride) : 0.0f;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kUpdateRowsPerLane; ++j) {
        const int r = lane + 32 * j;
        if (r >= 1 && r + K < L) hist[int64_t(r + K) * ps.stride] = v[j];
    }
    if (lane < K) {
        if (K - lane < L) hist[int64_t(K - lane) * ps.stride] = c;
        pending[int64_t(lane) * ps.stride] = 0.0f;
    }
    if (lane == 0) {
        hist[0] = 0.0f;
        *scale = s;
        *scale_inv = __fdiv_rn(1.0f, s);
    }
}

}  // namespace dev
}  // namespace ct
