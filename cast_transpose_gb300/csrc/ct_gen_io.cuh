// ct_gen_io.cuh -- loads and stores for any alignment: 8 bf16 (or 16 bytes)
// shifted out of the two aligned 16-byte blocks that cover them, and row
// segments of FP8 codes written as aligned 16-byte blocks whose bytes are
// gathered from neighbouring lanes (masked only at the two segment ends).
// Shared by the general kernels and by the direct-load kernel's transposed
// stores when rows is not a multiple of 16.
#pragma once

#include "ct_internal.h"

#include <cuda_runtime.h>
#include <stdint.h>

namespace ct {
namespace gen {

// Word k + j of w[0..7], k in 0..3 (static indexing only).
__device__ __forceinline__ uint32_t pick(const uint32_t (&w)[8], int j, int k) {
    const uint32_t a = w[j], b = w[j + 1], c = w[j + 2], d = w[j + 3];
    return k == 0 ? a : k == 1 ? b : k == 2 ? c : d;
}

// Zero the elements n..7 of an 8-element chunk.
__device__ __forceinline__ uint4 keep_first(uint4 v, int n) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i >= n) w[i >> 1] &= (i & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 16 bytes that start at byte m (0..15) of the 32 held by lo, hi.
__device__ __forceinline__ uint4 extract16(const uint4& lo, const uint4& hi, int m) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const int k = m >> 2, sh = 8 * (m & 3);
    const uint32_t t0 = pick(w, 0, k), t1 = pick(w, 1, k), t2 = pick(w, 2, k),
                   t3 = pick(w, 3, k), t4 = pick(w, 4, k);
    return make_uint4(__funnelshift_r(t0, t1, sh), __funnelshift_r(t1, t2, sh),
                      __funnelshift_r(t2, t3, sh), __funnelshift_r(t3, t4, sh));
}

// Zero the bytes n..15.
__device__ __forceinline__ uint4 keep_first_bytes(uint4 v, int n) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i >= n) w[i >> 2] &= ~(0xFFu << (8 * (i & 3)));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Word i (0..3) of w, by selects (no indexed access, so w stays in registers).
__device__ __forceinline__ uint32_t word_of(const uint32_t (&w)[4], int i) {
    return i == 0 ? w[0] : i == 1 ? w[1] : i == 2 ? w[2] : w[3];
}

__device__ __forceinline__ uint8_t byte_of(const uint32_t (&w)[4], int i) {
    return static_cast<uint8_t>(word_of(w, i >> 2) >> (8 * (i & 3)));
}

// Store the K words d[0..K-1] (4K bytes) at dst, where h = dst & 3 is 1, 2
// or 3: the 4 - h head bytes, K - 1 whole aligned words shifted across
// registers (funnel shift by 8h bits), then the h tail bytes.
template <int K>
__device__ __forceinline__ void store_words_unaligned(uint8_t* dst, const uint32_t (&d)[K], int h) {
    const uint32_t first = d[0], last = d[K - 1];
    uint8_t* base = dst - h;   // 4-byte aligned
#pragma unroll
    for (int j = 1; j < K; ++j)
        reinterpret_cast<uint32_t*>(base)[j] = __funnelshift_r(d[j - 1], d[j], 8 * (4 - h));
    uint8_t* tail = base + 4 * K;
    if (h == 1) {
        dst[0] = static_cast<uint8_t>(first);
        *reinterpret_cast<uint16_t*>(dst + 1) = static_cast<uint16_t>(first >> 8);
        tail[0] = static_cast<uint8_t>(last >> 24);
    } else if (h == 2) {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(first);
        *reinterpret_cast<uint16_t*>(tail) = static_cast<uint16_t>(last >> 16);
    } else {
        dst[0] = static_cast<uint8_t>(first);
        *reinterpret_cast<uint16_t*>(tail) = static_cast<uint16_t>(last >> 8);
        tail[2] = static_cast<uint8_t>(last >> 24);
    }
}

// Bytes 0..n-1 of the 8 in q to dst.
__device__ __forceinline__ void store8(uint8_t* dst, uint2 q, int n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    if (n == 8) {
        if ((a & 7) == 0) {
            __stcs(reinterpret_cast<uint2*>(dst), q);
            return;
        }
        if ((a & 3) == 0) {
            reinterpret_cast<uint32_t*>(dst)[0] = q.x;
            reinterpret_cast<uint32_t*>(dst)[1] = q.y;
            return;
        }
        const uint32_t d[2] = {q.x, q.y};
        store_words_unaligned<2>(dst, d, static_cast<int>(a & 3));
        return;
    }
    const uint32_t w[4] = {q.x, q.y, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < n) dst[i] = byte_of(w, i);
}

// ---- row segments written as aligned 16-byte blocks ------------------------
// A row segment of L <= 128 bytes at any address `seg` is held in registers
// as 16-byte pieces (piece k = segment bytes [16k, 16k + 16)).  With m =
// seg & 15, the aligned 16-byte block k (address seg - m + 16k) holds segment
// bytes [16k - m, 16k - m + 16): the top m bytes of piece k - 1 and the low
// 16 - m bytes of piece k.  Every block is stored with one 16-byte store
// except those cut by the segment ends (the first, the last), whose bytes
// inside the segment are stored in aligned pieces of 8, 4, 2 and 1 bytes;
// no byte outside the segment is touched.

// Store bytes [lo, hi) of the 16 in w at blk (16-byte aligned), in aligned
// pieces.
__device__ __forceinline__ void store_range(uint8_t* blk, const uint32_t (&w)[4], int lo, int hi) {
    while (lo < hi) {
        const uint32_t wd = word_of(w, lo >> 2);
        if ((lo & 7) == 0 && lo + 8 <= hi) {
            *reinterpret_cast<uint2*>(blk + lo) = make_uint2(wd, word_of(w, (lo >> 2) + 1));
            lo += 8;
        } else if ((lo & 3) == 0 && lo + 4 <= hi) {
            *reinterpret_cast<uint32_t*>(blk + lo) = wd;
            lo += 4;
        } else if ((lo & 1) == 0 && lo + 2 <= hi) {
            *reinterpret_cast<uint16_t*>(blk + lo) = static_cast<uint16_t>(wd >> (8 * (lo & 3)));
            lo += 2;
        } else {
            blk[lo] = static_cast<uint8_t>(wd >> (8 * (lo & 3)));
            lo += 1;
        }
    }
}

// Block k of a segment (see above), given pieces k - 1 (`prev`, unused for
// k == 0) and k (`cur`); `last`: also store block k + 1 (the block after the
// last piece, holding its top m bytes) when the segment reaches into it.
__device__ __forceinline__ void store_block(uint8_t* seg, int L, int k, const uint32_t (&prev)[4],
                                            const uint32_t (&cur)[4], bool last) {
    const int m = static_cast<int>(reinterpret_cast<uintptr_t>(seg) & 15);
    if (16 * k - m >= L) return;                 // block entirely past the segment end
    uint8_t* blk = seg - m + 16 * k;
    if (m == 0) {
        if (16 * k + 16 <= L) __stcs(reinterpret_cast<uint4*>(blk), make_uint4(cur[0], cur[1], cur[2], cur[3]));
        else store_range(blk, cur, 0, L - 16 * k);
        return;
    }
    const uint4 v4 = extract16(make_uint4(prev[0], prev[1], prev[2], prev[3]),
                               make_uint4(cur[0], cur[1], cur[2], cur[3]), 16 - m);
    const uint32_t v[4] = {v4.x, v4.y, v4.z, v4.w};
    const int lo = k == 0 ? m : 0;
    const int hi = min(16, L - 16 * k + m);
    if (lo == 0 && hi == 16) __stcs(reinterpret_cast<uint4*>(blk), v4);
    else store_range(blk, v, lo, hi);
    if (last && L - 16 * k - 16 + m > 0) {      // block k + 1: top m bytes of piece k
        const uint4 t4 = extract16(make_uint4(cur[0], cur[1], cur[2], cur[3]),
                                   make_uint4(0u, 0u, 0u, 0u), 16 - m);
        const uint32_t t[4] = {t4.x, t4.y, t4.z, t4.w};
        store_range(blk + 16, t, 0, min(16, L - 16 * k - 16 + m));
    }
}

// Bytes [lo, 16) (head) or [0, hi) (tail) of the 16 in w at blk (16-byte
// aligned), 0 < lo, hi < 16: whole words with word stores, the one cut word
// with a byte and/or a 2-byte store; straight-line predicated code.
__device__ __forceinline__ void store_head(uint8_t* blk, const uint32_t (&w)[4], int lo) {
    const int w0 = (lo + 3) >> 2;   // first whole word
#pragma unroll
    for (int i = 1; i < 4; ++i)
        if (i >= w0) reinterpret_cast<uint32_t*>(blk)[i] = w[i];
    const int r = lo & 3;
    const uint32_t cut = word_of(w, lo >> 2);
    uint8_t* cw = blk + (lo & ~3);
    if (r == 1 || r == 3) cw[r] = static_cast<uint8_t>(cut >> (8 * r));
    if (r == 1 || r == 2) *reinterpret_cast<uint16_t*>(cw + 2) = static_cast<uint16_t>(cut >> 16);
}
__device__ __forceinline__ void store_tail(uint8_t* blk, const uint32_t (&w)[4], int hi) {
    const int w1 = hi >> 2;         // whole words [0, w1)
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (i < w1) reinterpret_cast<uint32_t*>(blk)[i] = w[i];
    const int r = hi & 3;
    const uint32_t cut = word_of(w, w1);
    uint8_t* cw = blk + 4 * w1;
    if (r >= 2) *reinterpret_cast<uint16_t*>(cw) = static_cast<uint16_t>(cut);
    if (r == 1) cw[0] = static_cast<uint8_t>(cut);
    if (r == 3) cw[2] = static_cast<uint8_t>(cut >> 16);
}

// Full 128-byte segments (the common case) in aligned blocks: lanes 1..7 of
// the group store block b, lane 0 the head block (its top 16 - m bytes) and
// lane 7 also the tail block (the low m bytes of block 8).  Shorter
// segments go through store_block.
__device__ __forceinline__ void store_segment_x8(uint8_t* seg, int L, const uint32_t (&w)[4],
                                                      int b) {
    uint32_t prev[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) prev[i] = __shfl_up_sync(0xFFFFFFFFu, w[i], 1, 8);
    if (L <= 0) return;
    const int m = static_cast<int>(reinterpret_cast<uintptr_t>(seg) & 15);
    if (L < 128) {
        store_block(seg, L, b, prev, w, b == 7);
        return;
    }
    uint8_t* blk = seg - m + 16 * b;
    if (m == 0) {
        __stcs(reinterpret_cast<uint4*>(blk), make_uint4(w[0], w[1], w[2], w[3]));
        return;
    }
    const uint4 v4 = extract16(make_uint4(prev[0], prev[1], prev[2], prev[3]),
                               make_uint4(w[0], w[1], w[2], w[3]), 16 - m);
    const uint32_t v[4] = {v4.x, v4.y, v4.z, v4.w};
    if (b == 0) store_head(blk, v, m);
    else __stcs(reinterpret_cast<uint4*>(blk), v4);
    if (b == 7) {   // block 8: the top m bytes of piece 7
        const uint4 t4 = extract16(make_uint4(w[0], w[1], w[2], w[3]), make_uint4(0u, 0u, 0u, 0u),
                                   16 - m);
        const uint32_t t[4] = {t4.x, t4.y, t4.z, t4.w};
        store_tail(blk + 16, t, m);
    }
}

// ---- whole aligned blocks of a tile's transpose ---------------------------
// A 128x128 tile whose qT segments start at any byte (rows % 16 != 0, or a
// misaligned out_t): column j's segment starts a_j = (out_t + col * rows +
// row0) % 16 bytes into a 16-byte block.  An interior tile row owns the
// rows [row0 - a_j, row0 + 128 - a_j) of column j, eight whole aligned
// blocks, the first of which holds up to 15 rows of the tile above (its
// halo); the first tile row owns [0, 128 - a_j) and the last [row0 - a_j,
// rows), cut at the column ends.  The caller leaves the transpose in a
// column-major copy: column j at j * kColCopyPitch, the 16 halo rows
// (row0 - 16 .. row0 - 1) first, then the tile's rows.
constexpr int kHaloRows = 16;
constexpr int kColCopyPitch = kHaloRows + kTileRows;

// Interior tile rows: the 4 columns of one store instruction lie sigma =
// 2^LSIG apart, sigma such that their a_j differ by 4 (mod 16), so that their
// 4-byte loads fall in 4 distinct bank classes (d = 0 or 8 excepted).
template <int LSIG>
__device__ __forceinline__ void store_col_copy_interior(uint8_t* out_t, int64_t rows, int64_t cols,
                                                        int64_t row0, int64_t col0, const uint8_t* sqt,
                                                        int a0, int d, int k, int g4, int warp) {
    const int jb = 16 * warp + (g4 << LSIG);
    const int ab = a0 + jb * d;
    const int64_t ncol_left = cols - col0 - jb;   // columns jb + dj < cols - col0 are stored
    uint8_t* const dst = out_t + (col0 + jb) * rows + row0 + 16 * k;
    const uint8_t* const src = sqt + jb * kColCopyPitch + kHaloRows + 16 * k;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        constexpr int kMask = (1 << LSIG) - 1;
        const int dj = ((it >> LSIG) << (LSIG + 2)) + (it & kMask);   // compile-time
        const int aj = (ab + dj * d) & 15;
        // the block's first byte: src + dj * pitch - aj (dj * pitch is a multiple of 4)
        const uint32_t* p = reinterpret_cast<const uint32_t*>(src + dj * kColCopyPitch - ((aj + 3) & ~3));
        const int sh = 8 * ((-aj) & 3);
        const uint32_t w0 = p[0], w1 = p[1], w2 = p[2], w3 = p[3], w4 = p[4];
        if (dj < ncol_left)
            __stcs(reinterpret_cast<uint4*>(dst + dj * rows - aj),
                   make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                              __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh)));
    }
}

// Stores of the blocks of columns 16 * warp .. 16 * warp + 15 (one warp):
// each block read back at its offset with five 4-byte loads and four funnel
// shifts, then one 16-byte store; blocks cut at a column end are stored in
// aligned pieces.  sqt needs 32 bytes of slack after the last column.
__device__ __forceinline__ void store_col_copy_blocks(uint8_t* out_t, int64_t rows, int64_t cols,
                                                      int64_t rt, int64_t row0, int64_t col0,
                                                      const uint8_t* sqt, int lane, int warp) {
    // a_j = (a0 + j * d) % 16 for column j of the tile
    const int d = static_cast<int>(rows & 15);
    const int a0 = static_cast<int>((reinterpret_cast<uintptr_t>(out_t) + col0 * rows + row0) & 15);
    const int k = lane & 7, g4 = lane >> 3;   // block k of column group g4
    const bool last = row0 + kTileRows >= rows;
    if (rt > 0 && !last) {
        if (d & 1)
            store_col_copy_interior<2>(out_t, rows, cols, row0, col0, sqt, a0, d, k, g4, warp);
        else if (d & 2)
            store_col_copy_interior<1>(out_t, rows, cols, row0, col0, sqt, a0, d, k, g4, warp);
        else
            store_col_copy_interior<0>(out_t, rows, cols, row0, col0, sqt, a0, d, k, g4, warp);
    } else {   // first or last tile row: blocks 0 .. 8, cut to the rows the tile owns
        const int L = static_cast<int>(last ? rows - row0 : kTileRows);
        for (int e = lane; e < 16 * 9; e += 32) {
            const int jq = e / 9, kk = e - 9 * jq, j = 16 * warp + jq;
            if (col0 + j >= cols) continue;
            const int aj = (a0 + j * d) & 15;
            const int blk_row = 16 * kk - aj;   // tile row of the block's first byte
            const int own_lo = rt > 0 ? -aj : 0, own_hi = last ? L : kTileRows - aj;
            const int lo = max(0, own_lo - blk_row), hi = min(16, own_hi - blk_row);
            if (lo >= hi) continue;
            const int s = kHaloRows + blk_row;
            const uint32_t* p = reinterpret_cast<const uint32_t*>(sqt + j * kColCopyPitch + (s & ~3));
            const int sh = 8 * (s & 3);
            const uint32_t v[4] = {__funnelshift_r(p[0], p[1], sh), __funnelshift_r(p[1], p[2], sh),
                                   __funnelshift_r(p[2], p[3], sh), __funnelshift_r(p[3], p[4], sh)};
            uint8_t* blk = out_t + (col0 + j) * rows + row0 + blk_row;
            if (lo == 0 && hi == 16) __stcs(reinterpret_cast<uint4*>(blk), make_uint4(v[0], v[1], v[2], v[3]));
            else store_range(blk, v, lo, hi);
        }
    }
}

}  // namespace gen

}  // namespace ct
