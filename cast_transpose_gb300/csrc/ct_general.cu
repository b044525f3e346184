// ct_general.cu -- kernels for the cases the TMA path does not take, and the
// small kernels around it (sm_103a):
//   * general_cast_kernel: cast (+ transpose, + dbias partials) of a bf16
//     matrix of ANY shape and alignment, 128x128 tiles, widest aligned
//     loads and stores;
//   * dbias_finish_kernel: db[j] = sum over 128-row tiles of the partials,
//     compensated fp32, in a fixed order (deterministic), stored as fp32 or
//     rounded to bf16;
//   * scale_update_kernel: the delayed-scaling update of "[PyTorch] Refactor
//     FP8 workspaces in linear modules" (Motivations: scale update kernel,
//     infinite-scale case), one thread per tensor;
//   * transpose kernels for FP8 bytes (the lazy transpose-cache fill of the
//     same page), a 128x128-tile vectorised one for aligned shapes and a
//     128x128-tile one for any shape and alignment.
#include "ct_device.cuh"
#include "ct_internal.h"
#include "ct_gen_io.cuh"
#include "ct_update.cuh"

#include <cuda_bf16.h>

#include <cmath>
#include <mutex>


namespace ct {
namespace {

// ---------------------------------------------------------------------------
// General cast: any shape, x 2-byte aligned, out and out_t 1-byte aligned.
// Tile 128x128, 256 threads, the thread mapping of the direct-load kernel
// (pass 1: 8-column chunk c of rows rg + 16*it; pass 2: 16-row x 4-column
// byte blocks).  No byte outside the caller's buffers is touched:
//   * staging: the segment of each tile row in x (up to 256 bytes starting
//     at any even byte) is copied into shared memory as the aligned 16-byte
//     chunks that cover it, up to 17, with cp.async (nothing held in
//     registers while the copies are in flight); a chunk
//     that crosses the end of x copies only the bytes up to it, and the one
//     chunk that can start before x (its first) is read element by element;
//   * pass 1: the 8 elements of chunk c are five aligned 4-byte words of the
//     staged row, shifted by a uniform byte permute; amax, column sums and
//     cast as in the direct kernel;
//     elements past the row end are zeroed (they belong to the next row);
//     q is stored 8 bytes per thread, as aligned words shifted across
//     registers plus a short head and tail where the address is not aligned
//     (gen::store8);
//   * pass 2: the transposed 16-row blocks; when rows is a multiple of 16
//     and out_t is 16-byte aligned every block is one aligned 16-byte store,
//     otherwise each column's segment of qT is written as aligned 16-byte
//     blocks gathered from neighbouring lanes (gen::store_segment_x8).
// Measured on GB300 (8191x12287, both dimensions odd): 3.48 TB/s, limited by
// instruction issue on the integer pipe (ALU 64% of peak, 79% of scheduler
// cycles issue, DRAM 36% busy): the shifts and partial stores that
// misalignment costs.  Measured and dropped: aligned-block stores for q and
// qT with the end blocks written by a loop (1.63 TB/s); per-thread unaligned
// 16-byte stores of qT (2.98); q and qT written as aligned blocks from
// shared-memory words in a phase of their own after pass 1 (2.80).
constexpr int kStageRow = 17 * 16;   // staged bytes per tile row
constexpr int kGenSmem = kTileRows * kStageRow + kTileRows * kTileCols;
constexpr int kGenSmemDbias = kGenSmem + 8 * dev::kColsumStride * 4;

// One 16-byte staging chunk of x at src (16-byte aligned) into dst, if it
// holds bytes of the row segment that ends at send: a cp.async for the bytes
// inside x, or element loads for the first chunk of x when it starts before
// x.
__device__ __forceinline__ void stage_chunk(uint8_t* dst, uintptr_t src, uintptr_t send,
                                            uintptr_t xbeg, uintptr_t xend) {
    if (src >= send) return;   // past the segment
    if (src < xbeg) {
        uint32_t e[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uintptr_t ad = src + 2 * i;
            if (ad >= xbeg && ad < xend)
                e[i >> 1] |= uint32_t(*reinterpret_cast<const uint16_t*>(ad)) << (16 * (i & 1));
        }
        *reinterpret_cast<uint4*>(dst) = make_uint4(e[0], e[1], e[2], e[3]);
        return;
    }
    const uintptr_t left = xend - src;   // > 0: src is inside the segment
    dev::cp_async16(dst, reinterpret_cast<const void*>(src), left < 16 ? static_cast<int>(left) : 16);
}

template <int FMT, bool DBIAS>
__global__ void __launch_bounds__(256, DBIAS ? 3 : 4) general_cast_kernel(GeneralArgs a) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (a.noop != nullptr && *a.noop != 0.0f) return;
    extern __shared__ __align__(16) uint8_t gsmem[];
    uint8_t* xs = gsmem;                                   // [128][kStageRow]
    uint8_t* sq = gsmem + kTileRows * kStageRow;           // swizzled FP8 copy
    float* colsum = reinterpret_cast<float*>(sq + kTileRows * kTileCols);
    __shared__ unsigned s_amax[8];

    const int64_t rows = a.rows, cols = a.cols;
    const int64_t tiles_c = (cols + kTileCols - 1) / kTileCols;
    const int64_t tiles = ((rows + kTileRows - 1) / kTileRows) * tiles_c;
    const uintptr_t xbeg = reinterpret_cast<uintptr_t>(a.x);
    const uintptr_t xend = xbeg + 2 * uintptr_t(rows) * uintptr_t(cols);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid & 15, rg = tid >> 4;
    const int b = lane & 7, w = warp * 4 + (lane >> 3);
    const float scale = dev::cast_scale(a.scale, a.pend, lane);

    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t rt = tile / tiles_c;
        const int64_t row0 = rt * kTileRows, col0 = (tile - rt * tiles_c) * kTileCols;
        const int nrow = static_cast<int>(rows - row0 < kTileRows ? rows - row0 : kTileRows);
        const int ncol = static_cast<int>(cols - col0 < kTileCols ? cols - col0 : kTileCols);

        // ---- staging of the tile's row segments: consecutive threads on
        // consecutive chunks (17 per row), so each copy instruction of a warp
        // covers about two rows of contiguous chunks ----
        for (int i = tid; i < kTileRows * 17; i += 256) {
            const int r = i / 17, u = i - 17 * r;
            if (r >= nrow) break;
            const uintptr_t s0 = xbeg + 2 * uintptr_t((row0 + r) * cols + col0);
            stage_chunk(xs + r * kStageRow + 16 * u, (s0 & ~uintptr_t(15)) + 16 * uintptr_t(u),
                        s0 + 2 * uintptr_t(ncol), xbeg, xend);
        }
        dev::cp_async_wait_all();
        __syncthreads();

        // ---- pass 1: amax, column sums, cast, q and the FP8 copy ----
        uint32_t amax_pair = 0;
        float cs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) cs[j] = 0.0f;
        const int nv = ncol - 8 * c <= 0 ? 0 : (ncol - 8 * c >= 8 ? 8 : ncol - 8 * c);
        // Byte offset (even) of this thread's row segments within their first
        // staged chunk: the same for rows rg + 16*it (16 rows of x are a
        // multiple of 16 bytes).  Its 8 elements are words wo .. wo+4 of the
        // staged chunks, shifted by 2 bytes when mx % 4 == 2: five aligned
        // 4-byte shared loads and four byte permutes with a uniform selector.
        const int mx = static_cast<int>((xbeg + 2 * uintptr_t((row0 + rg) * cols + col0)) & 15);
        const int wo = mx >> 2;
        const uint32_t sel = (mx & 2) ? 0x5432u : 0x3210u;
#pragma unroll 2
        for (int it = 0; it < 8; ++it) {
            const int r = rg + 16 * it;
            const int64_t row = row0 + r;
            const int n = r < nrow ? nv : 0;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n > 0) {
                const uint32_t* rp = reinterpret_cast<const uint32_t*>(xs + r * kStageRow + 16 * c) + wo;
                const uint32_t w0 = rp[0], w1 = rp[1], w2 = rp[2], w3 = rp[3], w4 = rp[4];
                v = make_uint4(__byte_perm(w0, w1, sel), __byte_perm(w1, w2, sel),
                               __byte_perm(w2, w3, sel), __byte_perm(w3, w4, sel));
                if (n < 8) v = gen::keep_first(v, n);
            }
            amax_pair = dev::absmax_pair(amax_pair, v.x);
            amax_pair = dev::absmax_pair(amax_pair, v.y);
            amax_pair = dev::absmax_pair(amax_pair, v.z);
            amax_pair = dev::absmax_pair(amax_pair, v.w);
            if constexpr (DBIAS) {
                cs[0] += dev::bf16_lo(v.x); cs[1] += dev::bf16_hi(v.x);
                cs[2] += dev::bf16_lo(v.y); cs[3] += dev::bf16_hi(v.y);
                cs[4] += dev::bf16_lo(v.z); cs[5] += dev::bf16_hi(v.z);
                cs[6] += dev::bf16_lo(v.w); cs[7] += dev::bf16_hi(v.w);
            }
            const uint2 q8 = dev::cast8<FMT>(v, scale);
            if (a.out != nullptr && n > 0) gen::store8(a.out + row * cols + col0 + 8 * c, q8, n);
            *reinterpret_cast<uint2*>(sq + r * kTileCols + ((2 * c) ^ dev::swz(r)) * 4) = q8;
        }
        const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
        if (lane == 0) s_amax[warp] = m;
        if constexpr (DBIAS) {
#pragma unroll
            for (int j = 0; j < 8; ++j) cs[j] += __shfl_xor_sync(0xFFFFFFFFu, cs[j], 16);
            if (lane < 16) dev::colsum_store(colsum, warp, c, cs);
        }
        __syncthreads();

        if (tid == 0) {
            unsigned am = s_amax[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) am = am > s_amax[j] ? am : s_amax[j];
            if (am != 0) atomicMax(reinterpret_cast<unsigned*>(a.amax), am);
            if (tile == 0) *a.scale_inv = __fdiv_rn(1.0f, scale);
        }
        if constexpr (DBIAS) {
            if (tid < kTileCols && col0 + tid < cols) {
                float sum = colsum[dev::colsum_index(0, tid)];
#pragma unroll
                for (int j = 1; j < 8; ++j) sum += colsum[dev::colsum_index(j, tid)];
                a.partial[rt * cols + col0 + tid] = sum;
            }
        }

        // ---- pass 2: transposed 16-row blocks of four columns ----
        if (a.out_t != nullptr) {
            const uint32_t* sq32 = reinterpret_cast<const uint32_t*>(sq);
            uint32_t rw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * b + j;
                rw[j] = sq32[r * (kTileCols / 4) + (w ^ dev::swz(r))];
            }
            uint32_t o[4][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                dev::transpose4x4(rw[4 * g], rw[4 * g + 1], rw[4 * g + 2], rw[4 * g + 3], o[0][g],
                                  o[1][g], o[2][g], o[3][g]);
            if ((rows & 15) == 0 && (reinterpret_cast<uintptr_t>(a.out_t) & 15) == 0) {
                // every column's segment of qT starts on a 16-byte boundary
                if (16 * b < nrow) {
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        const int64_t col = col0 + 4 * w + kq;
                        if (col < cols)
                            __stcs(reinterpret_cast<uint4*>(a.out_t + col * rows + row0 + 16 * b),
                                   make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]));
                    }
                }
            } else {
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const int64_t col = col0 + 4 * w + kq;
                    gen::store_segment_x8(a.out_t + col * rows + row0, col < cols ? nrow : 0, o[kq], b);
                }
            }
        }
        __syncthreads();   // the staging, sq, colsum and s_amax are reused by the next tile
    }
}

// ---------------------------------------------------------------------------
// db[j] = sum over the `runs` partial rows of partial[t, j] (one row per
// band of tile rows, see dbias_units).  Block = 32 columns x 8 row groups;
// each thread sums every 8th partial row of its column (its loads for 64
// rows issued together, one round trip to L2), then the 8 group sums are
// added in a fixed order (deterministic), all compensated (dev::Kahan).
using dev::Kahan;

template <bool BF16_OUT>
__global__ void __launch_bounds__(256) dbias_finish_kernel(const float* __restrict__ partial,
                                                           int64_t runs, int64_t cols,
                                                           void* __restrict__ db,
                                                           const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ float part[8][32];
    __shared__ float comp[8][32];
    const int c = threadIdx.x & 31, g = threadIdx.x >> 5;
    for (int64_t col0 = int64_t(blockIdx.x) * 32; col0 < cols; col0 += int64_t(gridDim.x) * 32) {
        const int64_t j = col0 + c;
        Kahan k;
        if (j < cols) {   // eight rows per thread per batch, all loads issued first
            for (int64_t t0 = 0; t0 < runs; t0 += 64) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int64_t t = t0 + g + 8 * i;
                    v[i] = t < runs ? __ldcg(partial + t * cols + j) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (t0 + g + 8 * i < runs) k.add(v[i]);
            }
        }
        part[g][c] = k.sum;
        comp[g][c] = k.comp;
        __syncthreads();
        if (g == 0 && j < cols) {
            Kahan total;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                total.add(part[q][c]);
                total.add(-comp[q][c]);
            }
            if constexpr (BF16_OUT)
                static_cast<uint16_t*>(db)[j] = __bfloat16_as_ushort(__float2bfloat16_rn(total.sum));
            else
                static_cast<float*>(db)[j] = total.sum;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Delayed scaling (rule in ct_update.cuh): one warp per tensor for histories
// of up to 1024 rows, one thread per tensor beyond.
__global__ void __launch_bounds__(128) scale_update_warp_kernel(float* __restrict__ hist,
                                                                float* __restrict__ scale,
                                                                float* __restrict__ scale_inv,
                                                                int L, int n, int64_t stride,
                                                                float fp8_max,
                                                                float two_pow_margin,
                                                                int most_recent,
                                                                const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (i >= n) return;
    dev::update_column_warp(hist + i, stride, L, scale + i, scale_inv + i, fp8_max, two_pow_margin,
                            threadIdx.x & 31, most_recent);
}

__global__ void __launch_bounds__(128) scale_update_long_kernel(float* __restrict__ hist,
                                                                float* __restrict__ scale,
                                                                float* __restrict__ scale_inv,
                                                                int L, int n, int64_t stride,
                                                                float fp8_max,
                                                                float two_pow_margin,
                                                                int most_recent,
                                                                const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    dev::update_column_serial(hist + i, stride, L, scale + i, scale_inv + i, fp8_max,
                              two_pow_margin, most_recent);
}

// The K updates deferred by a run of casts (rule in ct_update.cuh), applied
// at once: one warp per tensor.
__global__ void __launch_bounds__(128) scale_update_pending_kernel(float* hist, float* pending,
                                                                   float* scale, float* scale_inv,
                                                                   int L, int K, int n,
                                                                   int64_t stride, float fp8_max,
                                                                   float two_pow_margin,
                                                                   int most_recent,
                                                                   const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (i >= n) return;
    const PendingScale ps{hist + i, scale + i, pending + i, stride, L, K, most_recent, fp8_max,
                          two_pow_margin};
    dev::apply_pending_warp(hist + i, pending + i, scale + i, scale_inv + i, ps, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// FP8 transpose, 128x128 byte tiles, 256 threads.  Loads are 16-byte row
// vectors; the tile is kept in shared memory with the same XOR swizzle as
// the cast kernel's FP8 copy (word w of row r at w ^ 4*(r/16)), so both the
// row-vector stores and the 16x4 column gathers are conflict-free.
// Tile schedule: without a noop flag one tile per CTA (loop_ctas == 0);
// with one, the first loop_ctas CTAs (one wave) take tiles b, b + loop_ctas,
// ... (loop_tiles each) and the CTAs after them one tile each of the rest,
// so a launch that its flag skips starts a few waves of CTAs.
__global__ void __launch_bounds__(256) transpose_fast_kernel(const uint8_t* __restrict__ in,
                                                             int64_t rows, int64_t cols,
                                                             uint8_t* __restrict__ out,
                                                             const float* noop, int64_t loop_ctas,
                                                             int64_t loop_tiles) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ __align__(16) uint32_t tile[kTileRows * (kTileCols / 4)];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t tiles_c = (cols + kTileCols - 1) / kTileCols;
    const int64_t tiles = ((rows + kTileRows - 1) / kTileRows) * tiles_c;
    int64_t first = blockIdx.x, stride = gridDim.x, count = tiles;
    if (loop_ctas > 0) {
        if (int64_t(blockIdx.x) < loop_ctas) {
            stride = loop_ctas;
            count = loop_tiles;
        } else {
            first = loop_ctas * loop_tiles + (blockIdx.x - loop_ctas);
            count = 1;
        }
    }
    int64_t t = first;
    for (int64_t k = 0; k < count && t < tiles; ++k, t += stride) {
        const int64_t rt = t / tiles_c;
        const int64_t row0 = rt * kTileRows, col0 = (t - rt * tiles_c) * kTileCols;
        // load: chunk ch (16 bytes = 4 words) of row r; 1024 chunks, 4 per thread
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i;
            const int r = idx >> 3, ch = idx & 7;
            const int64_t row = row0 + r, col = col0 + 16 * ch;
            v[i] = (row < rows && col < cols)
                       ? __ldg(reinterpret_cast<const uint4*>(in + row * cols + col))
                       : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i;
            const int r = idx >> 3, ch = idx & 7;
            *reinterpret_cast<uint4*>(&tile[r * 32 + ((4 * ch) ^ (4 * (r >> 4)))]) = v[i];
        }
        __syncthreads();
        const int b = lane & 7, w = warp * 4 + (lane >> 3);
        uint32_t rw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) rw[j] = tile[(16 * b + j) * 32 + (w ^ (4 * b))];
        uint32_t o[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
            dev::transpose4x4(rw[4 * g], rw[4 * g + 1], rw[4 * g + 2], rw[4 * g + 3], o[0][g],
                              o[1][g], o[2][g], o[3][g]);
        const int64_t row = row0 + 16 * b;
        if (row < rows) {
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const int64_t col = col0 + 4 * w + kq;
                if (col < cols)
                    *reinterpret_cast<uint4*>(out + col * rows + row) =
                        make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]);
            }
        }
        __syncthreads();
    }
}

// FP8 transpose of any shape and alignment, in 128x128 tiles (one per CTA,
// or a looping first wave: see transpose_odd_loop_kernel).
//   * Staging: row r of the tile is the byte segment in + g * cols + col0 of
//     ncol bytes, starting e_r = its address % 16 into a 16-byte chunk.  The
//     nine aligned chunks that cover it are copied as they are (cp.async, 16
//     bytes each, no register round trip; nine consecutive lanes per row, so
//     the copies of a warp are coalesced) into a 144-byte row of shared
//     memory, together with the 16 rows of the tile above (the halo that the
//     transposed stores below need).
//   * Gather: warp b takes tile rows 16b .. 16b + 15, one row per load
//     instruction: lane l reads the two aligned words that cover columns
//     4l .. 4l + 3 of the row (at byte e_r + 4l) and byte-permutes them into
//     one word, so a load touches 32 consecutive words (no bank conflict) and
//     e_r is the same for the whole warp.  Since e_{r+1} = e_r + cols (mod
//     16), e_r depends on the row within the 16-row block only.  Byte
//     permutes transpose each 4x4 block; the column pieces go to a
//     column-major copy, each lane's four columns in a rotated order that
//     keeps the copy's stores free of bank conflicts.  Warps 0 .. 3 also
//     take 4 halo rows each (warp 0 taking all 16 left the other seven
//     waiting for it at the barrier).
//   * Stores: gen::store_col_copy_blocks, whole aligned 16-byte blocks.
constexpr int kOddStgRows = gen::kHaloRows + kTileRows;   // 144 staged rows
constexpr int kOddStgPitch = 144;                         // 9 chunks of 16 bytes

// Copies of tile t's 144 staged rows into stg (cp.async, not waited for).
__device__ __forceinline__ void odd_stage_tile(const uint8_t* __restrict__ in, int64_t rows,
                                               int64_t cols, uint32_t t, uint32_t tiles_c,
                                               uint8_t* stg, int tid) {
    const uint32_t rt32 = t / tiles_c;
    const int64_t rt = rt32;
    const int64_t row0 = rt * kTileRows;
    const int64_t col0 = int64_t(t - rt32 * tiles_c) * kTileCols;
    const int ncol = static_cast<int>(cols - col0 < kTileCols ? cols - col0 : kTileCols);
    const uintptr_t ibeg = reinterpret_cast<uintptr_t>(in);
    const uintptr_t iend = ibeg + uintptr_t(rows) * uintptr_t(cols);

    // Staged row wr holds global row row0 - 16 + wr (rows before row 0 and
    // from `rows` on are not loaded); chunk k of it at byte 16k.  Thread
    // i < 252 copies chunk i % 9 of rows i / 9, i / 9 + 28, ...
    if (tid < 252) {
        const int k = tid % 9;
        const int wr_lo = rt > 0 ? 0 : gen::kHaloRows;
        const int64_t wr_hi64 = rows - row0 + gen::kHaloRows;
        const int wr_hi = wr_hi64 < kOddStgRows ? static_cast<int>(wr_hi64) : kOddStgRows;
        int wr = tid / 9;
        uintptr_t a = ibeg + uintptr_t(row0 - gen::kHaloRows + wr) * uintptr_t(cols) + uintptr_t(col0);
        const uintptr_t step = uintptr_t(28) * uintptr_t(cols);
        // Unless the tile holds the first or the last 16-byte block of `in`,
        // every chunk it copies lies within `in`: no per-chunk end checks.
        const uintptr_t first =
            ibeg + uintptr_t(row0 - gen::kHaloRows + wr_lo) * uintptr_t(cols) + uintptr_t(col0);
        const uintptr_t last_end =
            ibeg + uintptr_t(row0 - gen::kHaloRows + wr_hi - 1) * uintptr_t(cols) + uintptr_t(col0) +
            uintptr_t(ncol);
        const bool inside = (first & ~uintptr_t(15)) >= ibeg && ((last_end + 15) & ~uintptr_t(15)) <= iend;
        if (inside && wr_lo == 0 && wr_hi == kOddStgRows && ncol == kTileCols) {
            // A whole tile with its halo: all 144 rows, 128 bytes each (of
            // chunk 8 only when the row does not start on a 16-byte boundary),
            // unrolled, without the row range checks.
#pragma unroll
            for (int i = 0; i < 6; ++i) {
                const int w = wr + 28 * i;
                if (i == 5 && w >= kOddStgRows) break;
                const uintptr_t ai = a + uintptr_t(i) * step;
                if (k == 8 && (ai & 15) == 0) continue;
                dev::cp_async16(stg + w * kOddStgPitch + 16 * k,
                                reinterpret_cast<const void*>((ai & ~uintptr_t(15)) + 16 * uintptr_t(k)),
                                16);
            }
            wr = kOddStgRows;
        }
        for (; wr < kOddStgRows; wr += 28, a += step) {
            if (wr < wr_lo || wr >= wr_hi) continue;
            const int e = static_cast<int>(a & 15);
            if (16 * k - e >= ncol) continue;   // the chunk starts past the row's segment
            const uintptr_t c0 = (a & ~uintptr_t(15)) + 16 * uintptr_t(k);
            uint8_t* dst = stg + wr * kOddStgPitch + 16 * k;
            if (inside) {
                dev::cp_async16(dst, reinterpret_cast<const void*>(c0), 16);
            } else if (c0 >= ibeg) {
                const uintptr_t n = iend - c0;   // > 0: the chunk holds a byte of the segment
                dev::cp_async16(dst, reinterpret_cast<const void*>(c0), n < 16 ? static_cast<int>(n) : 16);
            } else {   // the chunk that holds the first byte of `in`: only its bytes from there on
                for (int i = static_cast<int>(ibeg - c0); i < 16 && c0 + i < iend; ++i)
                    dst[i] = reinterpret_cast<const uint8_t*>(c0)[i];
            }
        }
    }
}

// Tile t: its staged rows (copied here unless `staged`), the gather into the
// column-major copy, and the whole-block stores.  `next` >= 0: the copies of
// tile `next` are issued into stg once the gather is done, so that they land
// while this tile's stores run.
__device__ __forceinline__ void odd_transpose_tile(const uint8_t* __restrict__ in, int64_t rows,
                                                   int64_t cols, uint8_t* __restrict__ out,
                                                   uint32_t t, uint32_t tiles_c, uint8_t* stg,
                                                   uint8_t* sqt, int tid, int lane, int warp,
                                                   bool demote = false, bool staged = false,
                                                   int64_t next = -1) {
    const uint32_t rt32 = t / tiles_c;
    const int64_t rt = rt32;
    const int64_t row0 = rt * kTileRows;
    const int64_t col0 = int64_t(t - rt32 * tiles_c) * kTileCols;
    const int ncol = static_cast<int>(cols - col0 < kTileCols ? cols - col0 : kTileCols);
    const uintptr_t ibeg = reinterpret_cast<uintptr_t>(in);

    if (!staged) odd_stage_tile(in, rows, cols, t, tiles_c, stg, tid);
    dev::cp_async_wait_all();
    __syncthreads();
    if (demote) {   // the tile's own q rows, now staged, back to the normal L2 priority
        const int64_t g = row0 + (tid >> 1);
        if (g < rows) {   // the one or two 128-byte lines of row g's segment
            const uintptr_t a = ibeg + uintptr_t(g) * uintptr_t(cols) + uintptr_t(col0);
            const uintptr_t line = (a & ~uintptr_t(127)) + 128 * uintptr_t(tid & 1);
            if (line < a + uintptr_t(ncol))
                asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(line) : "memory");
        }
    }

    // Row jj of every 16-row block starts e_jj = (E0 + jj * cols) % 16 bytes
    // into its staged row (16 * cols = 0 mod 16), the same for every block.
    // Lane l's four columns 4l .. 4l + 3 are taken rotated by rot = (l / 2) %
    // 4 (byte c of its row word is column 4l + (c + rot) % 4), so that its
    // k-th 16-byte column store goes to column 4l + (k + rot) % 4: the 8
    // lanes of a store phase then hit 8 different 16-byte bank groups (with a
    // 144-byte column pitch, columns 4l + k alone would share 2 of them).
    const int cm = static_cast<int>(cols & 15);
    const int E0 = static_cast<int>(
        (ibeg + uintptr_t(row0 - gen::kHaloRows) * uintptr_t(cols) + uintptr_t(col0)) & 15);
    const int rot = (lane >> 1) & 3;
    const uint32_t sel0 = 0x3210u + 0x1111u * rot - (rot > 0 ? 0x4000u : 0u) -
                          (rot > 1 ? 0x0400u : 0u) - (rot > 2 ? 0x0040u : 0u);
    auto block = [&](int wr0, int off) {   // staged rows wr0 .. wr0 + 15 -> column copy at `off`
        const uint8_t* base = stg + wr0 * kOddStgPitch + 4 * lane;
        uint32_t rw[16];
        int e = E0;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(base + jj * kOddStgPitch + (e & ~3));
            rw[jj] = __byte_perm(w[0], w[1], sel0 + 0x1111u * static_cast<uint32_t>(e & 3));
            e = (e + cm) & 15;
        }
        uint32_t o[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
            dev::transpose4x4(rw[4 * g], rw[4 * g + 1], rw[4 * g + 2], rw[4 * g + 3], o[0][g],
                              o[1][g], o[2][g], o[3][g]);
        uint8_t* col = sqt + 4 * lane * gen::kColCopyPitch + off;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq)
            *reinterpret_cast<uint4*>(col + ((kq + rot) & 3) * gen::kColCopyPitch) =
                make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]);
    };
    block(gen::kHaloRows + 16 * warp, gen::kHaloRows + 16 * warp);
    if (rt > 0 && warp < 4) {   // halo rows 4 warp .. 4 warp + 3: one 4x4 block per lane
        const uint8_t* base = stg + 4 * warp * kOddStgPitch + 4 * lane;
        uint32_t rw[4];
        int e = (E0 + 4 * warp * cm) & 15;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(base + jj * kOddStgPitch + (e & ~3));
            rw[jj] = __byte_perm(w[0], w[1], sel0 + 0x1111u * static_cast<uint32_t>(e & 3));
            e = (e + cm) & 15;
        }
        uint32_t c[4];
        dev::transpose4x4(rw[0], rw[1], rw[2], rw[3], c[0], c[1], c[2], c[3]);
        uint8_t* col = sqt + 4 * lane * gen::kColCopyPitch + 4 * warp;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq)
            *reinterpret_cast<uint32_t*>(col + ((kq + rot) & 3) * gen::kColCopyPitch) = c[kq];
    }
    __syncthreads();   // the gather is done with stg
    if (next >= 0) odd_stage_tile(in, rows, cols, static_cast<uint32_t>(next), tiles_c, stg, tid);
    gen::store_col_copy_blocks(out, rows, cols, rt, row0, col0, sqt, lane, warp);
}

// One tile per CTA: calls without a noop flag.
__global__ void __launch_bounds__(256) transpose_odd_kernel(const uint8_t* __restrict__ in,
                                                            int64_t rows, int64_t cols,
                                                            uint8_t* __restrict__ out,
                                                            const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ __align__(16) uint8_t stg[kOddStgRows * kOddStgPitch];
    __shared__ __align__(16) uint8_t sqt[kTileCols * gen::kColCopyPitch + 32];
    const int tid = threadIdx.x;
    const uint32_t tiles_c = static_cast<uint32_t>((cols + kTileCols - 1) / kTileCols);
    odd_transpose_tile(in, rows, cols, out, blockIdx.x, tiles_c, stg, sqt, tid, tid & 31, tid >> 5);
}

// Calls with a noop flag, and the transpose right after the flat cast: the
// first loop_ctas CTAs (one wave) take tiles b, b + loop_ctas, ...
// (loop_tiles each) and the CTAs after them one tile each of the rest, so a
// launch that its flag skips starts few CTAs.  `reverse` (after the flat
// cast) takes the tiles from the last one back, since the last rows of q are
// the ones still in L2, and returns the lines of q that the cast stored with
// the evict-last priority to the normal one once a tile has staged them.
__global__ void __launch_bounds__(256, 4) transpose_odd_loop_kernel(const uint8_t* __restrict__ in,
                                                                    int64_t rows, int64_t cols,
                                                                    uint8_t* __restrict__ out,
                                                                    const float* noop,
                                                                    int loop_ctas, int loop_tiles,
                                                                    int reverse) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ __align__(16) uint8_t stg[kOddStgRows * kOddStgPitch];
    __shared__ __align__(16) uint8_t sqt[kTileCols * gen::kColCopyPitch + 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tiles_c = static_cast<uint32_t>((cols + kTileCols - 1) / kTileCols);
    const uint32_t tiles = static_cast<uint32_t>((rows + kTileRows - 1) / kTileRows) * tiles_c;
    uint32_t first = blockIdx.x, stride = 0, count = 1;
    if (blockIdx.x < uint32_t(loop_ctas)) {
        stride = loop_ctas;
        count = loop_tiles;
    } else {
        first = uint32_t(loop_ctas) * uint32_t(loop_tiles) + (blockIdx.x - loop_ctas);
    }
    // A tile's gather ends at the barrier in front of its stores; the copies
    // of the CTA's next tile are issued there, into the staging rows the
    // gather has finished with, and land while the stores run.
    uint32_t t = first;
    if (count > 0 && t < tiles)
        odd_stage_tile(in, rows, cols, reverse ? tiles - 1 - t : t, tiles_c, stg, tid);
    for (uint32_t kt = 0; kt < count && t < tiles; ++kt, t += stride) {
        const uint32_t tn = t + stride;
        const int64_t next = kt + 1 < count && tn < tiles ? int64_t(reverse ? tiles - 1 - tn : tn) : -1;
        odd_transpose_tile(in, rows, cols, out, reverse ? tiles - 1 - t : t, tiles_c, stg, sqt, tid,
                           lane, warp, reverse != 0, /*staged=*/true, next);
    }
}


// ---------------------------------------------------------------------------
// Flat cast: q[i] = fp8(x[i] * scale) over the n = rows * cols elements as
// one array.  The cast of an element does not depend on where its row
// starts, so with x 16-byte and q 8-byte aligned every 8-element chunk is one
// 16-byte load and one 8-byte store for any row length.  A CTA takes
// kFlatChunks consecutive chunks (its threads' eight loads all in flight, as
// in the direct kernel), and grids of thousands of CTAs let the hardware
// balance the SMs.  The n % 8 elements after the last whole chunk are
// converted by one thread.  Amax and scale_inv as in the tile kernels.
constexpr int kFlatPerThread = 8;
constexpr int64_t kFlatChunks = 256 * kFlatPerThread;

// The 8-byte store of a flat-cast chunk; KEEP: with the L2 evict-last
// priority (the transpose that reads q next lowers it again).
template <bool KEEP>
__device__ __forceinline__ void store_q8(uint2* p, uint2 v) {
    if (KEEP) {
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
        asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x),
                     "r"(v.y), "l"(pol)
                     : "memory");
    } else {
        *p = v;
    }
}

template <int FMT, bool KEEP>
__global__ void __launch_bounds__(256) cast_flat_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                        uint8_t* __restrict__ q, const float* scale_p,
                                                        float* amax, float* scale_inv,
                                                        const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ unsigned s_amax[8];
    const float scale = *scale_p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t chunks = n >> 3;
    const int64_t c0 = int64_t(blockIdx.x) * kFlatChunks + tid;
    uint4 v[kFlatPerThread];
#pragma unroll
    for (int u = 0; u < kFlatPerThread; ++u) {
        const int64_t ch = c0 + 256 * u;
        v[u] = ch < chunks ? __ldcs(reinterpret_cast<const uint4*>(x) + ch) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t amax_pair = 0;
#pragma unroll
    for (int u = 0; u < kFlatPerThread; ++u) {
        const int64_t ch = c0 + 256 * u;
        amax_pair = dev::absmax_pair(amax_pair, v[u].x);
        amax_pair = dev::absmax_pair(amax_pair, v[u].y);
        amax_pair = dev::absmax_pair(amax_pair, v[u].z);
        amax_pair = dev::absmax_pair(amax_pair, v[u].w);
        if (ch < chunks) store_q8<KEEP>(reinterpret_cast<uint2*>(q) + ch, dev::cast8<FMT>(v[u], scale));
    }
    if (blockIdx.x == 0 && tid == 0) {
        const int64_t t0 = chunks << 3;
        if (t0 < n) {   // the last n % 8 elements
            uint32_t e[4] = {0u, 0u, 0u, 0u};
            for (int64_t i = t0; i < n; ++i)
                e[(i - t0) >> 1] |= uint32_t(x[i]) << (16 * ((i - t0) & 1));
            const uint4 t = make_uint4(e[0], e[1], e[2], e[3]);
            amax_pair = dev::absmax_pair(amax_pair, t.x);
            amax_pair = dev::absmax_pair(amax_pair, t.y);
            amax_pair = dev::absmax_pair(amax_pair, t.z);
            amax_pair = dev::absmax_pair(amax_pair, t.w);
            const uint2 c = dev::cast8<FMT>(t, scale);
            for (int64_t i = t0; i < n; ++i) {
                const int k = static_cast<int>(i - t0);
                q[i] = static_cast<uint8_t>((k < 4 ? c.x : c.y) >> (8 * (k & 3)));
            }
        }
        *scale_inv = __fdiv_rn(1.0f, scale);
    }
    const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
    if (lane == 0) s_amax[warp] = m;
    __syncthreads();
    if (tid == 0) {
        unsigned a = s_amax[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = a > s_amax[w] ? a : s_amax[w];
        if (a != 0) atomicMax(reinterpret_cast<unsigned*>(amax), a);
    }
}

// The flat cast of an x that starts m bytes past a 16-byte boundary (m = 2,
// 4, .., 14, the same for every element): output chunk c, x[8c .. 8c + 7],
// is bytes m .. m + 15 of the aligned chunks c and c + 1 of xa = x - m bytes.
// A warp loads 32 consecutive aligned chunks G .. G + 31 and writes the 31
// output chunks G .. G + 30, lane l taking chunk G + l + 1 from lane l + 1 by
// a shuffle (so every 32nd aligned chunk is loaded twice, and no lane waits
// on a load of its own after the first).  Group g of a CTA's 48 groups (8
// warps x kShiftPerThread) starts at G = 31 (48 blockIdx + 8 u + warp).
// Six loads in flight per thread keep it within 48 registers: 5 CTAs per
// SM (8191x12287 cast only, against eight loads at 4 CTAs per SM: 6.67
// against 6.58 TB/s).
// Aligned chunk `chunks` (n / 8), the one that can reach past the end of x,
// is put together from x's elements, so no byte outside x is read except the
// m bytes before x in aligned chunk 0 (inside x's allocation, whose start is
// 16-byte aligned).
constexpr int kShiftPerThread = 6;
constexpr int64_t kShiftGroups = 8 * kShiftPerThread;   // 31-chunk groups per CTA

__device__ __forceinline__ uint4 flat_tail_chunk(const uint16_t* __restrict__ x, int64_t n,
                                                 int64_t first) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = first + 2 * k;
        const uint32_t lo = i >= 0 && i < n ? x[i] : 0u;
        const uint32_t hi = i + 1 >= 0 && i + 1 < n ? x[i + 1] : 0u;
        w[k] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Bytes m .. m + 15 of the 32-byte window (a, b), m = 4 * WD + 2 * H.
template <int WD>
__device__ __forceinline__ uint4 window16(const uint4& a, const uint4& b, int sh) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    return make_uint4(__funnelshift_r(w[WD], w[WD + 1], sh), __funnelshift_r(w[WD + 1], w[WD + 2], sh),
                      __funnelshift_r(w[WD + 2], w[WD + 3], sh), __funnelshift_r(w[WD + 3], w[WD + 4], sh));
}

template <int FMT, bool KEEP, int WD>
__device__ __forceinline__ void flat_shift_body(const uint16_t* __restrict__ x, int64_t n,
                                                uint8_t* __restrict__ q, float scale, int m,
                                                uint32_t& amax_pair) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* xa = reinterpret_cast<const uint4*>(reinterpret_cast<uintptr_t>(x) - m);
    const int64_t chunks = n >> 3;
    const int64_t g0 = int64_t(blockIdx.x) * kShiftGroups + warp;
    const int sh = 8 * (m & 3);
    uint4 a[kShiftPerThread];
#pragma unroll
    for (int u = 0; u < kShiftPerThread; ++u) {
        const int64_t j = 31 * (g0 + 8 * u) + lane;   // aligned chunk of this lane
        a[u] = j < chunks ? __ldcs(xa + j)
                          : (j == chunks ? flat_tail_chunk(x, n, 8 * j - m / 2) : make_uint4(0u, 0u, 0u, 0u));
    }
#pragma unroll
    for (int u = 0; u < kShiftPerThread; ++u) {
        const int64_t ch = 31 * (g0 + 8 * u) + lane;   // output chunk of this lane (lanes 0 .. 30)
        uint4 b;
        b.x = __shfl_down_sync(0xFFFFFFFFu, a[u].x, 1);
        b.y = __shfl_down_sync(0xFFFFFFFFu, a[u].y, 1);
        b.z = __shfl_down_sync(0xFFFFFFFFu, a[u].z, 1);
        b.w = __shfl_down_sync(0xFFFFFFFFu, a[u].w, 1);
        if (lane < 31 && ch < chunks) {
            const uint4 v = window16<WD>(a[u], b, sh);
            amax_pair = dev::absmax_pair(amax_pair, v.x);
            amax_pair = dev::absmax_pair(amax_pair, v.y);
            amax_pair = dev::absmax_pair(amax_pair, v.z);
            amax_pair = dev::absmax_pair(amax_pair, v.w);
            store_q8<KEEP>(reinterpret_cast<uint2*>(q) + ch, dev::cast8<FMT>(v, scale));
        }
    }
}

template <int FMT, bool KEEP>
__global__ void __launch_bounds__(256, 5) cast_flat_shift_kernel(const uint16_t* __restrict__ x,
                                                              int64_t n, uint8_t* __restrict__ q,
                                                              const float* scale_p, float* amax,
                                                              float* scale_inv, const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ unsigned s_amax[8];
    const float scale = *scale_p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = static_cast<int>(reinterpret_cast<uintptr_t>(x) & 15);
    uint32_t amax_pair = 0;
    switch (m >> 2) {   // the same for the whole grid
        case 0: flat_shift_body<FMT, KEEP, 0>(x, n, q, scale, m, amax_pair); break;
        case 1: flat_shift_body<FMT, KEEP, 1>(x, n, q, scale, m, amax_pair); break;
        case 2: flat_shift_body<FMT, KEEP, 2>(x, n, q, scale, m, amax_pair); break;
        default: flat_shift_body<FMT, KEEP, 3>(x, n, q, scale, m, amax_pair); break;
    }
    if (blockIdx.x == 0 && tid == 0) {
        const int64_t t0 = (n >> 3) << 3;
        if (t0 < n) {   // the last n % 8 elements
            uint32_t e[4] = {0u, 0u, 0u, 0u};
            for (int64_t i = t0; i < n; ++i)
                e[(i - t0) >> 1] |= uint32_t(x[i]) << (16 * ((i - t0) & 1));
            const uint4 t = make_uint4(e[0], e[1], e[2], e[3]);
            amax_pair = dev::absmax_pair(amax_pair, t.x);
            amax_pair = dev::absmax_pair(amax_pair, t.y);
            amax_pair = dev::absmax_pair(amax_pair, t.z);
            amax_pair = dev::absmax_pair(amax_pair, t.w);
            const uint2 c = dev::cast8<FMT>(t, scale);
            for (int64_t i = t0; i < n; ++i) {
                const int k = static_cast<int>(i - t0);
                q[i] = static_cast<uint8_t>((k < 4 ? c.x : c.y) >> (8 * (k & 3)));
            }
        }
        *scale_inv = __fdiv_rn(1.0f, scale);
    }
    const unsigned mx = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
    if (lane == 0) s_amax[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        unsigned a = s_amax[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = a > s_amax[w] ? a : s_amax[w];
        if (a != 0) atomicMax(reinterpret_cast<unsigned*>(amax), a);
    }
}

// ---------------------------------------------------------------------------
// The conversion step alone: out[i] = fp8(in[i]) through dev::cvt_fp8x2, the
// routine every cast kernel applies to x * scale.  Grid-stride over pairs of
// values; a trailing odd value is converted with a zero partner whose code is
// not stored.
template <int FMT>
__global__ void __launch_bounds__(256) convert_f32_kernel(const float* __restrict__ in, int64_t n,
                                                          uint8_t* __restrict__ out) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    const int64_t pairs = (n + 1) / 2;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < pairs; k += stride) {
        const int64_t i = 2 * k;
        const bool two = i + 1 < n;
        const uint32_t c = dev::cvt_fp8x2<FMT>(in[i], two ? in[i + 1] : 0.0f);
        out[i] = static_cast<uint8_t>(c);
        if (two) out[i + 1] = static_cast<uint8_t>(c >> 8);
    }
}

unsigned grid_for(int64_t tiles, int64_t cap) {
    if (tiles < 1) tiles = 1;
    return static_cast<unsigned>(tiles < cap ? tiles : cap);
}

// The general kernel's dynamic shared memory is above the default 48 KB
// limit: raise it once per device and variant.
template <int FMT, bool DBIAS>
cudaError_t general_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(general_cast_kernel<FMT, DBIAS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DBIAS ? kGenSmemDbias : kGenSmem);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

template <int FMT, bool DBIAS>
cudaError_t launch_general_t(const GeneralArgs& a, dim3 grid, cudaStream_t stream) {
    const cudaError_t e = general_smem_attr<FMT, DBIAS>();
    if (e != cudaSuccess) return e;
    return launch_pdl(general_cast_kernel<FMT, DBIAS>, grid, dim3(256),
                      DBIAS ? kGenSmemDbias : kGenSmem, stream, a);
}

}  // namespace

cudaError_t launch_general(const GeneralArgs& a, int fmt, cudaStream_t stream) {
    const int64_t tiles =
        ((a.rows + kTileRows - 1) / kTileRows) * ((a.cols + kTileCols - 1) / kTileCols);
    const dim3 grid(grid_for(tiles, int64_t(1) << 30));
    const bool dbias = a.partial != nullptr;
    if (fmt == 0)
        return dbias ? launch_general_t<0, true>(a, grid, stream)
                     : launch_general_t<0, false>(a, grid, stream);
    return dbias ? launch_general_t<1, true>(a, grid, stream)
                 : launch_general_t<1, false>(a, grid, stream);
}

cudaError_t launch_dbias_finish(const float* partial, int64_t runs, int64_t cols, void* dbias,
                                bool db_bf16, const float* noop, cudaStream_t stream) {
    const dim3 grid(grid_for((cols + 31) / 32, 1 << 16)), block(256);
    if (db_bf16)
        return launch_pdl(dbias_finish_kernel<true>, grid, block, 0, stream, partial, runs, cols,
                          dbias, noop);
    return launch_pdl(dbias_finish_kernel<false>, grid, block, 0, stream, partial, runs, cols,
                      dbias, noop);
}

cudaError_t launch_scale_update(float* hist, float* scale, float* scale_inv, int hist_len,
                                int count, int64_t stride, int fmt, int margin, int most_recent,
                                const float* noop, cudaStream_t stream) {
    const float fp8_max = fmt == 0 ? 448.0f : 57344.0f;
    const float two_pow_margin = std::ldexp(1.0f, margin);   // exact for 0 <= margin <= 126
    if (hist_len <= 32 * dev::kUpdateRowsPerLane) {
        const dim3 grid(static_cast<unsigned>((int64_t(count) * 32 + 127) / 128)), block(128);
        return launch_pdl(scale_update_warp_kernel, grid, block, 0, stream, hist, scale, scale_inv,
                          hist_len, count, stride, fp8_max, two_pow_margin, most_recent, noop);
    }
    const dim3 grid(static_cast<unsigned>((count + 127) / 128)), block(128);
    return launch_pdl(scale_update_long_kernel, grid, block, 0, stream, hist, scale, scale_inv,
                      hist_len, count, stride, fp8_max, two_pow_margin, most_recent, noop);
}

cudaError_t launch_scale_update_pending(float* hist, float* pending, float* scale,
                                        float* scale_inv, int hist_len, int K, int count,
                                        int64_t stride, int fmt, int margin, int most_recent,
                                        const float* noop, cudaStream_t stream) {
    const float fp8_max = fmt == 0 ? 448.0f : 57344.0f;
    const float two_pow_margin = std::ldexp(1.0f, margin);   // exact for 0 <= margin <= 126
    const dim3 grid(static_cast<unsigned>((int64_t(count) * 32 + 127) / 128)), block(128);
    return launch_pdl(scale_update_pending_kernel, grid, block, 0, stream, hist, pending, scale,
                      scale_inv, hist_len, K, count, stride, fp8_max, two_pow_margin, most_recent,
                      noop);
}

cudaError_t launch_convert_f32(const float* in, int64_t n, int fmt, uint8_t* out,
                               cudaStream_t stream) {
    const dim3 grid(grid_for(((n + 1) / 2 + 255) / 256, 152 * 16)), block(256);
    return fmt == 0 ? launch_pdl(convert_f32_kernel<0>, grid, block, 0, stream, in, n, out)
                    : launch_pdl(convert_f32_kernel<1>, grid, block, 0, stream, in, n, out);
}

cudaError_t launch_cast_flat(const uint16_t* x, int64_t n, uint8_t* q, const float* scale,
                             float* amax, float* scale_inv, int fmt, const float* noop,
                             cudaStream_t stream, bool keep_q) {
    const int64_t chunks = n >> 3;
    const dim3 grid(grid_for((chunks + kFlatChunks - 1) / kFlatChunks, int64_t(1) << 30)), block(256);
    if (reinterpret_cast<uintptr_t>(x) & 15) {
        const int64_t groups = (chunks + 30) / 31;
        const dim3 sgrid(grid_for((groups + kShiftGroups - 1) / kShiftGroups, int64_t(1) << 30));
        auto k = fmt == 0 ? (keep_q ? cast_flat_shift_kernel<0, true> : cast_flat_shift_kernel<0, false>)
                          : (keep_q ? cast_flat_shift_kernel<1, true> : cast_flat_shift_kernel<1, false>);
        return launch_pdl(k, sgrid, block, 0, stream, x, n, q, scale, amax, scale_inv, noop);
    }
    auto k = fmt == 0 ? (keep_q ? cast_flat_kernel<0, true> : cast_flat_kernel<0, false>)
                      : (keep_q ? cast_flat_kernel<1, true> : cast_flat_kernel<1, false>);
    return launch_pdl(k, grid, block, 0, stream, x, n, q, scale, amax, scale_inv, noop);
}

constexpr int64_t kTransposeLoopPercent = 90;

// One wave of the fast transpose kernel: SMs x resident CTAs (cached per device).
int transpose_wave_ctas() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, transpose_fast_kernel, 256, 0) !=
            cudaSuccess)
            return 0;
        cache[dev] = sms * per_sm;
    }
    return cache[dev];
}

// One wave of the odd-shape transpose's looping kernel: SMs x resident CTAs
// (cached per device).
int odd_transpose_wave_ctas() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, transpose_odd_loop_kernel, 256, 0) !=
            cudaSuccess)
            return 0;
        cache[dev] = sms * per_sm;
    }
    return cache[dev];
}

bool odd_transpose_loops_after_cast(int64_t rows, int64_t cols) {
    const int64_t tiles = ((rows + 127) / 128) * ((cols + 127) / 128);
    const int wave = odd_transpose_wave_ctas();
    return wave > 0 && tiles >= wave;
}

cudaError_t launch_transpose(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out,
                             const float* noop, bool fast, cudaStream_t stream, bool after_cast) {
    if (fast) {
        const int64_t tiles = ((rows + 127) / 128) * ((cols + 127) / 128);
        // Without a noop flag, one tile per CTA: the hardware hands tiles to
        // whichever SM frees a slot (16384x12288: 6.76 TB/s, against 6.47 with
        // 4096 CTAs looping).  With one, a looping first wave over
        // kTransposeLoopPercent of the tiles and one tile per CTA for the
        // rest; measured at 16384x12288, flag 0 / flag 1 (skipped): 70%
        // 6.66 TB/s / 5.4 us, 80% 6.63 / 4.5, 90% 6.43 / 2.6; one tile per
        // CTA 6.64 / 12.7.  A cached transpose is skipped on most calls.
        int64_t loop_ctas = 0, loop_tiles = 0, grid = tiles;
        const int wave = transpose_wave_ctas();
        if (noop != nullptr && wave > 0) {
            loop_ctas = wave;
            loop_tiles = tiles * kTransposeLoopPercent / 100 / wave;
            if (loop_tiles < 1) loop_tiles = 1;
            const int64_t rest = tiles - loop_ctas * loop_tiles;
            grid = loop_ctas + (rest > 0 ? rest : 0);
        }
        return launch_pdl(transpose_fast_kernel, dim3(grid_for(grid, int64_t(1) << 30)), dim3(256),
                          0, stream, in, rows, cols, out, noop, loop_ctas, loop_tiles);
    }
    // at most 2^40 elements (the API's shape check): at most 2^26 tiles.
    // With a noop flag, the same looping first wave as above.  So too right
    // after the flat cast: there the one-tile kernel (48 registers, 5 CTAs
    // per SM) loses to the looping one (4 CTAs per SM), though alone it wins;
    // 8191x12287 measured: cast + transpose 4.15 against 4.51 TB/s,
    // transpose alone 42.1 against 44.7 us.  After the cast the looping
    // launch also takes the tiles in reverse order (4.51 -> 4.59 TB/s).
    const int64_t tiles = ((rows + 127) / 128) * ((cols + 127) / 128);
    if (tiles <= 0 || tiles > INT32_MAX) return cudaErrorInvalidValue;
    const int wave = noop != nullptr || after_cast ? odd_transpose_wave_ctas() : 0;
    if (wave > 0) {
        const int64_t loop_ctas = wave;
        int64_t loop_tiles = tiles * kTransposeLoopPercent / 100 / wave;
        if (loop_tiles < 1) loop_tiles = 1;
        const int64_t rest = tiles - loop_ctas * loop_tiles;
        const int64_t grid = loop_ctas + (rest > 0 ? rest : 0);
        return launch_pdl(transpose_odd_loop_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                          stream, in, rows, cols, out, noop, static_cast<int>(loop_ctas),
                          static_cast<int>(loop_tiles), after_cast ? 1 : 0);
    }
    return launch_pdl(transpose_odd_kernel, dim3(static_cast<unsigned>(tiles)), dim3(256), 0, stream,
                      in, rows, cols, out, noop);
}

}  // namespace ct
