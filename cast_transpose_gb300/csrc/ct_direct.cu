// ct_direct.cu -- one tile per 256 threads, cast-transpose with direct vector loads (sm_103a).
//
// Operation ("[PyTorch] cuda graph support", DbiasCastTranspose example;
// "[PyTorch] Refactor FP8 workspaces in linear modules", Motivations): the
// same as the TMA kernel of ct_fast.cu -- q = fp8(x * scale), its transpose
// qT, max|x| max-merged into *amax, scale_inv = 1 / scale and (dbias) the
// fp32 column sums of x -- for launches large enough to fill the GPU many
// times over.
//
// Design: the 256 threads that own tile (rt, ct) issue all of its
// 128x128 bf16 tile as eight 16-byte loads per thread at once (16 threads
// cover one 256-byte row segment, 128 KB in flight per SM at 4 resident
// CTAs), then
//   * pass 1: converts each 8-element vector to 8 FP8 codes, stores them to q
//     (16 threads write one 128-byte line) and into the XOR-swizzled FP8 copy
//     of the tile in shared memory (dev::swz); keeps the amax as a SIMD max
//     of bf16 magnitudes and, for dbias, 8 column sums per thread;
//   * one barrier among the tile's 256 threads;
//   * pass 2: each thread gathers a 16-row x 4-column byte block of the copy,
//     transposes it with byte permutes and writes four 16-byte vectors of qT
//     (8 threads write one 128-byte line).
// No pipeline state crosses tiles, so the kernel has no waits; the latency of
// one tile's loads is hidden by the other resident tiles.  Grids cover the
// tile count (thousands of CTAs, many waves of 152 SMs x 4 tiles); the TMA
// kernel keeps the launches too small for that to pay.
//
// Calls that pass a noop flag take direct_loop_kernel instead: the same
// passes, but a first wave of CTAs that loops over most of the tiles, so a
// launch that its flag skips starts a few waves of CTAs instead of
// thousands.
#include "ct_device.cuh"
#include "ct_gen_io.cuh"
#include "ct_internal.h"

#include <climits>
#include <mutex>


namespace ct {
namespace {

// A tile is processed by 256 threads.  A CTA runs TPC tiles side by side:
// 256 * TPC threads in TPC independent groups, group g on tile
// blockIdx.x * TPC + g, each group with its own named barrier.  Registers
// (64 per thread) allow 1024 threads per SM, i.e. 4 tiles in flight per SM
// either way.  Cast + transpose runs 2 tiles per CTA: the same rate as 1
// (6.87-6.89 against 6.89-6.91 TB/s on 16384x12288, back to back) while a
// launch skipped by the noop flag starts half as many CTAs (6.8 against
// 12.7 us); 4 tiles per CTA lost 10% (1 CTA per SM).  Cast only (6.84
// against 6.96 TB/s) and dbias (75 against 64 us) keep 1 tile per CTA.
constexpr int kDirectThreads = 256;
constexpr int kDirectWarps = kDirectThreads / 32;

template <bool WRITE_T, bool DBIAS>
constexpr int tiles_per_cta() { return WRITE_T && !DBIAS ? 2 : 1; }

constexpr int64_t kLoopPercent = 80;
constexpr int64_t kRestWaves = 8;


// The tensor of a list launch that owns global tile `tile`: the last entry
// whose first tile is <= tile (entries are non-empty and in tile order).
template <int NT>
__device__ __forceinline__ int owner(const DirectParams<NT>& p, int64_t tile) {
    if constexpr (NT == 1) {
        return 0;
    } else {
        int lo = 0, hi = p.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.t[mid].tile_begin <= tile) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
}

template <int TPC>
__device__ __forceinline__ void tile_sync(int g) {
    if constexpr (TPC == 1) __syncthreads();
    else dev::group_sync(g);
}

using dev::colsum_index;
using dev::kColsumStride;

// Transposed stores when rows % 16 != 0.  The qT segment of column j of a
// tile (rows row0 .. row0 + 127) then starts a_j = (col * rows + row0) % 16
// bytes into a 16-byte block, a different offset for every column.  The
// tile instead owns the rows [row0 - a_j, row0 + 128 - a_j) of column j:
// eight whole aligned 16-byte blocks, the first of which holds the last a_j
// rows of the tile above (the halo: its last 16 rows are loaded, cast and
// transposed with the tile).  Pass 2 writes the transposed bytes into a
// column-major copy (kOddPitch bytes per column: 16 halo rows, then the
// tile's 128); a third pass reads each block back at its offset (five 4-byte
// loads, four funnel shifts) and stores it with one 16-byte store.  The first
// tile row owns [0, 128 - a_j) and the last [row0 - a_j, rows): their blocks
// at the column ends are stored masked.
constexpr int kHaloRows = gen::kHaloRows;
constexpr int kOddPitch = gen::kColCopyPitch;

// Word wd of halo row h (0 .. 15, copy row 128 + h) lives at wd ^ halo_swz(h):
// the 8 lanes that read one word from rows 2b, 2b + 1 (b = 0 .. 7) then hit 8
// distinct groups of 4 banks, and every 8-byte row store stays whole.
__device__ __forceinline__ int halo_swz(int h) { return 4 * ((h >> 1) & 7); }

// Passes 2 (end) and 3 of the odd-row path, per warp: warp W transposes
// the 4-column words 4W .. 4W + 3, i.e. columns 16W .. 16W + 15, and stores
// exactly those columns' blocks, so it synchronises with itself only.
// o: the thread's transposed pieces (rows 16b .. 16b + 15 of columns
// 4w .. 4w + 3); sq32: the row-major copy, halo rows at 128 .. 143; sqt: the
// column-major copy.
__device__ __forceinline__ void odd_transpose_stores(const FastTensor& T, int64_t rt, int64_t row0,
                                                     int64_t col0, const uint32_t* sq32,
                                                     const uint32_t (&o)[4][4], int b, int w,
                                                     int lane, int warp, uint8_t* sqt) {
    const int64_t rows = T.rows, cols = T.cols;
#pragma unroll
    for (int kq = 0; kq < 4; ++kq)
        *reinterpret_cast<uint4*>(sqt + (4 * w + kq) * kOddPitch + kHaloRows + 16 * b) =
            make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]);
    if (rt > 0) {   // halo rows 2b and 2b + 1 of word w: two bytes of each of its columns
        const int r0 = kTileRows + 2 * b, r1 = r0 + 1;
        const uint32_t h0 = sq32[r0 * (kTileCols / 4) + (w ^ halo_swz(2 * b))];
        const uint32_t h1 = sq32[r1 * (kTileCols / 4) + (w ^ halo_swz(2 * b + 1))];
#pragma unroll
        for (int kq = 0; kq < 4; ++kq)
            *reinterpret_cast<uint16_t*>(sqt + (4 * w + kq) * kOddPitch + 2 * b) =
                static_cast<uint16_t>(__byte_perm(h0, h1, kq | ((4 + kq) << 4)));
    }
    __syncwarp();

    gen::store_col_copy_blocks(T.out_t, rows, cols, rt, row0, col0, sqt, lane, warp);
}

// EARLY: the launch issues work before the wait for the preceding kernel
// (x_ready loads, or first-wave L2 prefetches); without it the kernel is
// compiled without that path.  ODD: rows % 16 != 0 (one tensor, one tile per
// CTA, with the transpose); otherwise rows % 16 == 0.
template <int NT, int FMT, bool WRITE_T, bool DBIAS, int TPC, bool EARLY, bool ODD>
__global__ void __launch_bounds__(kDirectThreads * TPC, 4 / TPC)
    direct_cast_transpose_kernel(const __grid_constant__ DirectParams<NT> p) {
    static_assert(!ODD || (NT == 1 && TPC == 1 && WRITE_T), "the odd-row path is single-tile");
    // The next kernel of the stream may be scheduled as soon as this grid's
    // last wave is resident; it waits for this grid on the device.
    dev::pdl_launch_dependents();
    // Work issued before the wait for the preceding kernel (see below) needs
    // the tile coordinates first; every other CTA waits, and reads the noop
    // flag, before spending anything on them.
    const bool early = EARLY && (p.x_ready || blockIdx.x < p.prefetch_ctas);
    if (!early) {
        dev::pdl_wait();
        if (p.noop != nullptr && *p.noop != 0.0f) return;
    }

    __shared__ __align__(16) uint8_t
        sq_all[TPC][WRITE_T ? (kTileRows + (ODD ? kHaloRows : 0)) * kTileCols : 16];
    __shared__ __align__(16) float colsum_all[TPC][DBIAS ? kDirectWarps * kColsumStride : 4];
    __shared__ unsigned s_amax_all[TPC][kDirectWarps];
    // ODD: the column-major copy, and room for the last column's fifth word
    __shared__ __align__(16) uint8_t sqt[ODD ? kTileCols * kOddPitch + 32 : 16];

    // Tile coordinates come from the launch parameters only, so they are
    // known before the dependency wait.
    const int g = TPC == 1 ? 0 : static_cast<int>(threadIdx.x / kDirectThreads);
    const int tid = threadIdx.x % kDirectThreads, lane = tid & 31, warp = tid >> 5;
    const int64_t tile = static_cast<int64_t>(blockIdx.x) * TPC + g;
    if (tile >= p.total_tiles) return;   // a whole group of the last CTA: no barrier involves it
    uint8_t* sq = sq_all[g];
    float* colsum = colsum_all[g];
    unsigned* s_amax = s_amax_all[g];
    const int ti = owner(p, tile);
    const FastTensor& T = p.t[ti];
    const int64_t rows = T.rows, cols = T.cols;
    const int64_t local = tile - T.tile_begin;
    const int64_t rt = local / T.tile_cols;
    const int64_t row0 = rt * kTileRows, col0 = (local - rt * T.tile_cols) * kTileCols;
    const int tfmt = T.fmt;
    float scale = 0.0f;
    if constexpr (!EARLY) scale = *T.scale;   // after the wait: the preceding kernel may write it

    // pass-1 mapping: column chunk c (8 columns), rows rg + 16 * it
    const int c = tid & 15, rg = tid >> 4;
    const bool col_ok = col0 + 8 * c < cols;   // cols % 8 == 0: the chunk is whole
    const uint16_t* xin = p.x[ti] + col0 + 8 * c;
    uint4 v[8];
    // Before the wait for the preceding kernel (EARLY launches only): with
    // the caller's promise that no running kernel writes x (x_ready), the
    // tile itself is loaded; otherwise the CTAs of the first wave -- the ones
    // that can be resident while the preceding kernel still runs -- only ask
    // for their tile rows, and those of the second wave's tiles, to be
    // prefetched into L2: a hint that cannot return stale data (every write
    // lands in L2).
    bool loaded = false;
    if constexpr (EARLY) {
        if (early) {
            if (p.x_ready) {
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int64_t row = row0 + rg + 16 * it;
                    v[it] = (col_ok && row < rows)
                                ? __ldcs(reinterpret_cast<const uint4*>(xin + row * cols))
                                : make_uint4(0u, 0u, 0u, 0u);
                }
                loaded = true;
                // and the first wave's CTAs ask for the second wave's tiles, as below
                if constexpr (NT == 1) {
                    if (blockIdx.x < p.prefetch_ctas && tid < kTileRows) {
                        const int64_t tp = tile + int64_t(p.prefetch_ctas) * TPC;
                        if (tp < p.total_tiles) {
                            const int64_t rtp = tp / T.tile_cols;
                            const int64_t rp = rtp * kTileRows + tid;
                            const int64_t cp = (tp - rtp * T.tile_cols) * kTileCols;
                            if (rp < rows) {
                                const int64_t ncp = cols - cp < kTileCols ? cols - cp : kTileCols;
                                dev::prefetch_l2_bulk(p.x[ti] + rp * cols + cp,
                                                      static_cast<uint32_t>(2 * ncp));
                            }
                        }
                    }
                }
            } else if constexpr (NT == 1) {
                // threads 0..127: row tid of this CTA's tile; threads 128..255:
                // row tid - 128 of the tile of the CTA one wave later (whose
                // own first loads then find its rows in L2)
                const int64_t tp = tile + (tid < kTileRows ? 0 : int64_t(p.prefetch_ctas) * TPC);
                if (tp < p.total_tiles) {
                    const int64_t rtp = tp / T.tile_cols;
                    const int64_t rp = rtp * kTileRows + (tid & (kTileRows - 1));
                    const int64_t cp = (tp - rtp * T.tile_cols) * kTileCols;
                    if (rp < rows) {
                        const int64_t ncp = cols - cp < kTileCols ? cols - cp : kTileCols;
                        dev::prefetch_l2_bulk(p.x[ti] + rp * cols + cp, static_cast<uint32_t>(2 * ncp));
                    }
                }
            }
            dev::pdl_wait();
            if (p.noop != nullptr && *p.noop != 0.0f) return;
        }
        scale = *T.scale;
    }
    if (!loaded) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int64_t row = row0 + rg + 16 * it;
            v[it] = (col_ok && row < rows) ? __ldcs(reinterpret_cast<const uint4*>(xin + row * cols))
                                           : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    uint4 vh = make_uint4(0u, 0u, 0u, 0u);   // ODD: row row0 - 16 + rg of the halo
    if constexpr (ODD) {
        if (rt > 0 && col_ok && (rows & 15) != 8) vh = __ldcs(reinterpret_cast<const uint4*>(xin + (row0 - kHaloRows + rg) * cols));
    }

    uint32_t amax_pair = 0;
    float cs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cs[j] = 0.0f;
    uint8_t* qrow = T.out + row0 * cols + col0 + 8 * c;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = rg + 16 * it;
        amax_pair = dev::absmax_pair(amax_pair, v[it].x);
        amax_pair = dev::absmax_pair(amax_pair, v[it].y);
        amax_pair = dev::absmax_pair(amax_pair, v[it].z);
        amax_pair = dev::absmax_pair(amax_pair, v[it].w);
        if constexpr (DBIAS) {
            cs[0] += dev::bf16_lo(v[it].x); cs[1] += dev::bf16_hi(v[it].x);
            cs[2] += dev::bf16_lo(v[it].y); cs[3] += dev::bf16_hi(v[it].y);
            cs[4] += dev::bf16_lo(v[it].z); cs[5] += dev::bf16_hi(v[it].z);
            cs[6] += dev::bf16_lo(v[it].w); cs[7] += dev::bf16_hi(v[it].w);
        }
        // FMT < 0: the tensor's own format (uniform over the CTA)
        const uint2 q8 = FMT >= 0  ? dev::cast8<FMT < 0 ? 0 : FMT>(v[it], scale)
                         : tfmt == 0 ? dev::cast8<0>(v[it], scale)
                                     : dev::cast8<1>(v[it], scale);
        if (col_ok && row0 + r < rows) __stcs(reinterpret_cast<uint2*>(qrow + r * cols), q8);
        if constexpr (WRITE_T)   // words 2c, 2c+1 of row r
            *reinterpret_cast<uint2*>(sq + r * kTileCols + ((2 * c) ^ dev::swz(r)) * 4) = q8;
    }
    if constexpr (ODD) {   // the halo rows go to rows 128 .. 143 of the copy
        const int r = kTileRows + rg;
        *reinterpret_cast<uint2*>(sq + r * kTileCols + ((2 * c) ^ halo_swz(rg)) * 4) =
            dev::cast8<FMT < 0 ? 0 : FMT>(vh, scale);
    }
    const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
    if (lane == 0) s_amax[warp] = m;
    if constexpr (DBIAS) {   // fold the warp's two row groups (lanes l, l + 16)
#pragma unroll
        for (int j = 0; j < 8; ++j) cs[j] += __shfl_xor_sync(0xFFFFFFFFu, cs[j], 16);
        if (lane < 16) dev::colsum_store(colsum, warp, c, cs);
    }
    tile_sync<TPC>(g);

    if (tid == 0) {
        unsigned a = s_amax[0];
#pragma unroll
        for (int w = 1; w < kDirectWarps; ++w) a = a > s_amax[w] ? a : s_amax[w];
        if (a != 0) atomicMax(reinterpret_cast<unsigned*>(T.amax), a);
        if (local == 0) *T.scale_inv = __fdiv_rn(1.0f, scale);
    }
    if constexpr (DBIAS) {   // one partial row per tile row, warps summed in order
        if (tid < kTileCols && col0 + tid < cols) {
            float sum = colsum[colsum_index(0, tid)];
#pragma unroll
            for (int w = 1; w < kDirectWarps; ++w) sum += colsum[colsum_index(w, tid)];
            p.partial[rt * cols + col0 + tid] = sum;
        }
    }

    if constexpr (WRITE_T) {
        // pass-2 mapping: rows 16 * b .. 16 * b + 15, 4-column word w
        const int b = lane & 7, w = warp * 4 + (lane >> 3);
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
        if constexpr (!ODD) {   // rows % 16 == 0: whole, 16-byte aligned blocks
            const int64_t row = row0 + 16 * b;
            if (row < rows) {
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const int64_t col = col0 + 4 * w + kq;
                    if (col < cols)
                        __stcs(reinterpret_cast<uint4*>(T.out_t + col * rows + row),
                               make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]));
                }
            }
        } else if ((rows & 15) == 8) {
            // every column's segment starts 0 or 8 bytes into a block: its
            // neighbouring-lane pieces and 8-byte edge stores cost less
            // than the halo (6.23 against 5.85 TB/s on 8200x12288)
            const int L = static_cast<int>(rows - row0 < kTileRows ? rows - row0 : kTileRows);
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const int64_t col = col0 + 4 * w + kq;
                gen::store_segment_x8(T.out_t + col * rows + row0, col < cols ? L : 0, o[kq], b);
            }
        } else {
            odd_transpose_stores(T, rt, row0, col0, sq32, o, b, w, lane, warp, sqt);
        }
    }
}

// Tile `tile` of a launch: the tensor that owns it, its first row and column,
// and its index within the tensor (0: the tile that writes scale_inv).
struct LoopPos {
    int ti, row0, col0, local;
};

template <int NT>
__device__ __forceinline__ LoopPos loop_pos(const DirectParams<NT>& p, int tile) {
    LoopPos r;
    r.ti = owner(p, tile);
    const FastTensor& T = p.t[r.ti];
    r.local = tile - static_cast<int>(T.tile_begin);
    const int tc = static_cast<int>(T.tile_cols);
    const int rt = r.local / tc;
    r.row0 = rt * kTileRows;
    r.col0 = (r.local - rt * tc) * kTileCols;
    return r;
}

// The eight 16-byte loads of one thread (rows rg + 16 * it of column chunk c)
// of the tile at `t`; rows % 16 == 0, rows and cols below 2^31.
template <int NT>
__device__ __forceinline__ void loop_load(const DirectParams<NT>& p, const LoopPos& t, int c, int rg,
                                          uint4 (&v)[8]) {
    const FastTensor& T = p.t[t.ti];
    const int rows = static_cast<int>(T.rows), cols = static_cast<int>(T.cols);
    const bool col_ok = t.col0 + 8 * c < cols;
    const int nr = (rows - t.row0) >> 4;   // 16-row blocks left in the tensor
    const uint16_t* src = p.x[t.ti] + static_cast<int64_t>(t.row0 + rg) * cols + t.col0 + 8 * c;
#pragma unroll
    for (int it = 0; it < 8; ++it)
        v[it] = (col_ok && it < nr)
                    ? __ldcs(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(16 * it) * cols))
                    : make_uint4(0u, 0u, 0u, 0u);
}

// Cast (+ transpose) for calls that pass a noop flag (rows % 16 == 0, one
// tensor or a list).  Every CTA of the direct kernel starts, waits, reads
// the flag and exits, so a skipped launch costs about one CTA turnover per
// CTA (6.8 us for the 6144 CTAs of 16384x12288).  Here the first wave of
// CTAs (loop_ctas: SMs x resident CTAs) loops: group gi of its G groups of
// 256 threads takes tiles gi + k * G for k < loop_tiles, loading tile k + 1
// into registers as soon as the current one no longer needs them (during
// its qT stores).  The CTAs after the first wave take rest_chunk
// consecutive tiles per group from the remainder; the hardware hands them to
// whichever SM frees a slot first, which evens out SMs that stream slower
// than others (measured per group on GB300: 5.0 to 6.4 us per tile, so a
// grid that only loops ends with its slowest SM, 140 against 117 us).
// Amax is merged per tile, as in the direct kernel.
template <int NT, int FMT, bool WRITE_T, int TPC>
__global__ void __launch_bounds__(kDirectThreads * TPC, 4 / TPC)
    direct_loop_kernel(const __grid_constant__ DirectParams<NT> p) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (p.noop != nullptr && *p.noop != 0.0f) return;

    __shared__ __align__(16) uint8_t sq_all[TPC][WRITE_T ? kTileRows * kTileCols : 16];
    __shared__ unsigned s_amax_all[TPC][kDirectWarps];
    const int g = TPC == 1 ? 0 : static_cast<int>(threadIdx.x / kDirectThreads);
    const int tid = threadIdx.x % kDirectThreads, lane = tid & 31, warp = tid >> 5;
    const int total = static_cast<int>(p.total_tiles);
    const int groups = p.loop_ctas * TPC;
    int tile, step, last;
    if (static_cast<int>(blockIdx.x) < p.loop_ctas) {
        tile = static_cast<int>(blockIdx.x) * TPC + g;
        step = groups;
        last = tile + (p.loop_tiles - 1) * step;
    } else {
        const int u = (static_cast<int>(blockIdx.x) - p.loop_ctas) * TPC + g;
        tile = groups * p.loop_tiles + u * p.rest_chunk;
        step = 1;
        last = tile + p.rest_chunk - 1;
    }
    if (last >= total) last = total - 1;
    if (tile >= total) return;   // a whole group: no barrier involves it
    uint8_t* sq = sq_all[g];
    unsigned* s_amax = s_amax_all[g];
    const int c = tid & 15, rg = tid >> 4;
    const int b = lane & 7, w = warp * 4 + (lane >> 3);   // pass-2 mapping

    LoopPos cur = loop_pos(p, tile);
    uint4 v[8];
    loop_load(p, cur, c, rg, v);
    for (;;) {
        const FastTensor& T = p.t[cur.ti];
        const int rows = static_cast<int>(T.rows), cols = static_cast<int>(T.cols);
        const float scale = *T.scale;
        const int tfmt = T.fmt;
        {
            uint32_t amax_pair = 0;
            const bool col_ok = cur.col0 + 8 * c < cols;
            const int nr = (rows - cur.row0) >> 4;
            uint8_t* qrow = T.out + static_cast<int64_t>(cur.row0 + rg) * cols + cur.col0 + 8 * c;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = rg + 16 * it;
                amax_pair = dev::absmax_pair(amax_pair, v[it].x);
                amax_pair = dev::absmax_pair(amax_pair, v[it].y);
                amax_pair = dev::absmax_pair(amax_pair, v[it].z);
                amax_pair = dev::absmax_pair(amax_pair, v[it].w);
                // FMT < 0: the tensor's own format (uniform over the group)
                const uint2 q8 = FMT >= 0  ? dev::cast8<FMT < 0 ? 0 : FMT>(v[it], scale)
                                 : tfmt == 0 ? dev::cast8<0>(v[it], scale)
                                             : dev::cast8<1>(v[it], scale);
                if (col_ok && it < nr)
                    __stcs(reinterpret_cast<uint2*>(qrow + static_cast<int64_t>(16 * it) * cols), q8);
                if constexpr (WRITE_T)
                    *reinterpret_cast<uint2*>(sq + r * kTileCols + ((2 * c) ^ dev::swz(r)) * 4) = q8;
            }
            const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
            if (lane == 0) s_amax[warp] = m;
        }
        const int next = tile + step;
        tile_sync<TPC>(g);
        if (tid == 0) {
            unsigned a = s_amax[0];
#pragma unroll
            for (int k = 1; k < kDirectWarps; ++k) a = a > s_amax[k] ? a : s_amax[k];
            if (a != 0) atomicMax(reinterpret_cast<unsigned*>(T.amax), a);
            if (cur.local == 0) *T.scale_inv = __fdiv_rn(1.0f, scale);
        }
        LoopPos nxt = cur;
        if constexpr (WRITE_T) {
            uint32_t o[4][4];
            {
                const uint32_t* sq32 = reinterpret_cast<const uint32_t*>(sq);
                uint32_t rw[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = 16 * b + j;
                    rw[j] = sq32[r * (kTileCols / 4) + (w ^ dev::swz(r))];
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dev::transpose4x4(rw[4 * k], rw[4 * k + 1], rw[4 * k + 2], rw[4 * k + 3],
                                      o[0][k], o[1][k], o[2][k], o[3][k]);
            }
            // qT columns 0-1 of the block, the next tile's loads, columns 2-3
            const bool row_ok = cur.row0 + 16 * b < rows;
            uint8_t* dst = T.out_t + static_cast<int64_t>(cur.col0 + 4 * w) * rows + cur.row0 + 16 * b;
#pragma unroll
            for (int kq = 0; kq < 2; ++kq)
                if (row_ok && cur.col0 + 4 * w + kq < cols)
                    __stcs(reinterpret_cast<uint4*>(dst + static_cast<int64_t>(kq) * rows),
                           make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]));
            if (next <= last) {
                nxt = loop_pos(p, next);
                loop_load(p, nxt, c, rg, v);
            }
#pragma unroll
            for (int kq = 2; kq < 4; ++kq)
                if (row_ok && cur.col0 + 4 * w + kq < cols)
                    __stcs(reinterpret_cast<uint4*>(dst + static_cast<int64_t>(kq) * rows),
                           make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]));
        } else {
            if (next <= last) {
                nxt = loop_pos(p, next);
                loop_load(p, nxt, c, rg, v);
            }
        }
        if (next > last) break;
        tile = next;
        cur = nxt;
        tile_sync<TPC>(g);   // the shared copy and the amax slots are rewritten next
    }
}

// SMs of the current device (cached per device).
int sm_count() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

template <int NT, int FMT, bool WRITE_T, bool DBIAS, int TPC, bool ODD = false>
cudaError_t launch_tpc(const DirectParams<NT>& p, cudaStream_t stream) {
    const int64_t grid = (p.total_tiles + TPC - 1) / TPC;
    // The first wave (SMs x resident CTAs) prefetches its tiles, and the
    // second wave's, into L2 before the dependency wait, on the
    // one-tile-per-CTA variants of calls that have no noop flag.  Measured on
    // GB300: dbias 8192x12288 65.1 -> 63.3 us with the first wave's tiles,
    // 62.6 -> 61.6 us adding the second's (a third and fourth: 62.5, 63.5 us);
    // cast only +1.7%, then +0.5%.  With two tiles per CTA the prefetch cost
    // 2.5-3%, and a call that its flag skips would still pay for the prefetch
    // (6.8 -> 12.4 us).
    const dim3 g(static_cast<unsigned>(grid)), b(kDirectThreads * TPC);
    if constexpr (NT == 1) {   // lists never work early
        DirectParams<1> q = p;
        q.prefetch_ctas = (TPC == 1 && p.noop == nullptr) ? sm_count() * 4 : 0;
        if (q.x_ready || q.prefetch_ctas > 0)
            return launch_pdl(direct_cast_transpose_kernel<1, FMT, WRITE_T, DBIAS, TPC, true, ODD>, g, b,
                              0, stream, q);
    }
    return launch_pdl(direct_cast_transpose_kernel<NT, FMT, WRITE_T, DBIAS, TPC, false, ODD>, g, b, 0,
                      stream, p);
}

// The looping kernel's index arithmetic is in 32 bits, and its loads take
// whole 16-row blocks.
template <int NT>
bool loop_fits(const DirectParams<NT>& p) {
    for (int i = 0; i < p.n; ++i) {
        const FastTensor& T = p.t[i];
        if (T.rows % 16 != 0 || T.rows >= INT_MAX || T.cols >= INT_MAX) return false;
    }
    return true;
}

template <int NT, int FMT, bool WRITE_T, bool DBIAS>
cudaError_t launch_one(const DirectParams<NT>& p, cudaStream_t stream) {
    if (p.total_tiles <= 0 || p.total_tiles > INT_MAX) return cudaErrorInvalidValue;
    constexpr int TPC = tiles_per_cta<WRITE_T, DBIAS>();
    // rows % 16 != 0 (single tensors only): 1 tile per CTA, measured faster
    // for the transposed stores at any alignment (4.85 against 4.08 TB/s on
    // 8191x12288)
    if constexpr (NT == 1)
        if (p.t[0].rows % 16 != 0) return launch_tpc<NT, FMT, WRITE_T, DBIAS, 1, WRITE_T>(p, stream);
    // Calls with a noop flag: the looping first wave covers kLoopPercent of
    // the tiles.  Measured for 16384x12288 cast + transpose on GB300, flag 0 /
    // flag 1: 60% 6.81 TB/s / 3.4 us, 70% 6.78 / 2.9, 80% 6.75 / 2.25, 90%
    // 6.60 / 1.6; the direct kernel 6.90 TB/s / 6.8 us.  The remainder goes in
    // chunks of rest_chunk tiles per group, sized so that it spans about
    // kRestWaves waves of groups (one tile per group at 16384x12288; a list
    // of 300 K tiles would otherwise start 30 K CTAs to skip).
    if constexpr (!DBIAS) {
        const int sms = sm_count();
        if (p.noop != nullptr && !p.x_ready && sms > 0 && p.total_tiles < INT_MAX / 2 &&
            loop_fits(p)) {
            DirectParams<NT> q = p;
            q.loop_ctas = sms * (4 / TPC);
            const int64_t groups = static_cast<int64_t>(q.loop_ctas) * TPC;
            int64_t lt = p.total_tiles * kLoopPercent / 100 / groups;
            if (lt < 1) lt = 1;
            q.loop_tiles = static_cast<int>(lt);
            const int64_t rest = p.total_tiles - groups * lt;
            int64_t chunk = rest / (kRestWaves * groups);
            if (chunk < 1) chunk = 1;
            q.rest_chunk = static_cast<int>(chunk);
            q.prefetch_ctas = 0;
            const int64_t units = rest > 0 ? (rest + chunk - 1) / chunk : 0;
            const int64_t grid = q.loop_ctas + (units + TPC - 1) / TPC;
            const dim3 g(static_cast<unsigned>(grid)), b(kDirectThreads * TPC);
            return launch_pdl(direct_loop_kernel<NT, FMT, WRITE_T, TPC>, g, b, 0, stream, q);
        }
    }
    return launch_tpc<NT, FMT, WRITE_T, DBIAS, TPC>(p, stream);
}

}  // namespace

cudaError_t launch_direct(const DirectParams<1>& p, int fmt, bool dbias, int variant,
                          cudaStream_t stream) {
    if (variant == 1)
        return fmt == 0 ? launch_one<1, 0, false, false>(p, stream)
                        : launch_one<1, 1, false, false>(p, stream);
    if (dbias)
        return fmt == 0 ? launch_one<1, 0, true, true>(p, stream)
                        : launch_one<1, 1, true, true>(p, stream);
    return fmt == 0 ? launch_one<1, 0, true, false>(p, stream)
                    : launch_one<1, 1, true, false>(p, stream);
}

cudaError_t launch_direct_list(const DirectParams<kMaxListPerLaunch>& p, int fmt,
                               cudaStream_t stream) {
    if (fmt < 0) return launch_one<kMaxListPerLaunch, -1, true, false>(p, stream);
    return fmt == 0 ? launch_one<kMaxListPerLaunch, 0, true, false>(p, stream)
                    : launch_one<kMaxListPerLaunch, 1, true, false>(p, stream);
}

}  // namespace ct
