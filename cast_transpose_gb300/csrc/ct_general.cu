// ct_general.cu -- kernels for the cases the TMA path does not take, and the
// small kernels around it (sm_103a):
//   * general_cast_kernel: cast (+ transpose, + dbias partials) of a bf16
//     matrix of ANY shape and alignment, 128x32 tiles, element-wise loads;
//   * dbias_finish_kernel: db[j] = sum over 128-row tiles of the partials,
//     compensated fp32, in a fixed order (deterministic);
//   * scale_update_kernel: the delayed-scaling update of "[PyTorch] Refactor
//     FP8 workspaces in linear modules" (Motivations: scale update kernel,
//     infinite-scale case), one thread per tensor;
//   * transpose kernels for FP8 bytes (the lazy transpose-cache fill of the
//     same page), a 128x128-tile vectorised one and a general one.
#include "ct_device.cuh"
#include "ct_internal.h"
#include "ct_update.cuh"

#include <cmath>

namespace ct {
namespace {

// ---------------------------------------------------------------------------
// General cast: tile = 128 rows x 32 columns, 256 threads; thread (c, g)
// handles column c and rows g + 8*i, i = 0..15.
constexpr int kGenCols = 32;

template <int FMT, bool DBIAS>
__global__ void __launch_bounds__(256) general_cast_kernel(GeneralArgs a) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (a.noop != nullptr && *a.noop != 0.0f) return;
    __shared__ uint8_t tileq[kTileRows][kGenCols + 4];
    __shared__ float colsum[8][kGenCols];
    __shared__ unsigned s_amax;

    const int64_t tiles_c = (a.cols + kGenCols - 1) / kGenCols;
    const int64_t tiles = ((a.rows + kTileRows - 1) / kTileRows) * tiles_c;
    const int tid = threadIdx.x;
    const int c = tid & 31;
    const int g = tid >> 5;
    const float scale = *a.scale;
    uint32_t amax = 0;
    if (tid == 0) s_amax = 0;
    __syncthreads();

    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t rt = tile / tiles_c;
        const int64_t row0 = rt * kTileRows;
        const int64_t col0 = (tile - rt * tiles_c) * kGenCols;
        const int64_t col = col0 + c;
        float cs = 0.0f;
        // all 16 loads of the thread first (memory-level parallelism), then
        // the conversions and stores
        uint16_t xv[16];
        const bool col_ok = col < a.cols;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t row = row0 + g + 8 * i;
            xv[i] = (col_ok && row < a.rows) ? __ldg(a.x + row * a.cols + col) : uint16_t(0);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = g + 8 * i;
            const int64_t row = row0 + r;
            uint8_t code = 0;
            if (col_ok && row < a.rows) {
                const uint32_t bits = xv[i];
                const uint32_t mag = (bits & 0x7FFFu) << 16;
                amax = mag > amax ? mag : amax;
                const float f = __uint_as_float(bits << 16);
                if (DBIAS) cs += f;
                code = static_cast<uint8_t>(dev::cvt_fp8x2<FMT>(__fmul_rn(f, scale), 0.0f));
                if (a.out) a.out[row * a.cols + col] = code;
            }
            tileq[r][c] = code;
        }
        if (DBIAS) colsum[g][c] = cs;
        __syncthreads();
        if (a.out_t) {
            // lanes run along rows of x, i.e. along a row of the transpose
            const int r = tid & (kTileRows - 1);
            const int64_t row = row0 + r;
            for (int cc = tid >> 7; cc < kGenCols; cc += 2) {
                const int64_t tc = col0 + cc;
                if (row < a.rows && tc < a.cols) a.out_t[tc * a.rows + row] = tileq[r][cc];
            }
        }
        if (DBIAS && tid < kGenCols && col < a.cols) {
            float s = colsum[0][tid];
            for (int j = 1; j < 8; ++j) s += colsum[j][tid];
            a.partial[rt * a.cols + col] = s;
        }
        if (tile == 0 && tid == 0) *a.scale_inv = __fdiv_rn(1.0f, scale);
        __syncthreads();
    }
    const unsigned m = __reduce_max_sync(0xFFFFFFFFu, amax);
    if ((tid & 31) == 0 && m != 0) atomicMax(&s_amax, m);
    __syncthreads();
    if (tid == 0 && s_amax != 0) atomicMax(reinterpret_cast<unsigned*>(a.amax), s_amax);
}

// ---------------------------------------------------------------------------
// db[j] = sum over the `runs` partial rows of partial[t, j] (one row per
// band of tile rows, see dbias_units).  Block = 32 columns x 8 row groups;
// each thread sums every 8th partial row of its column, then the 8 group
// sums are added in a fixed order (deterministic).  The sums are
// compensated (Kahan) fp32: the error stays within a few fp32 ulps of the sum
// of magnitudes for any number of row tiles, without fp64 arithmetic, which
// runs at a small fraction of the fp32 rate on this GPU.
struct Kahan {
    float sum = 0.0f, comp = 0.0f;
    __device__ __forceinline__ void add(float v) {
        const float y = __fsub_rn(v, comp);
        const float t = __fadd_rn(sum, y);
        comp = __fsub_rn(__fsub_rn(t, sum), y);
        sum = t;
    }
};

__global__ void __launch_bounds__(256) dbias_finish_kernel(const float* __restrict__ partial,
                                                           int64_t runs, int64_t cols,
                                                           float* __restrict__ db,
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
        if (j < cols) {
#pragma unroll 4
            for (int64_t t = g; t < runs; t += 8) k.add(partial[t * cols + j]);
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
            db[j] = total.sum;
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

// ---------------------------------------------------------------------------
// FP8 transpose, 128x128 byte tiles, 256 threads.  Loads are 16-byte row
// vectors; the tile is kept in shared memory with the same XOR swizzle as
// the cast kernel's FP8 copy (word w of row r at w ^ 4*(r/16)), so both the
// row-vector stores and the 16x4 column gathers are conflict-free.
__global__ void __launch_bounds__(256) transpose_fast_kernel(const uint8_t* __restrict__ in,
                                                             int64_t rows, int64_t cols,
                                                             uint8_t* __restrict__ out,
                                                             const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ __align__(16) uint32_t tile[kTileRows * (kTileCols / 4)];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t tiles_c = (cols + kTileCols - 1) / kTileCols;
    const int64_t tiles = ((rows + kTileRows - 1) / kTileRows) * tiles_c;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
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

// General byte transpose: 32x32 tiles, any shape and alignment.
__global__ void __launch_bounds__(256) transpose_general_kernel(const uint8_t* __restrict__ in,
                                                                int64_t rows, int64_t cols,
                                                                uint8_t* __restrict__ out,
                                                                const float* noop) {
    dev::pdl_launch_dependents();
    dev::pdl_wait();
    if (noop != nullptr && *noop != 0.0f) return;
    __shared__ uint8_t tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t tiles_c = (cols + 31) / 32;
    const int64_t tiles = ((rows + 31) / 32) * tiles_c;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t rt = t / tiles_c;
        const int64_t row0 = rt * 32, col0 = (t - rt * tiles_c) * 32;
        uint8_t v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = row0 + ty + 8 * i, col = col0 + tx;
            v[i] = (row < rows && col < cols) ? __ldg(in + row * cols + col) : uint8_t(0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) tile[ty + 8 * i][tx] = v[i];
        __syncthreads();
        for (int cc = ty; cc < 32; cc += 8) {
            const int64_t col = col0 + cc, row = row0 + tx;
            if (row < rows && col < cols) out[col * rows + row] = tile[tx][cc];
        }
        __syncthreads();
    }
}

unsigned grid_for(int64_t tiles, int64_t cap) {
    if (tiles < 1) tiles = 1;
    return static_cast<unsigned>(tiles < cap ? tiles : cap);
}

}  // namespace

cudaError_t launch_general(const GeneralArgs& a, int fmt, cudaStream_t stream) {
    const int64_t tiles =
        ((a.rows + kTileRows - 1) / kTileRows) * ((a.cols + kGenCols - 1) / kGenCols);
    const dim3 grid(grid_for(tiles, 1 << 20)), block(256);
    const bool dbias = a.partial != nullptr;
    if (fmt == 0)
        return dbias ? launch_pdl(general_cast_kernel<0, true>, grid, block, 0, stream, a)
                     : launch_pdl(general_cast_kernel<0, false>, grid, block, 0, stream, a);
    return dbias ? launch_pdl(general_cast_kernel<1, true>, grid, block, 0, stream, a)
                 : launch_pdl(general_cast_kernel<1, false>, grid, block, 0, stream, a);
}

cudaError_t launch_dbias_finish(const float* partial, int64_t runs, int64_t cols, float* dbias,
                                const float* noop, cudaStream_t stream) {
    const dim3 grid(grid_for((cols + 31) / 32, 1 << 16)), block(256);
    return launch_pdl(dbias_finish_kernel, grid, block, 0, stream, partial, runs, cols, dbias, noop);
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

cudaError_t launch_transpose(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out,
                             const float* noop, bool fast, cudaStream_t stream) {
    if (fast) {
        const int64_t tiles = ((rows + 127) / 128) * ((cols + 127) / 128);
        return launch_pdl(transpose_fast_kernel, dim3(grid_for(tiles, 4096)), dim3(256), 0, stream,
                          in, rows, cols, out, noop);
    }
    const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
    return launch_pdl(transpose_general_kernel, dim3(grid_for(tiles, 1 << 20)), dim3(256), 0,
                      stream, in, rows, cols, out, noop);
}

}  // namespace ct
