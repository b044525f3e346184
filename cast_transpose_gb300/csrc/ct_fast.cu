// ct_fast.cu -- TMA-staged persistent cast-transpose kernel (sm_103a).
//
// Operation ("[PyTorch] cuda graph support", DbiasCastTranspose example;
// "[PyTorch] Refactor FP8 workspaces in linear modules", Motivations): for a
// bf16 matrix x and an fp32 scale, write q = fp8(x * scale) row-major, its
// transpose qT, max-merge max|x| into *amax, write the tensor's own
// scale_inv = 1 / scale, and (dbias variant) the fp32 column sums of x.
//
// Design (HBM-bound stream, 4 bytes of traffic per element, no contraction):
//   * persistent CTAs, one per SM, walk 128x128 tiles round-robin; tile t of
//     CTA b is b + k * gridDim.x, so concurrently running CTAs touch
//     neighbouring tiles and whole rows of x stream through DRAM pages;
//   * one thread issues 2-D TMA loads of 32 KB bf16 tiles into a ring of
//     STAGES shared-memory buffers, each guarded by an mbarrier; the loads
//     carry an L2 evict-first hint since x is read once;
//   * pass 1 (all 256 threads): each thread reads 16-byte row vectors of the
//     staged tile (8 threads cover 128 contiguous bytes: no bank conflict),
//     converts 8 bf16 to 8 FP8 codes (fp32 multiply, cvt.rn.satfinite),
//     stores them straight to q (16 threads write one full 128-byte line) and
//     into an XOR-swizzled FP8 copy of the tile in shared memory; it also
//     keeps the running amax and, for dbias, per-column fp32 sums;
//   * one CTA barrier per tile; after it the stage is refilled by TMA;
//   * pass 2: each thread gathers a 16-row x 4-column byte block from the
//     swizzled copy (conflict-free), transposes it with byte permutes and
//     writes four 16-byte vectors of qT (8 threads write one 128-byte line);
//   * the FP8 copy and the column-sum scratch are double-buffered, so pass 2
//     of tile k overlaps pass 1 of tile k+1 without a second barrier;
//   * amax: per-thread SIMD max of bf16 magnitudes, warp reduction, one
//     shared atomic per warp and ONE global atomicMax per CTA per tensor;
//   * every mbarrier wait is bounded (about 2 s), after which the CTA sets a
//     diagnostic bit, waits (bounded) for its own TMA loads and returns.
#include "ct_device.cuh"
#include "ct_internal.h"

#include <mutex>

namespace ct {

__device__ unsigned int g_device_error;

namespace {

constexpr int kStageBytes = kTileRows * kTileCols * 2;   // bf16 tile
constexpr int kSqBytes = kTileRows * kTileCols;          // FP8 copy
constexpr int kColsumFloats = 8 * kTileCols;              // [warp][col]

template <int STAGES, bool WRITE_T, bool DBIAS>
struct SmemLayout {
    static constexpr int stage_off = 0;
    static constexpr int sq_off = STAGES * kStageBytes;
    static constexpr int colsum_off = sq_off + (WRITE_T ? 2 * kSqBytes : 0);
    static constexpr int mbar_off = colsum_off + (DBIAS ? 2 * kColsumFloats * 4 : 0);
    static constexpr int amax_off = mbar_off + STAGES * 8;
    static constexpr int abort_off = amax_off + 8;
    static constexpr int bytes = abort_off + 8 + 128;   // +128: base alignment slack
};

template <int NT, int FMT, int STAGES, bool WRITE_T, bool DBIAS>
__global__ void __launch_bounds__(kThreads, 1)
    fast_cast_transpose_kernel(const __grid_constant__ FastParams<NT> p) {
    using L = SmemLayout<STAGES, WRITE_T, DBIAS>;
    if (p.noop != nullptr && *p.noop != 0.0f) return;

    const int64_t first = blockIdx.x;
    const int64_t G = gridDim.x;
    if (first >= p.total_tiles) return;
    const int64_t my_tiles = (p.total_tiles - first + G - 1) / G;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t* stages = smem + L::stage_off;
    uint8_t* sq = smem + L::sq_off;
    float* colsum = reinterpret_cast<float*>(smem + L::colsum_off);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::mbar_off);
    unsigned* s_amax = reinterpret_cast<unsigned*>(smem + L::amax_off);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::abort_off);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // ---- producer state (thread 0 only) ------------------------------------
    int icur = 0;            // tensor of the next tile to load
    int64_t issued = 0;      // tiles of this CTA whose load has been issued
    uint64_t policy = 0;

    auto issue = [&](int64_t kk) {
        const int64_t tile = first + kk * G;
        while (tile >= p.t[icur].tile_end) ++icur;
        const FastTensor& T = p.t[icur];
        const int64_t local = tile - T.tile_begin;
        const int64_t rt = local / T.tile_cols;
        const int64_t ctl = local - rt * T.tile_cols;
        const int s = static_cast<int>(kk % STAGES);
        dev::mbar_arrive_expect_tx(&mbar[s], kStageBytes);
        dev::tma_load_2d(stages + s * kStageBytes, &p.map[icur],
                         static_cast<int32_t>(ctl * kTileCols),
                         static_cast<int32_t>(rt * kTileRows), &mbar[s], policy);
    };

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) dev::mbar_init(&mbar[s], 1);
        s_amax[0] = 0;
        s_amax[1] = 0;
        *s_abort = 0;
        dev::fence_barrier_init();
        policy = dev::policy_evict_first();
        for (; issued < my_tiles && issued < STAGES; ++issued) issue(issued);
    }
    __syncthreads();

    // ---- consumer state ----------------------------------------------------
    int cur = 0;                // tensor of the current tile
    uint32_t amax_pair = 0;     // running bf16 magnitude max (pair form)

    // pass-1 mapping: column chunk c (8 columns), rows rg + 16*it
    const int c = tid & 15;
    const int rg = tid >> 4;
    // pass-2 mapping: 16-row block b, 4-column word w
    const int b = lane & 7;
    const int w = warp * 4 + (lane >> 3);

    for (int64_t k = 0; k < my_tiles; ++k) {
        const int64_t tile = first + k * G;
        while (tile >= p.t[cur].tile_end) ++cur;
        const FastTensor& T = p.t[cur];
        const int64_t rows = T.rows, cols = T.cols;
        const int64_t local = tile - T.tile_begin;
        const int64_t rt = local / T.tile_cols;
        const int64_t row0 = rt * kTileRows;
        const int64_t col0 = (local - rt * T.tile_cols) * kTileCols;
        const float scale = *T.scale;
        const int s = static_cast<int>(k % STAGES);
        const uint32_t parity = static_cast<uint32_t>((k / STAGES) & 1);
        const int sb = static_cast<int>(k & 1);
        uint8_t* sqb = sq + sb * kSqBytes;

        float cs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) cs[j] = 0.0f;

        if (!dev::mbar_wait_bounded(&mbar[s], parity)) {
            *s_abort = 1;
        } else {
            // ---------------- pass 1 ----------------
            const uint8_t* in = stages + s * kStageBytes;
            uint4 v[8];
#pragma unroll
            for (int it = 0; it < 8; ++it)
                v[it] = *reinterpret_cast<const uint4*>(in + (rg + 16 * it) * (kTileCols * 2) + c * 16);
            const bool col_ok = col0 + 8 * c < cols;
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
                const uint2 q8 = dev::cast8<FMT>(v[it], scale);
                if (col_ok && row0 + r < rows)
                    *reinterpret_cast<uint2*>(qrow + r * cols) = q8;
                if constexpr (WRITE_T) {
                    // word index 2c of row r, XOR-swizzled by 4 * (r / 16)
                    *reinterpret_cast<uint2*>(sqb + r * kTileCols + ((2 * c) ^ (4 * it)) * 4) = q8;
                }
            }
            if constexpr (DBIAS) {
#pragma unroll
                for (int j = 0; j < 8; ++j) cs[j] += __shfl_xor_sync(0xFFFFFFFFu, cs[j], 16);
                if (lane < 16) {
                    float4* dst = reinterpret_cast<float4*>(colsum + sb * kColsumFloats +
                                                            warp * kTileCols + 8 * c);
                    dst[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
                    dst[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
                }
            }
        }

        // End of this CTA's run over the current tensor: fold the amax.
        const bool last_of_run = (k + 1 == my_tiles) || (tile + G >= T.tile_end);
        if (last_of_run) {
            const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
            if (lane == 0 && m != 0) atomicMax(&s_amax[sb], m);
            amax_pair = 0;
        }

        __syncthreads();

        if (*s_abort) {
            if (tid == 0) {
                atomicOr(&g_device_error, kErrWaitTimeout);
                for (int64_t kk = k; kk < issued; ++kk)
                    (void)dev::mbar_wait_bounded(&mbar[kk % STAGES],
                                                 static_cast<uint32_t>((kk / STAGES) & 1));
            }
            return;
        }

        if (tid == 0) {
            if (issued < my_tiles) {   // refill the stage pass 1 just released
                issue(issued);
                ++issued;
            }
            if (last_of_run) {
                const unsigned m = s_amax[sb];
                s_amax[sb] = 0;
                if (m != 0) atomicMax(reinterpret_cast<unsigned*>(T.amax), m);
            }
            if (local == 0) *T.scale_inv = __fdiv_rn(1.0f, scale);
        }

        // ---------------- pass 2 ----------------
        if constexpr (WRITE_T) {
            const uint32_t* sq32 = reinterpret_cast<const uint32_t*>(sqb);
            uint32_t rw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) rw[j] = sq32[(16 * b + j) * (kTileCols / 4) + (w ^ (4 * b))];
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
                        *reinterpret_cast<uint4*>(T.out_t + col * rows + row) =
                            make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]);
                }
            }
        }
        if constexpr (DBIAS) {
            if (tid < kTileCols && col0 + tid < cols) {
                const float* src = colsum + sb * kColsumFloats + tid;
                float sum = src[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) sum += src[j * kTileCols];
                p.partial[rt * cols + col0 + tid] = sum;
            }
        }
    }
}

// ---- launch configuration ---------------------------------------------------
constexpr int kStages = 4;

struct LaunchCache {
    std::mutex mu;
    int sms[64] = {0};
    bool attr_done[64][16] = {};
};
LaunchCache g_cache;

template <typename Kernel>
cudaError_t prepare(Kernel kernel, int key, int smem_bytes, int* sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_cache.mu);
    if (g_cache.sms[dev] == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_cache.sms[dev] = sms;
    }
    if (!g_cache.attr_done[dev][key]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        g_cache.attr_done[dev][key] = true;
    }
    *sms_out = g_cache.sms[dev];
    return cudaSuccess;
}

template <int NT, int FMT, bool WRITE_T, bool DBIAS>
cudaError_t launch_variant(const FastParams<NT>& p, int key, cudaStream_t stream) {
    using L = SmemLayout<kStages, WRITE_T, DBIAS>;
    auto kernel = fast_cast_transpose_kernel<NT, FMT, kStages, WRITE_T, DBIAS>;
    int sms = 0;
    cudaError_t e = prepare(kernel, key, L::bytes, &sms);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.total_tiles < sms ? p.total_tiles : sms;
    kernel<<<static_cast<unsigned>(grid), kThreads, L::bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fast(const FastParams<1>& p, int fmt, bool dbias, int variant,
                        cudaStream_t stream) {
    if (variant == 1) {
        return fmt == 0 ? launch_variant<1, 0, false, false>(p, 0, stream)
                        : launch_variant<1, 1, false, false>(p, 1, stream);
    }
    if (dbias) {
        return fmt == 0 ? launch_variant<1, 0, true, true>(p, 2, stream)
                        : launch_variant<1, 1, true, true>(p, 3, stream);
    }
    return fmt == 0 ? launch_variant<1, 0, true, false>(p, 4, stream)
                    : launch_variant<1, 1, true, false>(p, 5, stream);
}

cudaError_t launch_fast_list(const FastParams<kMaxListPerLaunch>& p, int fmt,
                             cudaStream_t stream) {
    return fmt == 0 ? launch_variant<kMaxListPerLaunch, 0, true, false>(p, 6, stream)
                    : launch_variant<kMaxListPerLaunch, 1, true, false>(p, 7, stream);
}

cudaError_t read_device_error(unsigned* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

}  // namespace ct
