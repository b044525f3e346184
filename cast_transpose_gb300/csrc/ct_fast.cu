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
//     CTA b is b + k * gridDim.x in an order of bands of 16 tile rows,
//     column-major inside a band, so the tiles in flight at one time form a
//     compact block of x, q and qT;
//   * the producer maps tile indices to coordinates and hands them to the
//     consumers in shared memory next to the staged tile, off their path;
//   * a dedicated producer warp (one elected lane) issues 2-D TMA loads of
//     32 KB bf16 tiles into a ring of STAGES shared-memory buffers: a "full"
//     mbarrier per stage completes on the TMA transaction bytes, an "empty"
//     mbarrier per stage completes when all consumer warps have read it; the
//     loads carry an L2 evict-first hint since x is read once, and the
//     outputs are written with streaming (evict-first) stores;
//   * pass 1 (all 256 threads): each thread reads 16-byte row vectors of the
//     staged tile (8 threads cover 128 contiguous bytes: no bank conflict),
//     converts 8 bf16 to 8 FP8 codes (fp32 multiply, cvt.rn.satfinite),
//     stores them straight to q (16 threads write one full 128-byte line) and
//     into an XOR-swizzled FP8 copy of the tile in shared memory; it also
//     keeps the running amax and, for dbias, per-column fp32 sums;
//   * one barrier per tile among the consumer warps only (named barrier 1);
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
#include "ct_update.cuh"

#include <mutex>

namespace ct {

__device__ unsigned int g_device_error;

namespace {

constexpr int kStageBytes = kTileRows * kTileCols * 2;   // bf16 tile
constexpr int kSqBytes = kTileRows * kTileCols;          // FP8 copy

// Consumer threads per CTA of the TMA kernel (512 was measured on GB300 and
// was slower; the mappings below are written for 256).
constexpr int kFastThreads = 256;
static_assert(kFastThreads == 256, "the pass-1 and pass-2 mappings assume 256 threads");
constexpr int kWarps = kFastThreads / 32;
constexpr int kColsumFloats = kWarps * kTileCols;         // [warp][col]

// Shared-memory layout of the FP8 copy of a tile: see dev::swz.
using dev::swz;

// Where a staged tile came from.  Written by the producer thread before it
// arms the stage's mbarrier, read by the consumers after the barrier phase
// completes (the arrive releases, the wait acquires), so only one thread
// ever maps tile indices to coordinates.
struct StageInfo {
    int32_t tensor;        // index into p.t / p.map
    int32_t last;          // 1: this CTA's last tile of that tensor
    int32_t rt;            // tile row
    int32_t ct;            // tile column
    int32_t seg_end;       // dbias: 1 = last tile of this CTA's run down the strip
    int32_t seg;           // dbias: partial-sum row of that run (see dbias_segment)
};

// Dbias tile schedule (dbias_units in ct_internal.h): CTA b takes units b,
// b+G, ... and within a unit walks down its band's tile rows, summing the
// columns over the band before writing one partial row.
struct DbiasSchedule {
    int64_t H, last_h, S, full_units;   // band height, last band height, strips, units of height H
    int64_t F;                          // this CTA's units of height H
    uint32_t tiles;                     // this CTA's tiles
};
__device__ __forceinline__ DbiasSchedule dbias_schedule(int64_t R, int64_t S, uint32_t b, uint32_t G) {
    const DbiasUnits du = dbias_units(R, R < kDbiasBand ? R : kDbiasBand);
    DbiasSchedule d;
    d.H = du.H;
    d.last_h = du.last_h;
    d.S = S;
    d.full_units = (du.bands - 1) * S;
    const int64_t U = du.bands * S;
    const int64_t M = b < U ? (U - b + G - 1) / G : 0;
    d.F = b < d.full_units ? (d.full_units - b + G - 1) / G : 0;
    d.tiles = static_cast<uint32_t>(d.F * d.H + (M - d.F) * d.last_h);
    return d;
}

template <int STAGES, bool WRITE_T, bool DBIAS>
struct SmemLayout {
    static constexpr int stage_off = 0;
    static constexpr int sq_off = STAGES * kStageBytes;
    static constexpr int colsum_off = sq_off + (WRITE_T ? 2 * kSqBytes : 0);
    static constexpr int full_off = colsum_off + (DBIAS ? 2 * kColsumFloats * 4 : 0);
    static constexpr int empty_off = full_off + STAGES * 8;
    static constexpr int info_off = empty_off + STAGES * 8;
    static constexpr int amax_off = info_off + STAGES * int(sizeof(StageInfo));
    static constexpr int abort_off = amax_off + 8;
    static constexpr int bytes = abort_off + 8 + 128;   // +128: base alignment slack
};

// Order of the tiles of one tensor: bands of kBand tile rows, column-major
// inside a band, so that the ~150 tiles in flight at once form a block about
// kBand tiles tall.  The transposed output then receives kBand x 128 bytes
// of every row it touches at the same time, not 128 scattered bytes.
// Measured on GB300 (4096x4096 step): bands of 16 beat 8 by 1%, and 2, 4,
// 32 and 64 were slower.
constexpr uint32_t kBand = 16;

__device__ __forceinline__ void tile_coords(uint32_t local, uint32_t tile_rows, uint32_t tile_cols,
                                            int32_t& rt, int32_t& ct) {
    const uint32_t band = local / (kBand * tile_cols);
    const uint32_t rem = tile_rows - band * kBand;
    const uint32_t h = rem < kBand ? rem : kBand;
    const uint32_t idx = local - band * kBand * tile_cols;
    const uint32_t c = idx / h;
    ct = static_cast<int32_t>(c);
    rt = static_cast<int32_t>(band * kBand + (idx - c * h));
}

// Block: kFastThreads consumer threads (warps 0 .. kWarps-1) plus one
// producer warp (warp kWarps) whose lane 0 drives the TMA pipeline.
constexpr int kBlockThreads = kFastThreads + 32;

// PEND: a single tensor whose scale comes from deferred updates (p.pend);
// the other instantiations are compiled without that code.
template <int NT, int FMT, int STAGES, int MINB, bool WRITE_T, bool DBIAS, bool PEND = false>
__global__ void __launch_bounds__(kBlockThreads, MINB)
    fast_cast_transpose_kernel(const __grid_constant__ FastParams<NT> p) {
    static_assert(!PEND || (NT == 1 && WRITE_T && !DBIAS), "deferred updates: cast-transpose");
    using L = SmemLayout<STAGES, WRITE_T, DBIAS>;
    // Rows of the staged tile loaded per batch in pass 1: all at once for the
    // most loads in flight, 4 when registers are tight.
    constexpr int kBatch = (DBIAS && MINB > 1) ? 4 : 8;
    // When the next kernel of the stream may be scheduled.  Without dbias it
    // is typically a one-warp scale update or the next cast, which either
    // fits beside this kernel or cannot start before its CTAs leave: let it be
    // scheduled right away, hiding its launch.  With dbias it is always the
    // column-sum finish kernel, hundreds of blocks that would sit next to this
    // kernel's for its whole run: schedule it from each CTA's last tile on.
    if constexpr (!DBIAS) dev::pdl_launch_dependents();

    const uint32_t first = blockIdx.x;
    const uint32_t G = gridDim.x;
    if (first >= p.total_tiles) return;
    // round-robin tiles (b, b+G, ...), or for dbias round-robin band units
    DbiasSchedule dsch{};
    if constexpr (DBIAS) dsch = dbias_schedule(p.t[0].tile_rows, p.t[0].tile_cols, first, G);
    const uint32_t my_tiles =
        DBIAS ? dsch.tiles : static_cast<uint32_t>((p.total_tiles - first + G - 1) / G);
    if (my_tiles == 0) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t* stages = smem + L::stage_off;
    uint8_t* sq = smem + L::sq_off;
    float* colsum = reinterpret_cast<float*>(smem + L::colsum_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::empty_off);
    StageInfo* info = reinterpret_cast<StageInfo*>(smem + L::info_off);
    unsigned* s_amax = reinterpret_cast<unsigned*>(smem + L::amax_off);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::abort_off);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            dev::mbar_init(&full[s], 1);           // producer's arrive + TMA bytes
            dev::mbar_init(&empty[s], kWarps);     // one arrive per consumer warp
        }
        s_amax[0] = 0;
        s_amax[1] = 0;
        *s_abort = 0;
        dev::fence_barrier_init();
    }
    __syncthreads();

    // =============================== producer ================================
    if (warp == kWarps) {
        if (lane != 0) return;
        // L2 policy of the tile loads: x is read once, so with the transpose
        // (2 output streams) it is marked evict-first to leave L2 to the
        // writes; the cast alone measured faster with the normal policy.
        const uint64_t policy = WRITE_T ? dev::policy_evict_first() : dev::policy_evict_normal();
        int icur = 0;
        uint32_t issued = 0;
        // Where tile kk of this CTA comes from; `ic` is the list entry of the
        // previous call's tile (tiles only move forward through the list).
        auto locate = [&](uint32_t kk, int& ic, StageInfo& inf) {
            if constexpr (DBIAS) {
                int64_t m, off, h;
                if (int64_t(kk) < dsch.F * dsch.H) {
                    m = kk / dsch.H;
                    off = kk - m * dsch.H;
                    h = dsch.H;
                } else {
                    const int64_t k2 = kk - dsch.F * dsch.H;
                    m = dsch.F + k2 / dsch.last_h;
                    off = k2 - (m - dsch.F) * dsch.last_h;
                    h = dsch.last_h;
                }
                const int64_t u = int64_t(first) + m * G;
                const int64_t band = u / dsch.S;
                inf.tensor = 0;
                inf.last = kk + 1 == my_tiles;
                inf.ct = static_cast<int32_t>(u - band * dsch.S);
                inf.rt = static_cast<int32_t>(band * dsch.H + off);
                inf.seg_end = off + 1 == h;
                inf.seg = static_cast<int32_t>(band);
            } else {
                const int64_t tile = int64_t(first) + int64_t(kk) * G;
                while (tile >= p.t[ic].tile_end) ++ic;
                const FastTensor& T = p.t[ic];
                inf.tensor = ic;
                inf.last = (kk + 1 == my_tiles) || (tile + G >= T.tile_end);
                tile_coords(static_cast<uint32_t>(tile - T.tile_begin),
                            static_cast<uint32_t>(T.tile_rows), static_cast<uint32_t>(T.tile_cols),
                            inf.rt, inf.ct);
                inf.seg_end = 0;
                inf.seg = 0;
            }
        };
        auto issue = [&](uint32_t kk) {
            const int s = static_cast<int>(kk % STAGES);
            StageInfo inf;
            locate(kk, icur, inf);
            info[s] = inf;
            dev::mbar_arrive_expect_tx(&full[s], kStageBytes);
            dev::tma_load_2d(stages + s * kStageBytes, &p.map[icur], inf.ct * kTileCols,
                             inf.rt * kTileRows, &full[s], policy);
        };
        // The preceding kernel in the stream may still run until the
        // dependency wait returns, and it may be the one writing x: by default
        // all of this CTA's tiles are only prefetched into L2 before the wait
        // (a hint, which cannot leave stale data behind; launches here have
        // under 2048 tiles, at most 64 MB) and loaded after it.  Measured on
        // the 4096x4096 weight step: 114.7 -> 111.0 us per step against only
        // the first STAGES tiles.  When the caller promises that no running
        // kernel writes x (x_ready), the first STAGES tiles are loaded before
        // the wait, overlapping the preceding kernel (prefetching the others
        // as well cost 95.2 -> 99.8 us there).
        if (p.x_ready) {
            for (; issued < my_tiles && issued < STAGES; ++issued) issue(issued);
        } else {
            int ic = 0;
            for (uint32_t kk = 0; kk < my_tiles; ++kk) {
                StageInfo inf;
                locate(kk, ic, inf);
                dev::tma_prefetch_l2_2d(&p.map[ic], inf.ct * kTileCols, inf.rt * kTileRows);
            }
        }
        dev::pdl_wait();
        bool stop = p.noop != nullptr && *p.noop != 0.0f;
        for (; !stop && issued < my_tiles && issued < STAGES; ++issued) issue(issued);
        for (; !stop && issued < my_tiles; ++issued) {
            const uint32_t kk = issued;
            if (!dev::mbar_wait_bounded(&empty[kk % STAGES], ((kk / STAGES) - 1) & 1u, s_abort)) {
                // The consumers stopped (or never released a stage): flag it.
                *s_abort = 1;
                atomicOr(&g_device_error, kErrWaitTimeout);
                break;
            }
            issue(kk);
        }
        // Stay until the loads still in flight into this CTA's shared memory
        // have landed (bounded), whether or not the consumers still want them.
        const uint32_t lo = issued > STAGES ? issued - STAGES : 0;
        for (uint32_t kk = lo; kk < issued; ++kk)
            (void)dev::mbar_wait_bounded(&full[kk % STAGES], (kk / STAGES) & 1u);
        return;
    }

    // Consumers read data the preceding kernel may have written (the noop
    // flag, the scale, the amax slot): wait for it to complete first.
    dev::pdl_wait();
    if (p.noop != nullptr && *p.noop != 0.0f) return;
    // single tensors with deferred updates: the scale, derived once per warp
    // here, where every consumer warp is whole
    float pend_scale = 0.0f;
    if constexpr (PEND) pend_scale = dev::pending_scale_warp(p.pend, lane);

    // =============================== consumers ===============================
    int cur = -1;               // tensor of the current run, and its fields:
    float scale = 0.0f;         // loaded once per run, not once per tile
    int64_t rows = 0, cols = 0;
    uint8_t* out = nullptr;
    uint8_t* out_t = nullptr;
    int tfmt = 0;               // per-tensor format (list launches with FMT < 0)
    uint32_t amax_pair = 0;     // running bf16 magnitude max (pair form)
    float cs[8];                // dbias: column sums of this thread's 8 columns over
#pragma unroll                  // the current run down a strip
    for (int j = 0; j < 8; ++j) cs[j] = 0.0f;

    // pass-1 mapping: column chunk c (8 columns), rows rg + kRowStep*it
    constexpr int kRowStep = kFastThreads / 16;           // 16
    constexpr int kRowsPerThread = kTileRows / kRowStep;  // 8
    const int c = tid & 15;
    const int rg = tid >> 4;
    // pass-2 mapping: block b of kBlockRows rows, 4-column word w
    constexpr int kBlockRows = 16;
    constexpr int kBlocks = kTileRows / kBlockRows;       // 8
    const int b = lane % kBlocks;
    const int w = warp * (32 / kBlocks) + lane / kBlocks;

    for (uint32_t k = 0; k < my_tiles; ++k) {
        if (DBIAS && k + 1 == my_tiles) dev::pdl_launch_dependents();
        const int s = static_cast<int>(k % STAGES);
        const int sb = static_cast<int>(k & 1u);
        uint8_t* sqb = sq + sb * kSqBytes;
        int64_t row0 = 0, col0 = 0;
        int32_t seg = 0;
        bool last = false, first_tile = false, seg_end = false;

        if (!dev::mbar_wait_bounded(&full[s], (k / STAGES) & 1u, s_abort)) {
            *s_abort = 1;
        } else {
            const StageInfo inf = info[s];
            if (inf.tensor != cur) {
                cur = inf.tensor;
                scale = PEND ? pend_scale : *p.t[cur].scale;
                rows = p.t[cur].rows;
                cols = p.t[cur].cols;
                out = p.t[cur].out;
                out_t = p.t[cur].out_t;
                tfmt = p.t[cur].fmt;
            }
            seg = inf.seg;
            seg_end = inf.seg_end != 0;
            row0 = int64_t(inf.rt) * kTileRows;
            col0 = int64_t(inf.ct) * kTileCols;
            last = inf.last != 0;
            first_tile = inf.rt == 0 && inf.ct == 0;

            // ---------------- pass 1 ----------------
            const uint8_t* in = stages + s * kStageBytes;
            const bool col_ok = col0 + 8 * c < cols;
            uint8_t* qrow = out + row0 * cols + col0 + 8 * c;
#pragma unroll
            for (int it0 = 0; it0 < kRowsPerThread; it0 += kBatch) {
                uint4 v[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j)
                    v[j] = *reinterpret_cast<const uint4*>(
                        in + (rg + kRowStep * (it0 + j)) * (kTileCols * 2) + c * 16);
                if (it0 + kBatch == kRowsPerThread) {
                    // every read of this stage has been issued and its value is
                    // in a register: hand the stage back to the producer
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&empty[s]);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int it = it0 + j;
                    const int r = rg + kRowStep * it;
                    amax_pair = dev::absmax_pair(amax_pair, v[j].x);
                    amax_pair = dev::absmax_pair(amax_pair, v[j].y);
                    amax_pair = dev::absmax_pair(amax_pair, v[j].z);
                    amax_pair = dev::absmax_pair(amax_pair, v[j].w);
                    if constexpr (DBIAS) {
                        cs[0] += dev::bf16_lo(v[j].x); cs[1] += dev::bf16_hi(v[j].x);
                        cs[2] += dev::bf16_lo(v[j].y); cs[3] += dev::bf16_hi(v[j].y);
                        cs[4] += dev::bf16_lo(v[j].z); cs[5] += dev::bf16_hi(v[j].z);
                        cs[6] += dev::bf16_lo(v[j].w); cs[7] += dev::bf16_hi(v[j].w);
                    }
                    // FMT < 0: the format is the tensor's own (uniform per tile)
                    const uint2 q8 = FMT >= 0  ? dev::cast8<FMT < 0 ? 0 : FMT>(v[j], scale)
                                     : tfmt == 0 ? dev::cast8<0>(v[j], scale)
                                                 : dev::cast8<1>(v[j], scale);
                    if (col_ok && row0 + r < rows)
                        __stcs(reinterpret_cast<uint2*>(qrow + r * cols), q8);
                    if constexpr (WRITE_T)   // words 2c, 2c+1 of row r
                        *reinterpret_cast<uint2*>(sqb + r * kTileCols + ((2 * c) ^ swz(r)) * 4) = q8;
                }
            }
            if constexpr (DBIAS) {
                if (seg_end) {   // end of the run: fold the two row groups of the warp
#pragma unroll
                    for (int j = 0; j < 8; ++j) cs[j] += __shfl_xor_sync(0xFFFFFFFFu, cs[j], 16);
                    if (lane < 16) {
                        float4* dst = reinterpret_cast<float4*>(colsum + sb * kColsumFloats +
                                                                warp * kTileCols + 8 * c);
                        dst[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
                        dst[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) cs[j] = 0.0f;
                }
            }
        }

        // End of this CTA's run over the current tensor: fold the amax.
        if (last) {
            const unsigned m = __reduce_max_sync(0xFFFFFFFFu, dev::pair_to_f32_bits(amax_pair));
            if (lane == 0 && m != 0) atomicMax(&s_amax[sb], m);
            amax_pair = 0;
        }

        dev::consumer_sync(kFastThreads);
        if (*s_abort) {
            if (tid == 0) atomicOr(&g_device_error, kErrWaitTimeout);
            return;   // the producer drains its own loads
        }

        if (tid == 0) {
            if (last) {
                const unsigned m = s_amax[sb];
                s_amax[sb] = 0;
                if (m != 0) atomicMax(reinterpret_cast<unsigned*>(p.t[cur].amax), m);
            }
            if (first_tile) *p.t[cur].scale_inv = __fdiv_rn(1.0f, scale);
        }

        // ---------------- pass 2 ----------------
        if constexpr (WRITE_T) {
            const uint32_t* sq32 = reinterpret_cast<const uint32_t*>(sqb);
            uint32_t rw[kBlockRows];
#pragma unroll
            for (int j = 0; j < kBlockRows; ++j) {
                const int r = kBlockRows * b + j;
                rw[j] = sq32[r * (kTileCols / 4) + (w ^ swz(r))];
            }
            constexpr int kGroups = kBlockRows / 4;
            uint32_t o[4][kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g)
                dev::transpose4x4(rw[4 * g], rw[4 * g + 1], rw[4 * g + 2], rw[4 * g + 3], o[0][g],
                                  o[1][g], o[2][g], o[3][g]);
            const int64_t row = row0 + kBlockRows * b;
            if (row < rows) {
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const int64_t col = col0 + 4 * w + kq;
                    if (col >= cols) continue;
                    if constexpr (kGroups == 4)
                        __stcs(reinterpret_cast<uint4*>(out_t + col * rows + row),
                               make_uint4(o[kq][0], o[kq][1], o[kq][2], o[kq][3]));
                    else
                        __stcs(reinterpret_cast<uint2*>(out_t + col * rows + row),
                               make_uint2(o[kq][0], o[kq][1]));
                }
            }
        }
        if constexpr (DBIAS) {
            if (seg_end && tid < kTileCols && col0 + tid < cols) {
                const float* src = colsum + sb * kColsumFloats + tid;
                float sum = src[0];
#pragma unroll
                for (int j = 1; j < kWarps; ++j) sum += src[j * kTileCols];
                p.partial[int64_t(seg) * cols + col0 + tid] = sum;
            }
        }
    }
}

// ---- launch configuration ---------------------------------------------------
// Pipeline depth: 4 stages while each CTA has few tiles (the prologue loads
// dominate: keep as many in flight as possible), 3 stages for long runs
// (measured on GB300: fewer outstanding tile loads per SM leave DRAM more
// room for the output writes and sustain a higher read+write rate).
// Resident CTAs per SM: 1 (2 was measured and was slower).
constexpr int kMinBlocks = 1;
constexpr int kStagesShort = 4;
constexpr int kStagesLong = 3;
constexpr int64_t kLongRunTiles = 16;   // tiles per CTA from which the long setting wins

struct LaunchCache {
    std::mutex mu;
    int sms[64] = {0};
    bool attr_done[64][32] = {};
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

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lock(g_cache.mu);
        if (g_cache.sms[dev]) return g_cache.sms[dev];
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

template <int NT, int FMT, int STAGES, bool WRITE_T, bool DBIAS, bool PEND>
cudaError_t launch_stages(const FastParams<NT>& p, int key, cudaStream_t stream) {
    using L = SmemLayout<STAGES, WRITE_T, DBIAS>;
    auto kernel = fast_cast_transpose_kernel<NT, FMT, STAGES, kMinBlocks, WRITE_T, DBIAS, PEND>;
    int sms = 0;
    cudaError_t e = prepare(kernel, key, L::bytes, &sms);
    if (e != cudaSuccess) return e;
    const int64_t slots = int64_t(sms) * kMinBlocks;
    const int64_t grid = p.total_tiles < slots ? p.total_tiles : slots;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kBlockThreads), L::bytes,
                      stream, p);
}

template <int NT, int FMT, bool WRITE_T, bool DBIAS, bool PEND = false>
cudaError_t launch_variant(const FastParams<NT>& p, int key, cudaStream_t stream) {
    const int64_t slots = int64_t(device_sms()) * kMinBlocks;
    if (slots > 0 && p.total_tiles > kLongRunTiles * slots)
        return launch_stages<NT, FMT, kStagesLong, WRITE_T, DBIAS, PEND>(p, 2 * key + 1, stream);
    return launch_stages<NT, FMT, kStagesShort, WRITE_T, DBIAS, PEND>(p, 2 * key, stream);
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
    if (p.pend.hist != nullptr)
        return fmt == 0 ? launch_variant<1, 0, true, false, true>(p, 9, stream)
                        : launch_variant<1, 1, true, false, true>(p, 10, stream);
    return fmt == 0 ? launch_variant<1, 0, true, false>(p, 4, stream)
                    : launch_variant<1, 1, true, false>(p, 5, stream);
}

cudaError_t launch_fast_list(const FastParams<kMaxListPerLaunch>& p, int fmt,
                             cudaStream_t stream) {
    if (fmt < 0) return launch_variant<kMaxListPerLaunch, -1, true, false>(p, 8, stream);
    return fmt == 0 ? launch_variant<kMaxListPerLaunch, 0, true, false>(p, 6, stream)
                    : launch_variant<kMaxListPerLaunch, 1, true, false>(p, 7, stream);
}

namespace {
// The mbarrier expects one arrival that never comes: the wait must give up
// after limit_ns, leave a mark in the diagnostic word and return, exactly as
// the tile-load waits of the cast kernels do.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    dev::mbar_init(&bar, 1);
    dev::fence_barrier_init();
    if (!dev::mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(&g_device_error, kErrSelftestTimeout);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t limit_us, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(uint64_t(limit_us) * 1000ull);
    return cudaGetLastError();
}

cudaError_t read_device_error(unsigned* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

}  // namespace ct
