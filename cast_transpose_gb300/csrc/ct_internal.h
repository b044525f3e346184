// ct_internal.h -- shared declarations between the host ABI layer and the
// CUDA translation units of the cast-transpose library.  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ct {

// Tile of the TMA-staged kernels: 128 rows x 128 columns of bf16 (32 KB),
// processed by 256 threads.  Dbias partial sums are kept per 128-row tile by
// every kernel, so the workspace layout is [ceil(rows/128), cols] fp32.
constexpr int kTileRows = 128;
constexpr int kTileCols = 128;
constexpr int kThreads = 256;
constexpr int kMaxListPerLaunch = 64;

// Bits of the device diagnostic word.
constexpr unsigned kErrWaitTimeout = 1u;      // a kernel's mbarrier wait gave up
constexpr unsigned kErrSelftestTimeout = 2u;  // the bounded-wait self-test gave up (expected)

// One tensor of a TMA-path launch.  Pointers are device pointers.
// Deferred scale updates (ct_update.cuh, "deferred updates"): a cast that
// derives its scale from the history column as it stood before its run, the
// scale then, and the amaxes of the run's earlier casts (pending rows).
struct PendingScale {
    const float* hist;     // history column before the run, row stride `stride` (null: none)
    const float* scale0;   // the column's scale before the run
    const float* pending;  // pending rows of the column, row stride `stride`
    int64_t stride;
    int L;                 // history length, 1 .. 1024
    int k;                 // updates deferred so far, 0 .. min(32, L)
    int most_recent;       // the "most recent" rule: a_j = c_j
    float fp8_max;
    float two_pow_margin;
};

struct FastTensor {
    uint8_t* out;          // [rows, cols] FP8 codes (may be null: not written)
    uint8_t* out_t;        // [cols, rows] FP8 codes (null when no transpose)
    const float* scale;
    float* amax;
    float* scale_inv;
    int64_t rows;
    int64_t cols;
    int64_t tile_begin;    // first global tile index of this tensor
    int64_t tile_end;      // one past its last global tile index
    int64_t tile_cols;     // tiles per row of tiles
    int64_t tile_rows;     // rows of tiles
    int32_t fmt;           // FP8 format (read only by list launches with fmt < 0)
};

template <int NT>
struct FastParams {
    CUtensorMap map[NT];   // TMA descriptors of the bf16 inputs (64-B aligned)
    FastTensor t[NT];
    int n;
    int64_t total_tiles;
    const float* noop;     // nullable device flag
    float* partial;        // dbias partials [ceil(rows/128), cols], or null
    int x_ready;           // caller's promise: no kernel still running writes x
                           // (the first tiles may be loaded before the dependency wait)
    PendingScale pend;     // single tensors: deferred-update scale (pend.hist null: t[0].scale)
};

// Arguments of the general (any shape / alignment) kernels.
struct GeneralArgs {
    const uint16_t* x;
    uint8_t* out;          // may be null
    uint8_t* out_t;        // may be null
    const float* scale;
    float* amax;
    float* scale_inv;
    float* partial;        // dbias partials or null
    int64_t rows;
    int64_t cols;
    const float* noop;
    PendingScale pend;     // deferred-update scale (pend.hist null: *scale)
};

enum class Fmt : int { E4M3 = 0, E5M2 = 1 };

// Launch with programmatic stream serialisation allowed (see pdl_wait in
// ct_device.cuh): the kernel may be scheduled while its predecessor in the
// stream still runs, and waits for it on the device.  Recorded as a
// programmatic edge when the stream is being captured into a graph.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- launchers (return cudaGetLastError() of the launch) -----------------
// TMA path.  `variant`: 0 = cast + transpose, 1 = cast only.  `dbias`
// requires n == 1 and variant 0.
cudaError_t launch_fast(const FastParams<1>& p, int fmt, bool dbias, int variant,
                        cudaStream_t stream);
// fmt < 0: each tensor's own t[i].fmt.
cudaError_t launch_fast_list(const FastParams<kMaxListPerLaunch>& p, int fmt,
                             cudaStream_t stream);

// Direct-load path (ct_direct.cu): one CTA per 128x128 tile, x read with
// plain 16-byte loads; same eligibility as the TMA path (rows % 16 == 0,
// cols % 8 == 0, 16-byte aligned x, out and out_t).  Chosen for launches of
// at least kDirectMinTiles tiles (at most INT32_MAX), where it sustains a
// higher read+write rate than the persistent TMA kernel; the persistent
// kernel keeps the smaller launches, whose tiles it spreads evenly and whose
// first loads it overlaps with the previous kernel.
template <int NT>
struct DirectParams {
    const uint16_t* x[NT];  // bf16 inputs
    FastTensor t[NT];
    int n;
    int64_t total_tiles;
    const float* noop;      // nullable device flag
    float* partial;         // dbias partials [ceil(rows/128), cols] (one row per tile row), or null
    int x_ready;            // caller's promise: no kernel still running writes x
                            // (the tiles may be loaded before the dependency wait)
    int prefetch_ctas;      // CTAs (from block 0) that prefetch their tile into L2 before the wait
    int loop_ctas;          // looping launches: CTAs that loop over loop_tiles tiles per group,
    int loop_tiles;         // then rest_chunk consecutive tiles per group for the CTAs after them
    int rest_chunk;
};
constexpr int64_t kDirectMinTiles = 2048;
// `variant`: 0 = cast + transpose, 1 = cast only; `dbias` requires variant 0.
cudaError_t launch_direct(const DirectParams<1>& p, int fmt, bool dbias, int variant,
                          cudaStream_t stream);
// fmt < 0: each tensor's own t[i].fmt.
cudaError_t launch_direct_list(const DirectParams<kMaxListPerLaunch>& p, int fmt,
                               cudaStream_t stream);

// General path.
cudaError_t launch_general(const GeneralArgs& a, int fmt, cudaStream_t stream);
// q[i] = fp8(x[i] * scale) over n elements as one array (x 16-byte, q 8-byte
// aligned), amax max-merged, scale_inv written.  `keep_q`: q is stored with
// the L2 evict-last priority, for a transpose that reads it next (which
// lowers the priority again as it stages the lines).
cudaError_t launch_cast_flat(const uint16_t* x, int64_t n, uint8_t* q, const float* scale,
                             float* amax, float* scale_inv, int fmt, const float* noop,
                             cudaStream_t stream, bool keep_q = false);

// Dbias schedule and partial sums.  The TMA kernel splits the R = ceil(rows
// / 128) tile rows into bands of H = min(kDbiasBand, R) tile rows (the last
// band may be shorter) and hands out "units" -- one band of one 128-column strip,
// unit u = band * S + strip -- round-robin to its CTAs.  A CTA walks down
// the H tiles of a unit, sums its columns over them, and writes one partial
// row per band: partial[band][col].  CTAs running at the same time work on
// neighbouring strips of the same band, i.e. on the same rows of x.  The
// general kernel writes one partial row per tile row, i.e. H = 1.
struct DbiasUnits {
    int64_t H;        // tile rows per full band
    int64_t bands;    // ceil(R / H)
    int64_t last_h;   // tile rows of the last band
};
__host__ __device__ __forceinline__ DbiasUnits dbias_units(int64_t R, int64_t H) {
    DbiasUnits u;
    u.H = H;
    u.bands = (R + H - 1) / H;
    u.last_h = R - (u.bands - 1) * H;
    return u;
}
// Band height: 4 measured best on GB300 (shorter bands balance the last
// wave of units better, longer ones write fewer partial rows).
constexpr int64_t kDbiasBand = 4;

// Dbias finish: db[j] = sum of the `runs` partial rows (compensated fp32),
// stored as fp32, or (db_bf16) rounded to bf16, nearest even.
cudaError_t launch_dbias_finish(const float* partial, int64_t runs, int64_t cols, void* dbias,
                                bool db_bf16, const float* noop, cudaStream_t stream);

// Scale update of `count` columns of a [hist_len, stride] history (scale and
// scale_inv indexed like the columns).
cudaError_t launch_scale_update(float* hist, float* scale, float* scale_inv, int hist_len,
                                int count, int64_t stride, int fmt, int margin, int most_recent,
                                const float* noop, cudaStream_t stream);
// The K deferred updates of `count` columns (hist_len <= 1024, 1 <= K <=
// min(32, hist_len)); pending is [K, stride].
cudaError_t launch_scale_update_pending(float* hist, float* pending, float* scale,
                                        float* scale_inv, int hist_len, int K, int count,
                                        int64_t stride, int fmt, int margin, int most_recent,
                                        const float* noop, cudaStream_t stream);

// FP8 byte transpose.  `fast` requires rows % 16 == 0, cols % 16 == 0 and
// 16-byte aligned pointers.  `after_cast` (odd shapes, only where
// odd_transpose_loops_after_cast holds): the transpose of a q that the flat
// cast has just stored with the L2 evict-last priority; the looping launch
// then takes the tiles in reverse order and demotes the lines it stages.
cudaError_t launch_transpose(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out,
                             const float* noop, bool fast, cudaStream_t stream,
                             bool after_cast = false);
// Whether a rows x cols odd-shape transpose has at least one wave of tiles
// for the looping launch (smaller ones keep one tile per CTA after the cast).
bool odd_transpose_loops_after_cast(int64_t rows, int64_t cols);

// FP8 conversion of n fp32 values (no scale): the cast kernels' conversion step.
cudaError_t launch_convert_f32(const float* in, int64_t n, int fmt, uint8_t* out,
                               cudaStream_t stream);

// Diagnostic word (device of the calling thread).
cudaError_t read_device_error(unsigned* value, bool clear);

// Bounded-wait self-test: one CTA waits `limit_us` on an mbarrier that
// nothing completes, then records kErrSelftestTimeout and returns.
cudaError_t launch_wait_selftest(uint32_t limit_us, cudaStream_t stream);

// Number of SMs and persistent CTAs per SM for the TMA kernels of this
// device (cached per device).
int persistent_grid(int variant_key, int device);

}  // namespace ct
