// ct_api.cu -- the C ABI of include/cast_transpose.h: host-side argument
// checks, TMA descriptor encoding and dispatch between the persistent
// TMA-staged kernel (fast shapes, under kDirectMinTiles tiles), the
// direct-load kernel (fast shapes, from kDirectMinTiles tiles on, and odd
// row counts), the flat cast with the FP8 transpose of q (other shapes and
// x alignments with q 8-byte aligned), and the general kernel (everything
// else).  No device memory is allocated here, no stream or device is
// synchronised, and no device memory is read, so every call can be captured
// in a CUDA graph.
#include "../../include/cast_transpose.h"
#include "ct_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

namespace {

// Deferred updates: the longest history and run they take.
constexpr int kPendingMaxHist = 1024;
constexpr int kPendingMaxRun = 32;

using ct::DirectParams;
using ct::FastParams;
using ct::FastTensor;

// ---- driver entry point for TMA descriptor encoding -------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 [rows, cols] row-major, box 128 x 128, zero fill outside the matrix.
bool encode_bf16_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {ct::kTileCols, ct::kTileRows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- argument checks ---------------------------------------------------------
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;   // TMA coordinates are int32

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
};
inline Range range_of(const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}
inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

bool shape_ok(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return false;
    if (rows == 0 || cols == 0) return true;
    // element offsets must fit in int64 with room for the bf16 byte offsets
    return rows <= (int64_t(1) << 40) / cols;
}

// The fast kernels store 16-row blocks of the transpose as 16-byte vectors
// (rows % 16) and read 8-element row chunks as 16-byte vectors (cols % 8,
// which also makes the TMA row stride a multiple of 16 bytes).
bool fast_shape(int64_t rows, int64_t cols) {
    return rows % 16 == 0 && cols % 8 == 0 && rows <= kMaxDim && cols <= kMaxDim;
}

// Checks shared by the single-tensor cast entry points.
// An empty matrix (rows or cols == 0) passes with any pointers, NULL included:
// nothing is launched and nothing is written for it.
int check_cast(const void* x, int64_t rows, int64_t cols, const float* scale, float* amax,
               float* scale_inv, void* out, void* out_t, bool need_t, int fmt) {
    if (fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    if (!shape_ok(rows, cols)) return CT_ERR_SHAPE;
    if (rows == 0 || cols == 0) return CT_OK;
    if (!x || !scale || !amax || !scale_inv || !out || (need_t && !out_t)) return CT_ERR_NULL;
    if (!aligned(x, 2) || !aligned(scale, 4) || !aligned(amax, 4) || !aligned(scale_inv, 4))
        return CT_ERR_ALIGN;
    const int64_t n = rows * cols;
    const Range rx = range_of(x, 2 * n), rq = range_of(out, n);
    const Range rs = range_of(scale, 4), ra = range_of(amax, 4), ri = range_of(scale_inv, 4);
    Range outs[4] = {rq, ra, ri, {0, 0}};
    int nouts = 3;
    if (out_t) outs[nouts++] = range_of(out_t, n);
    for (int i = 0; i < nouts; ++i) {
        if (overlap(outs[i], rx) || overlap(outs[i], rs)) return CT_ERR_ALIAS;
        for (int j = i + 1; j < nouts; ++j)
            if (overlap(outs[i], outs[j])) return CT_ERR_ALIAS;
    }
    return CT_OK;
}

bool fast_eligible(const void* x, int64_t rows, int64_t cols, const void* out, const void* out_t) {
    return fast_shape(rows, cols) && aligned(x, 16) && aligned(out, 16) &&
           (out_t == nullptr || aligned(out_t, 16)) && encode_fn() != nullptr;
}

// rows % 16 != 0 with whole 16-byte row chunks: the direct-load kernel, whose
// transposed stores then take any alignment (the last 16-row block short).
bool ragged_rows_eligible(const void* x, int64_t rows, int64_t cols, const void* out,
                          const void* out_t) {
    return rows % 16 != 0 && cols % 8 == 0 && rows <= kMaxDim && cols <= kMaxDim &&
           aligned(x, 16) && aligned(out, 16) && (out_t == nullptr || aligned(out_t, 16));
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? CT_OK : CT_ERR_CUDA; }

void fill_tensor(FastTensor& t, const void* out, const void* out_t, const float* scale,
                 float* amax, float* scale_inv, int64_t rows, int64_t cols, int64_t tile_begin) {
    t.out = static_cast<uint8_t*>(const_cast<void*>(out));
    t.out_t = static_cast<uint8_t*>(const_cast<void*>(out_t));
    t.scale = scale;
    t.amax = amax;
    t.scale_inv = scale_inv;
    t.rows = rows;
    t.cols = cols;
    t.tile_cols = (cols + ct::kTileCols - 1) / ct::kTileCols;
    t.tile_rows = (rows + ct::kTileRows - 1) / ct::kTileRows;
    t.tile_begin = tile_begin;
    t.tile_end = tile_begin + t.tile_rows * t.tile_cols;
}

// `runs_out` (dbias only): the number of partial rows the launched kernel
// writes per column (one per band of tile rows on the TMA path, one per tile
// row on the direct and general paths).  `x_ready`: CT_X_READY (TMA and
// direct paths).  `pend`: deferred-update scale source (cast-transpose only:
// the TMA kernel for every aligned shape, else the general kernel), or null
// to cast with *scale.
int cast_impl(const void* x, int64_t rows, int64_t cols, const float* scale, float* amax,
              float* scale_inv, void* out, void* out_t, float* partial, int fmt,
              const float* noop, cudaStream_t stream, int64_t* runs_out = nullptr,
              bool x_ready = false, const ct::PendingScale* pend = nullptr) {
    const int64_t R = (rows + ct::kTileRows - 1) / ct::kTileRows;
    const bool ragged_rows = ragged_rows_eligible(x, rows, cols, out, out_t);
    if (ragged_rows || fast_eligible(x, rows, cols, out, out_t)) {
        const int64_t tiles = R * ((cols + ct::kTileCols - 1) / ct::kTileCols);
        if ((ragged_rows || tiles >= ct::kDirectMinTiles) && tiles <= INT32_MAX && !pend) {
            DirectParams<1> d;
            std::memset(&d, 0, sizeof(d));
            d.x[0] = static_cast<const uint16_t*>(x);
            fill_tensor(d.t[0], out, out_t, scale, amax, scale_inv, rows, cols, 0);
            d.n = 1;
            d.total_tiles = tiles;
            d.noop = noop;
            d.partial = partial;
            d.x_ready = x_ready ? 1 : 0;
            if (runs_out) *runs_out = R;
            return cuda_status(ct::launch_direct(d, fmt, partial != nullptr, out_t ? 0 : 1, stream));
        }
    }
    if (fast_eligible(x, rows, cols, out, out_t)) {
        FastParams<1> p;
        std::memset(&p, 0, sizeof(p));
        if (!encode_bf16_map(&p.map[0], x, rows, cols)) return CT_ERR_CUDA;
        fill_tensor(p.t[0], out, out_t, scale, amax, scale_inv, rows, cols, 0);
        p.n = 1;
        p.total_tiles = p.t[0].tile_end;
        p.noop = noop;
        p.partial = partial;
        p.x_ready = x_ready ? 1 : 0;
        if (pend) p.pend = *pend;
        if (runs_out) *runs_out = ct::dbias_units(R, R < ct::kDbiasBand ? R : ct::kDbiasBand).bands;
        return cuda_status(ct::launch_fast(p, fmt, partial != nullptr, out_t ? 0 : 1, stream));
    }
    // With q 8-byte aligned, q is one flat array of rows * cols elements
    // whatever the row length: the flat cast writes it (an x off a 16-byte
    // boundary through the shifted variant).  With a transpose and rows % 16
    // != 0, the FP8 transpose of q then writes qT (8191x12287: 4.77 TB/s, x 2
    // bytes off 4.62, against 3.49 / 3.45 for the general kernel); with rows %
    // 16 == 0 the general kernel's transposed stores are aligned, and it stays
    // faster (8192x12284: 5.01 against 4.29 TB/s; x 2 bytes off 5.15 against
    // 4.30).
    if (partial == nullptr && pend == nullptr && out != nullptr && aligned(out, 8) &&
        (out_t == nullptr || rows % 16 != 0)) {
        // A transpose to follow over at least one wave of tiles: q is stored
        // with the L2 evict-last priority and read back by the looping launch,
        // which demotes its lines (ct::launch_transpose).
        const bool tfast = rows % 16 == 0 && cols % 16 == 0 && aligned(out, 16) &&
                           aligned(out_t, 16);
        const bool keep =
            out_t != nullptr && !tfast && ct::odd_transpose_loops_after_cast(rows, cols);
        const cudaError_t e = ct::launch_cast_flat(static_cast<const uint16_t*>(x), rows * cols,
                                                   static_cast<uint8_t*>(out), scale, amax,
                                                   scale_inv, fmt, noop, stream, /*keep_q=*/keep);
        if (e != cudaSuccess || out_t == nullptr) return cuda_status(e);
        return cuda_status(ct::launch_transpose(static_cast<const uint8_t*>(out), rows, cols,
                                                static_cast<uint8_t*>(out_t), noop, tfast,
                                                stream, /*after_cast=*/keep));
    }
    ct::GeneralArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.out = static_cast<uint8_t*>(out);
    a.out_t = static_cast<uint8_t*>(out_t);
    a.scale = scale;
    a.amax = amax;
    a.scale_inv = scale_inv;
    a.partial = partial;
    a.rows = rows;
    a.cols = cols;
    a.noop = noop;
    a.pend = pend ? *pend : ct::PendingScale{};
    if (runs_out) *runs_out = R;
    return cuda_status(ct::launch_general(a, fmt, stream));
}

int64_t row_tiles(int64_t rows) { return (rows + ct::kTileRows - 1) / ct::kTileRows; }

}  // namespace

extern "C" {

const char* ct_status_string(int status) {
    switch (status) {
        case CT_OK: return "CT_OK";
        case CT_ERR_NULL: return "CT_ERR_NULL: a required pointer is NULL";
        case CT_ERR_SHAPE: return "CT_ERR_SHAPE: invalid matrix shape";
        case CT_ERR_ALIGN: return "CT_ERR_ALIGN: misaligned buffer";
        case CT_ERR_FORMAT: return "CT_ERR_FORMAT: unknown FP8 format";
        case CT_ERR_ARG: return "CT_ERR_ARG: invalid argument";
        case CT_ERR_ALIAS: return "CT_ERR_ALIAS: overlapping buffers";
        case CT_ERR_WORKSPACE: return "CT_ERR_WORKSPACE: workspace missing or too small";
        case CT_ERR_CUDA: return "CT_ERR_CUDA: CUDA call failed";
        default: return "unknown status";
    }
}

int fp8_cast_transpose(const void* x, int64_t rows, int64_t cols, const float* scale,
                       float* amax, float* scale_inv, void* out, void* out_t, int fmt,
                       const float* noop_flag, void* stream) {
    const int st = check_cast(x, rows, cols, scale, amax, scale_inv, out, out_t, true, fmt);
    if (st != CT_OK) return st;
    if (rows == 0 || cols == 0) return CT_OK;
    return cast_impl(x, rows, cols, scale, amax, scale_inv, out, out_t, nullptr, fmt, noop_flag,
                     static_cast<cudaStream_t>(stream));
}

int fp8_cast_transpose_ex(const void* x, int64_t rows, int64_t cols, const float* scale,
                          float* amax, float* scale_inv, void* out, void* out_t, int fmt,
                          const float* noop_flag, unsigned flags, void* stream) {
    if (flags & ~static_cast<unsigned>(CT_X_READY)) return CT_ERR_ARG;
    const int st = check_cast(x, rows, cols, scale, amax, scale_inv, out, out_t, true, fmt);
    if (st != CT_OK) return st;
    if (rows == 0 || cols == 0) return CT_OK;
    return cast_impl(x, rows, cols, scale, amax, scale_inv, out, out_t, nullptr, fmt, noop_flag,
                     static_cast<cudaStream_t>(stream), nullptr, (flags & CT_X_READY) != 0);
}

int fp8_cast(const void* x, int64_t rows, int64_t cols, const float* scale, float* amax,
             float* scale_inv, void* out, int fmt, const float* noop_flag, void* stream) {
    const int st = check_cast(x, rows, cols, scale, amax, scale_inv, out, nullptr, false, fmt);
    if (st != CT_OK) return st;
    if (rows == 0 || cols == 0) return CT_OK;
    return cast_impl(x, rows, cols, scale, amax, scale_inv, out, nullptr, nullptr, fmt, noop_flag,
                     static_cast<cudaStream_t>(stream));
}

size_t fp8_dbias_cast_transpose_workspace_size(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    const size_t bytes = static_cast<size_t>(row_tiles(rows)) * static_cast<size_t>(cols) * 4;
    return (bytes + 15) & ~size_t(15);
}

int fp8_dbias_cast_transpose(const void* dy, int64_t rows, int64_t cols, const float* scale,
                             float* amax, float* scale_inv, void* out, void* out_t,
                             float* dbias, void* workspace, size_t workspace_bytes, int fmt,
                             const float* noop_flag, void* stream) {
    return fp8_dbias_cast_transpose_ex(dy, rows, cols, scale, amax, scale_inv, out, out_t, dbias,
                                       CT_DBIAS_FP32, workspace, workspace_bytes, fmt, noop_flag,
                                       stream);
}

int fp8_dbias_cast_transpose_ex(const void* dy, int64_t rows, int64_t cols, const float* scale,
                                float* amax, float* scale_inv, void* out, void* out_t,
                                void* dbias, int dbias_dtype, void* workspace,
                                size_t workspace_bytes, int fmt, const float* noop_flag,
                                void* stream) {
    const bool x_ready = (dbias_dtype & CT_DBIAS_X_READY) != 0;
    dbias_dtype &= ~static_cast<int>(CT_DBIAS_X_READY);
    if (dbias_dtype != CT_DBIAS_FP32 && dbias_dtype != CT_DBIAS_BF16) return CT_ERR_ARG;
    int st = check_cast(dy, rows, cols, scale, amax, scale_inv, out, out_t, true, fmt);
    if (st != CT_OK) return st;
    if (rows == 0 || cols == 0) return CT_OK;
    if (!dbias) return CT_ERR_NULL;
    const int64_t db_elem = dbias_dtype == CT_DBIAS_BF16 ? 2 : 4;
    if (!aligned(dbias, uintptr_t(db_elem))) return CT_ERR_ALIGN;
    const size_t need = fp8_dbias_cast_transpose_workspace_size(rows, cols);
    if (!workspace || workspace_bytes < need) return CT_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return CT_ERR_ALIGN;
    const int64_t n = rows * cols;
    const Range rdb = range_of(dbias, db_elem * cols), rws = range_of(workspace, int64_t(need));
    const Range others[6] = {range_of(dy, 2 * n), range_of(out, n), range_of(out_t, n),
                             range_of(scale, 4), range_of(amax, 4), range_of(scale_inv, 4)};
    if (overlap(rdb, rws)) return CT_ERR_ALIAS;
    for (const Range& r : others)
        if (overlap(rdb, r) || overlap(rws, r)) return CT_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* partial = static_cast<float*>(workspace);
    int64_t runs = 0;
    st = cast_impl(dy, rows, cols, scale, amax, scale_inv, out, out_t, partial, fmt, noop_flag, s,
                   &runs, x_ready);
    if (st != CT_OK) return st;
    return cuda_status(ct::launch_dbias_finish(partial, runs, cols, dbias,
                                               dbias_dtype == CT_DBIAS_BF16, noop_flag, s));
}

namespace {
// Shared by the single-format and per-tensor-format list entry points:
// fmts == nullptr means every entry uses `fmt`.
int multi_impl(const ct_tensor_desc* descs, const int* fmts, int n, int fmt,
               const float* noop_flag, cudaStream_t s) {
    if (n < 0) return CT_ERR_ARG;
    if (n == 0) return CT_OK;
    if (!descs) return CT_ERR_NULL;
    auto fmt_of = [&](int i) { return fmts ? fmts[i] : fmt; };
    if (!fmts && fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    for (int i = 0; i < n; ++i) {
        const ct_tensor_desc& d = descs[i];
        const int st = check_cast(d.x, d.rows, d.cols, d.scale, d.amax, d.scale_inv, d.out,
                                  d.out_t, true, fmt_of(i));
        if (st != CT_OK) return st;
    }
    // outputs of one entry must not overlap anything of another entry
    for (int i = 0; i < n; ++i) {
        const ct_tensor_desc& a = descs[i];
        if (a.rows == 0 || a.cols == 0) continue;
        const int64_t na = a.rows * a.cols;
        const Range oa[4] = {range_of(a.out, na), range_of(a.out_t, na), range_of(a.amax, 4),
                             range_of(a.scale_inv, 4)};
        for (int j = 0; j < n; ++j) {
            const ct_tensor_desc& b = descs[j];
            if (j == i || b.rows == 0 || b.cols == 0) continue;
            const int64_t nb = b.rows * b.cols;
            const Range ob[6] = {range_of(b.out, nb),   range_of(b.out_t, nb),
                                 range_of(b.amax, 4),   range_of(b.scale_inv, 4),
                                 range_of(b.x, 2 * nb), range_of(b.scale, 4)};
            for (const Range& r1 : oa)
                for (const Range& r2 : ob)
                    if (overlap(r1, r2)) return CT_ERR_ALIAS;
        }
    }
    // fast entries go into list launches of up to kMaxListPerLaunch tensors;
    // the others go through the single-tensor dispatch (the direct kernel for
    // rows % 16 != 0 with whole row chunks, else the general kernel)
    std::vector<int> fast, general;
    for (int i = 0; i < n; ++i) {
        const ct_tensor_desc& d = descs[i];
        if (d.rows == 0 || d.cols == 0) continue;
        (fast_eligible(d.x, d.rows, d.cols, d.out, d.out_t) ? fast : general).push_back(i);
    }
    for (size_t base = 0; base < fast.size(); base += ct::kMaxListPerLaunch) {
        const size_t end = std::min(fast.size(), base + size_t(ct::kMaxListPerLaunch));
        int64_t chunk_tiles = 0;
        for (size_t k = base; k < end; ++k) {
            const ct_tensor_desc& d = descs[fast[k]];
            chunk_tiles += row_tiles(d.rows) * ((d.cols + ct::kTileCols - 1) / ct::kTileCols);
        }
        if (chunk_tiles >= ct::kDirectMinTiles && chunk_tiles <= INT32_MAX) {
            static thread_local DirectParams<ct::kMaxListPerLaunch> q;
            std::memset(&q, 0, sizeof(q));
            int64_t tiles = 0;
            int m = 0;
            for (size_t k = base; k < end; ++k, ++m) {
                const ct_tensor_desc& d = descs[fast[k]];
                q.x[m] = static_cast<const uint16_t*>(d.x);
                fill_tensor(q.t[m], d.out, d.out_t, d.scale, d.amax, d.scale_inv, d.rows, d.cols,
                            tiles);
                q.t[m].fmt = fmt_of(fast[k]);
                tiles = q.t[m].tile_end;
            }
            q.n = m;
            q.total_tiles = tiles;
            q.noop = noop_flag;
            q.partial = nullptr;
            const int st = cuda_status(ct::launch_direct_list(q, fmts ? -1 : fmt, s));
            if (st != CT_OK) return st;
            continue;
        }
        static thread_local FastParams<ct::kMaxListPerLaunch> p;
        std::memset(&p, 0, sizeof(p));
        int64_t tiles = 0;
        int m = 0;
        for (size_t k = base; k < end; ++k, ++m) {
            const ct_tensor_desc& d = descs[fast[k]];
            if (!encode_bf16_map(&p.map[m], d.x, d.rows, d.cols)) return CT_ERR_CUDA;
            fill_tensor(p.t[m], d.out, d.out_t, d.scale, d.amax, d.scale_inv, d.rows, d.cols, tiles);
            p.t[m].fmt = fmt_of(fast[k]);
            tiles = p.t[m].tile_end;
        }
        // unused slots: empty tile ranges past the end
        for (int k = m; k < ct::kMaxListPerLaunch; ++k) {
            p.t[k].tile_begin = tiles;
            p.t[k].tile_end = tiles;
        }
        p.n = m;
        p.total_tiles = tiles;
        p.noop = noop_flag;
        p.partial = nullptr;
        const int st = cuda_status(ct::launch_fast_list(p, fmts ? -1 : fmt, s));
        if (st != CT_OK) return st;
    }
    for (int i : general) {
        const ct_tensor_desc& d = descs[i];
        const int st = cast_impl(d.x, d.rows, d.cols, d.scale, d.amax, d.scale_inv, d.out, d.out_t,
                                 nullptr, fmt_of(i), noop_flag, s);
        if (st != CT_OK) return st;
    }
    return CT_OK;
}
}  // namespace

int fp8_multi_cast_transpose(const ct_tensor_desc* descs, int n, int fmt,
                             const float* noop_flag, void* stream) {
    return multi_impl(descs, nullptr, n, fmt, noop_flag, static_cast<cudaStream_t>(stream));
}

int fp8_multi_cast_transpose_ex(const ct_tensor_desc* descs, const int* fmts, int n,
                                const float* noop_flag, void* stream) {
    if (n > 0 && !fmts) return CT_ERR_NULL;
    return multi_impl(descs, fmts, n, CT_E4M3, noop_flag, static_cast<cudaStream_t>(stream));
}

int fp8_amax_and_scale_update_ex(float* amax_history, float* scale, float* scale_inv,
                                 int hist_len, int n, int fmt, int margin, int amax_algo,
                                 const float* noop_flag, void* stream) {
    if (n < 0 || hist_len < 1 || margin < 0 || margin > 126) return CT_ERR_ARG;
    if (amax_algo != CT_AMAX_MAX && amax_algo != CT_AMAX_MOST_RECENT) return CT_ERR_ARG;
    if (fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    if (n == 0) return CT_OK;
    if (!amax_history || !scale || !scale_inv) return CT_ERR_NULL;
    if (!aligned(amax_history, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4))
        return CT_ERR_ALIGN;
    const Range rh = range_of(amax_history, int64_t(4) * hist_len * n);
    const Range rs = range_of(scale, int64_t(4) * n), ri = range_of(scale_inv, int64_t(4) * n);
    if (overlap(rh, rs) || overlap(rh, ri) || overlap(rs, ri)) return CT_ERR_ALIAS;
    return cuda_status(ct::launch_scale_update(amax_history, scale, scale_inv, hist_len, n, n, fmt,
                                               margin, amax_algo == CT_AMAX_MOST_RECENT ? 1 : 0,
                                               noop_flag, static_cast<cudaStream_t>(stream)));
}

int fp8_amax_and_scale_update(float* amax_history, float* scale, float* scale_inv,
                              int hist_len, int n, int fmt, int margin,
                              const float* noop_flag, void* stream) {
    return fp8_amax_and_scale_update_ex(amax_history, scale, scale_inv, hist_len, n, fmt, margin,
                                        CT_AMAX_MAX, noop_flag, stream);
}

int fp8_cast_transpose_pending(const void* x, int64_t rows, int64_t cols,
                               const float* amax_history, const float* scale, float* pending,
                               int hist_len, int n, int col, int k, int margin, int amax_algo,
                               float* scale_inv, void* out, void* out_t, int fmt,
                               const float* noop_flag, unsigned flags, void* stream) {
    if (flags & ~static_cast<unsigned>(CT_X_READY)) return CT_ERR_ARG;
    if (hist_len < 1 || hist_len > kPendingMaxHist || n < 1 || col < 0 || col >= n || k < 0 ||
        k >= kPendingMaxRun || k >= hist_len || margin < 0 || margin > 126)
        return CT_ERR_ARG;
    if (amax_algo != CT_AMAX_MAX && amax_algo != CT_AMAX_MOST_RECENT) return CT_ERR_ARG;
    if (!amax_history || !scale || !pending) return CT_ERR_NULL;
    if (!aligned(amax_history, 4) || !aligned(pending, 4)) return CT_ERR_ALIGN;
    float* amax = pending + int64_t(k) * n + col;
    const int st = check_cast(x, rows, cols, scale + col, amax, scale_inv, out, out_t, true, fmt);
    if (st != CT_OK) return st;
    if (rows == 0 || cols == 0) return CT_OK;
    // the outputs against the inputs the scale is derived from
    const Range rh = range_of(amax_history, int64_t(4) * hist_len * n);
    const Range rs = range_of(scale, int64_t(4) * n), rp = range_of(pending, int64_t(4) * k * n);
    const int64_t nq = rows * cols;
    const Range outs[4] = {range_of(out, nq), range_of(out_t, nq), range_of(scale_inv, 4),
                           range_of(amax, 4)};
    for (const Range& o : outs)
        if (overlap(o, rh) || overlap(o, rs) || overlap(o, rp)) return CT_ERR_ALIAS;
    ct::PendingScale ps;
    ps.hist = amax_history + col;
    ps.scale0 = scale + col;
    ps.pending = pending + col;
    ps.stride = n;
    ps.L = hist_len;
    ps.k = k;
    ps.most_recent = amax_algo == CT_AMAX_MOST_RECENT ? 1 : 0;
    ps.fp8_max = fmt == CT_E4M3 ? 448.0f : 57344.0f;
    ps.two_pow_margin = std::ldexp(1.0f, margin);
    return cast_impl(x, rows, cols, scale + col, amax, scale_inv, out, out_t, nullptr, fmt,
                     noop_flag, static_cast<cudaStream_t>(stream), nullptr,
                     (flags & CT_X_READY) != 0, &ps);
}

int fp8_amax_and_scale_update_pending(float* amax_history, float* scale, float* scale_inv,
                                      float* pending, int hist_len, int n, int run, int fmt,
                                      int margin, int amax_algo, const float* noop_flag,
                                      void* stream) {
    if (n < 0 || hist_len < 1 || hist_len > kPendingMaxHist || run < 1 ||
        run > kPendingMaxRun || run > hist_len || margin < 0 || margin > 126)
        return CT_ERR_ARG;
    if (amax_algo != CT_AMAX_MAX && amax_algo != CT_AMAX_MOST_RECENT) return CT_ERR_ARG;
    if (fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    if (n == 0) return CT_OK;
    if (!amax_history || !scale || !scale_inv || !pending) return CT_ERR_NULL;
    if (!aligned(amax_history, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4) ||
        !aligned(pending, 4))
        return CT_ERR_ALIGN;
    const Range rh = range_of(amax_history, int64_t(4) * hist_len * n);
    const Range rs = range_of(scale, int64_t(4) * n), ri = range_of(scale_inv, int64_t(4) * n);
    const Range rp = range_of(pending, int64_t(4) * run * n);
    const Range all[4] = {rh, rs, ri, rp};
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (overlap(all[i], all[j])) return CT_ERR_ALIAS;
    return cuda_status(ct::launch_scale_update_pending(
        amax_history, pending, scale, scale_inv, hist_len, run, n, n, fmt, margin,
        amax_algo == CT_AMAX_MOST_RECENT ? 1 : 0, noop_flag, static_cast<cudaStream_t>(stream)));
}

int fp8_transpose(const void* in, int64_t rows, int64_t cols, void* out, const float* noop_flag,
                  void* stream) {
    if (!shape_ok(rows, cols)) return CT_ERR_SHAPE;
    if (rows == 0 || cols == 0) return CT_OK;
    if (!in || !out) return CT_ERR_NULL;
    if (overlap(range_of(in, rows * cols), range_of(out, rows * cols))) return CT_ERR_ALIAS;
    const bool fast = rows % 16 == 0 && cols % 16 == 0 && aligned(in, 16) && aligned(out, 16);
    return cuda_status(ct::launch_transpose(static_cast<const uint8_t*>(in), rows, cols,
                                            static_cast<uint8_t*>(out), noop_flag, fast,
                                            static_cast<cudaStream_t>(stream)));
}

int ct_fp8_convert_f32(const float* in, int64_t n, int fmt, void* out, void* stream) {
    if (fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    if (n < 0 || n > (int64_t(1) << 40)) return CT_ERR_SHAPE;
    if (n == 0) return CT_OK;
    if (!in || !out) return CT_ERR_NULL;
    if (!aligned(in, 4)) return CT_ERR_ALIGN;
    if (overlap(range_of(in, 4 * n), range_of(out, n))) return CT_ERR_ALIAS;
    return cuda_status(ct::launch_convert_f32(in, n, fmt, static_cast<uint8_t*>(out),
                                              static_cast<cudaStream_t>(stream)));
}

int ct_selftest_bounded_wait(unsigned int limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 1000000u) return CT_ERR_ARG;
    return cuda_status(ct::launch_wait_selftest(limit_us, static_cast<cudaStream_t>(stream)));
}

int ct_device_error(unsigned int* value_out, int clear) {
    if (!value_out) return CT_ERR_NULL;
    return cuda_status(ct::read_device_error(value_out, clear != 0));
}

}  // extern "C"
