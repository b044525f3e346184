/*
 * cast_transpose.h -- C ABI of the GB300 (sm_103a) FP8 cast-transpose library.
 *
 * The library turns bf16 matrices into FP8 tensors for delayed-scaling
 * training: the FP8 bytes, their transpose, the amax that feeds the next
 * scale, and the tensor's own scale-inverse, all in one pass over HBM.
 *
 * Sources of the operations (pages of the NVIDIA TransformerEngine project):
 *   [A] "[PyTorch] cuda graph support": the DbiasCastTranspose example in the
 *       transpose-cache discussion (db = dy.sum(dim=0); dx = cast_transpose(dy),
 *       an FP8 tensor with its transpose cached); the feature list (amaxes
 *       reduced within the current iteration; transposes made persistent for
 *       graph capture; scale-inverses no longer frozen).
 *   [B] "[PyTorch] Refactor FP8 workspaces in linear modules": Motivations
 *       (the FP8 tensor keeps a private scale-inverse that matches its bytes;
 *       the scale update kernel; the too-tiny-amax / infinite-scale case;
 *       the cost of a separate scale-inverse initialisation launch) and the
 *       lazy transpose-caching bullet (the transpose kernel must still be
 *       captured in a CUDA graph and skipped at replay through a noop flag).
 *   [C] "[PyTorch] Userbuffers support in operation-based API": FP8 tensors
 *       are built on caller-provided data / data_transpose buffers.
 *
 * FP8 formats: E4M3 (bias 7, largest normal 448, no infinities) and E5M2
 * (bias 15, largest normal 57344), as in the OCP OFP8 specification.  The
 * cast computes q = fp8(fp32(x) * scale): one IEEE fp32 multiply, then
 * round-to-nearest-even with saturation (values beyond the largest normal
 * and +-Inf become +-max; NaN becomes the canonical NaN 0x7F).  No
 * flush-to-zero.
 *
 * Conventions that hold for every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller, unless the
 *     argument says "host".  Matrices are dense and row-major; "rows x cols"
 *     data has element (i, j) at offset i*cols + j; the transpose of a
 *     rows x cols matrix is a cols x rows matrix.
 *   - The library allocates no device memory, never synchronises the stream
 *     or the device, and never reads device memory from the host, so every
 *     call can be recorded in a CUDA graph.  `stream` is a cudaStream_t
 *     (NULL = the legacy default stream).
 *   - `noop_flag` (nullable) is a device fp32 scalar read by the kernels at
 *     run time: when it is nonzero the call writes nothing at all (no data,
 *     transpose, amax, scale-inverse, dbias, history or scale).  This is how
 *     a captured graph skips a cached transpose [B].
 *   - `amax` is max-merged: the kernel stores max(*amax, max|x|), comparing
 *     IEEE magnitude bit patterns (NaN above Inf, so a NaN in x propagates).
 *     *amax must hold a non-negative value (normally 0, the cleared current
 *     slot of the amax history) before the call.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error code and launches nothing.  rows == 0 or
 *     cols == 0 returns CT_OK without a launch and writes nothing (its
 *     pointers are then not checked and may be NULL).  A failed launch returns
 *     CT_ERR_CUDA.  Any shape and alignment is accepted.  Shapes with rows
 *     a multiple of 16 and cols a multiple of 8, with 16-byte-aligned
 *     buffers, take a fast path: a persistent TMA-staged kernel for launches
 *     under 2048 tiles of 128x128, a direct-load kernel (256 threads per
 *     tile) from 2048 tiles on.  Other row counts with cols a multiple of 8
 *     and aligned buffers take the direct-load kernel.  With out 8-byte
 *     aligned and no dbias, a plain cast (ct_fp8_cast) of any other shape or
 *     x alignment runs over the rows * cols elements as one flat array, and
 *     so does a cast-transpose with rows not a multiple of 16, followed by an
 *     FP8 transpose of out into out_t.  Everything else takes a slower
 *     general kernel.  All give identical results.
 *   - Calls are thread-safe; the library keeps no per-call state.  The first
 *     call of an entry point on a device also sets its kernels' shared-memory
 *     limit (cudaFuncSetAttribute, once per device): make that first call
 *     outside stream capture, as one makes a warm-up call before capturing.
 *   - Kernels are launched as programmatic dependents of the previous kernel
 *     in the stream: they may be scheduled while it still runs, and read or
 *     write nothing before it has completed.  A cast kernel may only ask for
 *     its first tiles of x to be prefetched into L2 meanwhile, a hint that
 *     cannot return stale data.  fp8_cast_transpose_ex with CT_X_READY (and
 *     fp8_dbias_cast_transpose_ex with CT_DBIAS_X_READY) lets it load them,
 *     under that flag's precondition.
 */
#ifndef CAST_TRANSPOSE_GB300_H
#define CAST_TRANSPOSE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CT_E4M3 = 0,
    CT_E5M2 = 1
} ct_fp8_format;

/* Rule for the amax that sets the next scale (fp8_amax_and_scale_update_ex). */
typedef enum {
    CT_AMAX_MAX = 0,          /* maximum over the whole history window          */
    CT_AMAX_MOST_RECENT = 1   /* the amax of the step that just ran (row 0) only */
} ct_amax_algo;

typedef enum {
    CT_OK = 0,
    CT_ERR_NULL = 1,        /* a required pointer is NULL                      */
    CT_ERR_SHAPE = 2,       /* negative size, or a size the kernels cannot index */
    CT_ERR_ALIGN = 3,       /* buffer misaligned for its element type          */
    CT_ERR_FORMAT = 4,      /* fmt is not CT_E4M3 / CT_E5M2                    */
    CT_ERR_ARG = 5,         /* other invalid scalar (history length, margin)   */
    CT_ERR_ALIAS = 6,       /* an output overlaps an input or another output   */
    CT_ERR_WORKSPACE = 7,   /* workspace missing or too small                  */
    CT_ERR_CUDA = 8         /* a CUDA runtime call or launch failed            */
} ct_status;

/* Human-readable name of a ct_status value (static string, never NULL). */
const char* ct_status_string(int status);

/*
 * fp8_cast_transpose -- [A] cast_transpose(dy), [B] private scale-inverse.
 *
 *   x          bf16 [rows, cols] input (read only)
 *   scale      fp32 scalar: the scale to cast with
 *   amax       fp32 scalar, max-merged with max|x| (see conventions)
 *   scale_inv  fp32 scalar output: 1 / *scale (IEEE division), the FP8
 *              tensor's own scale-inverse; must not alias `scale`
 *   out        uint8 [rows, cols] output: FP8 codes of x * scale
 *   out_t      uint8 [cols, rows] output: the transpose of `out`
 *   fmt        CT_E4M3 or CT_E5M2
 *   noop_flag  nullable fp32 device scalar; nonzero -> nothing is written
 *
 * Outputs must not overlap the input or each other.  Errors: CT_ERR_NULL,
 * CT_ERR_SHAPE, CT_ERR_ALIGN (x not 2-byte aligned), CT_ERR_FORMAT,
 * CT_ERR_ALIAS, CT_ERR_CUDA.
 */
int fp8_cast_transpose(const void* x, int64_t rows, int64_t cols,
                       const float* scale, float* amax, float* scale_inv,
                       void* out, void* out_t, int fmt,
                       const float* noop_flag, void* stream);

/* Flags of fp8_cast_transpose_ex. */
typedef enum {
    /* The caller promises that no kernel that may still be running when this
     * call's kernel starts writes x: x was produced by a copy or a kernel the
     * stream has already waited for, and the kernel just before this call in
     * the stream does not write it (for example, it is this library's scale
     * update, which writes only fp32 scalars).  The call may then load its
     * first tiles of x before the preceding kernel completes.  Without the
     * flag nothing of x is read until that kernel has completed. */
    CT_X_READY = 1u
} ct_cast_flags;

/*
 * fp8_cast_transpose_ex -- fp8_cast_transpose with `flags`, a bitwise OR of
 * ct_cast_flags values.  The pages have no counterpart: the flag only moves
 * the moment x is first read (see CT_X_READY), never what is computed.
 * Errors: as fp8_cast_transpose, plus CT_ERR_ARG for an unknown flag bit.
 */
int fp8_cast_transpose_ex(const void* x, int64_t rows, int64_t cols,
                          const float* scale, float* amax, float* scale_inv,
                          void* out, void* out_t, int fmt,
                          const float* noop_flag, unsigned flags, void* stream);

/*
 * fp8_dbias_cast_transpose -- [A] DbiasCastTranspose.backward:
 * db = dy.sum(dim=0) next to cast_transpose(dy), in one pass over dy.
 *
 *   dy, scale, amax, scale_inv, out, out_t, fmt, noop_flag: as in
 *              fp8_cast_transpose, with dy in place of x
 *   dbias      fp32 [cols] output: column sums of the unscaled dy,
 *              accumulated in fp32 per 128-row tile and with compensated
 *              (Kahan) fp32 across tiles; deterministic (the summation order
 *              depends only on the shape)
 *   workspace  device scratch of at least
 *              fp8_dbias_cast_transpose_workspace_size(rows, cols) bytes,
 *              16-byte aligned; its contents on entry are ignored and on exit
 *              undefined; calls that overlap in time need separate workspaces
 *
 * Two kernels are launched on `stream` (the fused pass, then a small
 * column-sum finish).  Errors: as fp8_cast_transpose, plus CT_ERR_WORKSPACE.
 */
int fp8_dbias_cast_transpose(const void* dy, int64_t rows, int64_t cols,
                             const float* scale, float* amax, float* scale_inv,
                             void* out, void* out_t, float* dbias,
                             void* workspace, size_t workspace_bytes, int fmt,
                             const float* noop_flag, void* stream);

/* Bytes of workspace fp8_dbias_cast_transpose needs for a rows x cols dy
 * (0 when rows or cols is 0 or negative). */
size_t fp8_dbias_cast_transpose_workspace_size(int64_t rows, int64_t cols);

/* Element type of fp8_dbias_cast_transpose_ex's db output, optionally OR'd
 * with CT_DBIAS_X_READY. */
typedef enum {
    CT_DBIAS_FP32 = 0,   /* fp32, as fp8_dbias_cast_transpose                   */
    CT_DBIAS_BF16 = 1,   /* the same fp32 column sum, rounded to bf16 (nearest
                            even; NaN -> 0x7FFF), e.g. for a bf16 bias         */
    CT_DBIAS_X_READY = 0x100  /* the CT_X_READY promise for dy (see
                                 ct_cast_flags): the first tiles of dy may be
                                 loaded before the preceding kernel completes */
} ct_dbias_dtype;

/*
 * fp8_dbias_cast_transpose_ex -- fp8_dbias_cast_transpose with the db element
 * type as an argument ([A] DbiasCastTranspose.backward: db is the gradient of
 * the bias, which a bf16 model keeps in bf16).
 *
 *   dbias        [cols] output of type dbias_dtype, 4-byte (fp32) or 2-byte
 *                (bf16) aligned; must not overlap the other buffers
 *   dbias_dtype  CT_DBIAS_FP32 or CT_DBIAS_BF16, optionally OR'd with
 *                CT_DBIAS_X_READY (the caller's CT_X_READY promise for dy)
 *   (every other argument as in fp8_dbias_cast_transpose)
 *
 * Errors: as fp8_dbias_cast_transpose, plus CT_ERR_ARG for an unknown
 * dbias_dtype.
 */
int fp8_dbias_cast_transpose_ex(const void* dy, int64_t rows, int64_t cols,
                                const float* scale, float* amax, float* scale_inv,
                                void* out, void* out_t, void* dbias, int dbias_dtype,
                                void* workspace, size_t workspace_bytes, int fmt,
                                const float* noop_flag, void* stream);

/* One entry of a tensor list (host memory; the pointers inside are device
 * pointers with the meaning they have in fp8_cast_transpose). */
typedef struct {
    const void* x;
    int64_t rows;
    int64_t cols;
    const float* scale;
    float* amax;
    float* scale_inv;
    void* out;
    void* out_t;
} ct_tensor_desc;

/*
 * fp8_multi_cast_transpose -- cast-transpose of a list of tensors, each with
 * its own scale, amax and scale-inverse, in one launch ([B]: many
 * FP8 weight workspaces are refreshed every step; one launch instead of one
 * per tensor keeps the host overhead flat).
 *
 *   descs      HOST array of n descriptors, read during the call only
 *   n          number of descriptors (>= 0); lists longer than 64 tensors,
 *              and tensors that miss the fast path's shape/alignment rules,
 *              are split across further launches on the same stream
 *   fmt        one FP8 format for the whole list
 *   noop_flag  as above, for the whole list
 *
 * Every descriptor is validated before anything is launched.  Entries with
 * rows == 0 or cols == 0 are skipped.  Distinct entries must not share
 * outputs.  Errors: as fp8_cast_transpose (the first bad entry decides).
 */
int fp8_multi_cast_transpose(const ct_tensor_desc* descs, int n, int fmt,
                             const float* noop_flag, void* stream);

/*
 * fp8_multi_cast_transpose_ex -- fp8_multi_cast_transpose with one FP8
 * format per tensor (e.g. E4M3 weights and E5M2 gradients in one launch).
 *
 *   fmts       HOST array of n formats (CT_E4M3 / CT_E5M2), read during the
 *              call only; NULL is CT_ERR_NULL when n > 0
 *
 * Everything else as fp8_multi_cast_transpose.  The format is uniform over a
 * 128x128 tile, so the kernel branches once per tile.
 */
int fp8_multi_cast_transpose_ex(const ct_tensor_desc* descs, const int* fmts, int n,
                                const float* noop_flag, void* stream);

/*
 * fp8_amax_and_scale_update -- the delayed-scaling scale update kernel [B]
 * for n tensors, including the infinite-scale guard.
 *
 *   amax_history  fp32 [hist_len, n] row-major; row 0 holds the amaxes of the
 *                 step that just ran (written by the cast kernels)
 *   scale         fp32 [n], read and written
 *   scale_inv     fp32 [n], written: 1 / scale (the recipe's copy; tensors
 *                 cast earlier keep their own copy, [B])
 *   hist_len      L >= 1;  n >= 0;  margin in [0, 126];  fmt as above
 *
 * For each tensor i:
 *   a = max over the L history rows of column i (NaN propagates);
 *   s = (fp8_max / a) / 2^margin in fp32 (fp8_max = 448 or 57344);
 *   scale[i] = s unless a is not > 0, a is not finite, or s is not finite
 *   (the too-tiny-amax case), in which case scale[i] is left as it was;
 *   scale_inv[i] = 1 / scale[i];
 *   then the window slides: row r takes row r-1 for r = L-1 .. 1, and row 0
 *   is set to 0, ready for the next step's max-merge.
 * One launch.  Buffers must not overlap.  Errors: CT_ERR_NULL, CT_ERR_ARG,
 * CT_ERR_FORMAT, CT_ERR_ALIGN, CT_ERR_ALIAS, CT_ERR_CUDA.
 */
int fp8_amax_and_scale_update(float* amax_history, float* scale, float* scale_inv,
                              int hist_len, int n, int fmt, int margin,
                              const float* noop_flag, void* stream);

/*
 * fp8_amax_and_scale_update_ex -- fp8_amax_and_scale_update with a choice of
 * the amax rule: CT_AMAX_MAX (the window maximum, as fp8_amax_and_scale_update)
 * or CT_AMAX_MOST_RECENT (row 0 alone: the scale follows the latest amax, the
 * older rows only ride along in the window).  Guard, scale_inv and the window
 * slide are the same.  Errors: as fp8_amax_and_scale_update; an unknown
 * amax_algo is CT_ERR_ARG.
 */
int fp8_amax_and_scale_update_ex(float* amax_history, float* scale, float* scale_inv,
                                 int hist_len, int n, int fmt, int margin, int amax_algo,
                                 const float* noop_flag, void* stream);

/*
 * Deferred scale updates -- a run of casts that share one amax-history
 * column, each of which would be followed by fp8_amax_and_scale_update_ex
 * (the delayed-scaling update of [B], run after every refresh of a weight's
 * FP8 copy).  The updates between the casts
 * sit on the stream's critical path: each cast has to wait for the update
 * before it.  Here cast k of the run instead derives the scale that the k
 * updates before it would have produced, from the history and the scale as
 * they stood before the run and from the amaxes of casts 0 .. k-1, and one
 * fp8_amax_and_scale_update_pending call after the run applies all of them.
 * Every cast's output and scale_inv, and the history, scale and scale_inv
 * after the run, are bit for bit those of the sequence
 *     for k in 0 .. K-1: fp8_cast_transpose_ex(x_k, ..., amax = history row 0
 *                            of the column, ...);
 *                        fp8_amax_and_scale_update_ex(...);
 * (with the same hist_len, fmt, margin and amax_algo).
 *
 * fp8_cast_transpose_pending -- cast k (0-based) of such a run.
 *
 *   x, rows, cols, scale_inv, out, out_t, fmt, noop_flag, flags
 *                 as fp8_cast_transpose_ex; scale_inv receives 1 / the derived
 *                 scale
 *   amax_history  fp32 [hist_len, n], read only: the history before the run
 *   scale         fp32 [n], read only: the scales before the run
 *   pending       fp32 [K, n] (K: the run's length), zero before cast 0 (and
 *                 left zero by fp8_amax_and_scale_update_pending); rows 0 .. k-1
 *                 are read (the amaxes of the earlier casts), row k is
 *                 max-merged with max|x| (as `amax` of fp8_cast_transpose)
 *   col           the history column, 0 <= col < n
 *   k             0 <= k < min(32, hist_len)
 *   hist_len, margin, amax_algo
 *                 those of the deferred updates (fp8_amax_and_scale_update_ex);
 *                 1 <= hist_len <= 1024; fp8_max is fmt's
 *
 * The scale: update j (0-based) sees the window c_j, c_{j-1}, .., c_0,
 * history rows 1 .. hist_len-1-j, where c_j is pending row j (c_0 also
 * max-merged with history row 0, the slot cast 0 would have merged into); the
 * cast uses the guarded candidate (fp8_max / a_j) / 2^margin of the latest
 * update j < k whose guard passes, else the scale before the run.  Every CTA
 * derives it with one warp after the dependency wait, in the same round trip
 * as the scale load it replaces.  The history, scale and pending rows 0 .. k-1
 * must not be written by a kernel that may still be running when this call's
 * kernel starts.  Outputs must not overlap x or each other, nor the history,
 * the scale or pending rows 0 .. k-1.  Errors: as fp8_cast_transpose_ex, plus
 * CT_ERR_ARG (hist_len, n, col, k, margin, amax_algo).
 */
int fp8_cast_transpose_pending(const void* x, int64_t rows, int64_t cols,
                               const float* amax_history, const float* scale, float* pending,
                               int hist_len, int n, int col, int k, int margin, int amax_algo,
                               float* scale_inv, void* out, void* out_t, int fmt,
                               const float* noop_flag, unsigned flags, void* stream);

/*
 * fp8_amax_and_scale_update_pending -- the `run` updates deferred by a run of
 * fp8_cast_transpose_pending calls, applied to all n columns at once.
 *
 *   amax_history  fp32 [hist_len, n]: on return, as `run` calls of
 *                 fp8_amax_and_scale_update_ex would leave it: row 0 = 0,
 *                 rows 1 .. run = c_{run-1} .. c_0, the older rows slid down
 *                 by `run`
 *   scale, scale_inv  fp32 [n]: the scale after the last update, 1 / scale
 *   pending       fp32 [run, n]: read, then set to 0
 *   run           1 <= run <= min(32, hist_len);  1 <= hist_len <= 1024
 *   fmt, margin, amax_algo, noop_flag  as fp8_amax_and_scale_update_ex
 *
 * One launch, one warp per column, every read before any write.  Buffers
 * must not overlap.  Errors: CT_ERR_NULL, CT_ERR_ARG, CT_ERR_FORMAT,
 * CT_ERR_ALIGN, CT_ERR_ALIAS, CT_ERR_CUDA.
 */
int fp8_amax_and_scale_update_pending(float* amax_history, float* scale, float* scale_inv,
                                      float* pending, int hist_len, int n, int run, int fmt,
                                      int margin, int amax_algo, const float* noop_flag,
                                      void* stream);

/*
 * fp8_transpose -- byte transpose of an existing FP8 tensor: the lazy
 * transpose-cache fill of [B] (transpose_2d(cache=True)), skippable through
 * the noop flag inside a captured graph.
 *
 *   in         uint8 [rows, cols]
 *   out        uint8 [cols, rows], must not overlap `in`
 */
int fp8_transpose(const void* in, int64_t rows, int64_t cols, void* out,
                  const float* noop_flag, void* stream);

/*
 * fp8_cast -- the cast without the transpose (Float8Tensor.to_float8 in the
 * FP8Linear example of [A]): out, amax and scale_inv as in
 * fp8_cast_transpose, no transposed output.
 */
int fp8_cast(const void* x, int64_t rows, int64_t cols, const float* scale,
             float* amax, float* scale_inv, void* out, int fmt,
             const float* noop_flag, void* stream);

/*
 * fp8_dbias_cast_transpose_noalloc -- fp8_dbias_cast_transpose without a
 * caller-provided workspace.  The pages have no counterpart to this entry
 * point: it exists for callers that cannot allocate device memory at the
 * point of the call -- code called from inside an allocator or a memory pool
 * (where allocating again would recurse or deadlock), and runtimes that
 * reserve all device memory up front and hand none out later.
 *
 *   dy, scale, amax, scale_inv, out, out_t, dbias, fmt, noop_flag, stream:
 *              exactly as in fp8_dbias_cast_transpose
 *
 * Scratch: a fixed 4 MiB array inside the library's device memory (every GPU
 * that loads the library holds it until the process exits).  The call itself
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  Limit: fp8_dbias_cast_transpose_workspace_size(rows, cols) <=
 * 4 MiB, i.e. ceil(rows/128) * cols <= 1,048,576 (8192 x 16384, say); larger
 * shapes return CT_ERR_WORKSPACE without launching anything.  The first call
 * on each device looks up the array's device address (once, with that device
 * current) and keeps it for the life of the process, so make that first call
 * before any stream capture, and do not call it again on a device after
 * cudaDeviceReset.  All calls share the one array, which keeps the last
 * call's contents; nothing in it has to start at zero (each call reads back
 * only the partial sums it wrote itself), but calls whose kernels overlap on
 * the GPU (different streams, or several threads) race on it: run them one
 * after another.
 * Errors: as fp8_dbias_cast_transpose, plus CT_ERR_WORKSPACE for too large
 * a shape and CT_ERR_CUDA if the address lookup fails.
 */
int fp8_dbias_cast_transpose_noalloc(const void* dy, int64_t rows, int64_t cols,
                                     const float* scale, float* amax, float* scale_inv,
                                     void* out, void* out_t, float* dbias, int fmt,
                                     const float* noop_flag, void* stream);

/*
 * ct_fp8_convert_f32 -- the FP8 conversion step of the cast kernels applied
 * to fp32 values as given: out[i] = fp8(in[i]), round to nearest even, values
 * beyond the largest normal and +-Inf saturate to +-max, NaN gives 0x7F, no
 * flush-to-zero.  It is the same device routine every cast kernel applies to
 * the product x * scale ("[PyTorch] cuda graph support": cast_transpose(dy);
 * FP8 formats as in the OCP OFP8 specification), exposed without the scale,
 * amax and layout around it so that the conversion itself can be checked
 * against a reference over any set of fp32 values (every bit pattern, say).
 *
 *   in    fp32 [n], 4-byte aligned (read only)
 *   n     number of values (>= 0; 0 returns CT_OK and launches nothing)
 *   fmt   CT_E4M3 or CT_E5M2
 *   out   uint8 [n] output, any alignment; must not overlap `in`
 *
 * One launch on `stream`.  Errors: CT_ERR_NULL, CT_ERR_SHAPE (n < 0),
 * CT_ERR_ALIGN, CT_ERR_FORMAT, CT_ERR_ALIAS, CT_ERR_CUDA.
 */
int ct_fp8_convert_f32(const float* in, int64_t n, int fmt, void* out, void* stream);

/*
 * ct_device_error -- diagnostic word of the current device.  Kernels that
 * wait on an mbarrier give up after a bounded time (about two seconds)
 * instead of hanging, set a bit here and return early; in a correct run it
 * stays 0.  Reads (synchronously) and optionally clears the word.
 * Bits: 1 = a tile-load wait timed out; 2 = ct_selftest_bounded_wait ran
 * (its wait always times out).
 */
int ct_device_error(unsigned int* value_out, int clear);

/*
 * ct_selftest_bounded_wait -- exercises the timeout path of the kernels'
 * bounded waits without any fault: one block waits `limit_us` microseconds
 * (1 .. 1,000,000) on a barrier that nothing completes, then sets bit 2 of
 * the diagnostic word and returns; the context stays usable.  For tests and
 * health checks.  Errors: CT_ERR_ARG, CT_ERR_CUDA.
 */
int ct_selftest_bounded_wait(unsigned int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CAST_TRANSPOSE_GB300_H */
