// ct_noalloc.cu -- fp8_dbias_cast_transpose for callers that cannot allocate.
//
// fp8_dbias_cast_transpose needs a device workspace for its per-tile column
// partial sums, and the caller provides it.  Some callers have no way to get
// one where they call it: code called from inside a memory allocator or a
// memory-pool callback (where allocating again would recurse or deadlock),
// and runtimes that reserve all device memory up front and hand out nothing
// more.  This entry point serves them: its scratch is a fixed array in the
// library's own device memory, reserved when the library is loaded on a GPU
// and held until the process exits, so the call itself allocates nothing.
// The array's address is looked up once per device and kept; after a
// cudaDeviceReset the module is loaded again elsewhere, so the entry point
// is not to be used on that device again.
#include "../../include/cast_transpose.h"
#include "ct_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// 4 MiB: enough for the per-128-row-tile fp32 partials of up to 1,048,576
// (row-tile, column) pairs, e.g. an 8192 x 16384 or a 32768 x 4096 dy.
constexpr size_t kScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_dbias_scratch[kScratchBytes];

// Device address of g_dbias_scratch on each device.  The array's name in
// host code is only a host-side handle, so the address is fetched once per
// device with that device current and cached.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

int scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dbias_scratch) != cudaSuccess || p == nullptr)
            return CT_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CT_OK;
}

}  // namespace

extern "C" int fp8_dbias_cast_transpose_noalloc(const void* dy, int64_t rows, int64_t cols,
                                                const float* scale, float* amax,
                                                float* scale_inv, void* out, void* out_t,
                                                float* dbias, int fmt, const float* noop_flag,
                                                void* stream) {
    if (fmt != CT_E4M3 && fmt != CT_E5M2) return CT_ERR_FORMAT;
    if (rows < 0 || cols < 0) return CT_ERR_SHAPE;
    if (rows == 0 || cols == 0) return CT_OK;
    // Every partial the finish step reads is written by this call's first
    // kernel, so the shared scratch needs no clearing between calls.
    if (fp8_dbias_cast_transpose_workspace_size(rows, cols) > kScratchBytes)
        return CT_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = scratch_on_current_device(&scratch);
    if (st != CT_OK) return st;
    return fp8_dbias_cast_transpose(dy, rows, cols, scale, amax, scale_inv, out, out_t, dbias,
                                    scratch, kScratchBytes, fmt, noop_flag, stream);
}
