// y = A^T x without a caller-supplied workspace.
//
// Some callers cannot allocate device memory: a host process whose device
// memory is owned entirely by its own allocator and refuses outside
// allocations, or a plug-in that is handed only the input and output buffers
// of one operation.  ds_gemv_transposed needs scratch memory for its split
// reduction (per-band counters and partial sums), which such a caller cannot
// provide.  This entry point takes that scratch from a fixed area compiled
// into the library instead: every GPU that loads the library holds
// kNoAllocScratchBytes of device memory for it until the process exits.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB

// The scratch area (zero at load).  Byte 0 is the error word, as in every
// workspace; the band counters and partial sums follow.  In host code this
// name is only a stand-in for the device variable: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[64] = {nullptr};

// Device address of the scratch area on the current device, looked up once
// per device (that first lookup is the set-up the header describes) and kept
// for the life of the process.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" DS_API size_t ds_gemv_transposed_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" DS_API int ds_gemv_transposed_noalloc(const void *A, int64_t a_len, int a_dtype, const float *x,
                                                 int64_t x_len, int64_t rows, int64_t cols, float *y, int64_t y_len,
                                                 ds_stream_t stream) {
    // the same shape checks as ds_gemv_transposed, before anything else
    if (rows < 1 || cols < 1) return DS_EMPTY_DIMENSION;
    if (rows > DS_MAX_DIM || cols > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (a_dtype != DS_F32 && a_dtype != DS_BF16) return DS_BAD_DTYPE;
    if (a_len != rows * cols) return DS_GEMV_A_LENGTH_MISMATCH;
    if (x_len != rows) return DS_GEMV_X_LENGTH_MISMATCH;
    if (y_len != cols) return DS_A_LENGTH_MISMATCH;
    if (!A || !x || !y) return DS_BAD_ARGUMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // a matrix the streamed kernel cannot take runs the plain-load kernel,
    // which uses no scratch at all
    if (!ds::gemv_t_uses_workspace(A, cols, a_dtype)) return ds::gemv_transposed_run(A, a_dtype, x, rows, cols, y,
                                                                                      nullptr, s);
    const size_t need = ds_gemv_workspace_bytes(rows, cols, a_dtype);
    if (need == 0 || need > kNoAllocScratchBytes) return DS_DIMENSION_TOO_LARGE;  // beyond the built-in area
    char *scratch = static_cast<char *>(scratch_on_current_device());
    if (!scratch) return DS_CUDA_ERROR;
    // The area keeps whatever the previous call left: the band counters must
    // start at zero.  The error word (byte 0) is left alone so that it keeps
    // any bit a kernel set until ds_gemv_transposed_noalloc_error reads it.
    const size_t zero_from = ds::kWsHeader, zero_to = ds::gemv_t_zeroed_bytes(cols, a_dtype);
    if (cudaMemsetAsync(scratch + zero_from, 0, zero_to - zero_from, s) != cudaSuccess) return DS_CUDA_ERROR;
    return ds::gemv_transposed_run(A, a_dtype, x, rows, cols, y, scratch, s);
}

extern "C" DS_API int ds_gemv_transposed_noalloc_error(int32_t *host_word, ds_stream_t stream) {
    if (!host_word) return DS_BAD_ARGUMENT;
    void *scratch = scratch_on_current_device();
    if (!scratch) return DS_CUDA_ERROR;
    return ds_workspace_error(scratch, host_word, stream);
}
