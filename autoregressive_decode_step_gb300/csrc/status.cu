// Status vocabulary, the contract's shape check, workspace error words and
// device queries.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ds {

int sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace ds

extern "C" DS_API const char *ds_status_name(int code) {
    switch (code) {
        case DS_OK: return "ds_ok";
        case DS_EMPTY_DIMENSION: return "ds_empty_dimension";
        case DS_A_LENGTH_MISMATCH: return "ds_a_length_mismatch";
        case DS_B_LENGTH_MISMATCH: return "ds_b_length_mismatch";
        case DS_DIMENSION_TOO_LARGE: return "ds_dimension_too_large";
        case DS_CACHE_LENGTH_MISMATCH: return "ds_cache_length_mismatch";
        case DS_NEW_LENGTH_MISMATCH: return "ds_new_length_mismatch";
        case DS_LOGITS_LENGTH_MISMATCH: return "ds_logits_length_mismatch";
        case DS_GEMV_A_LENGTH_MISMATCH: return "ds_gemv_a_length_mismatch";
        case DS_GEMV_X_LENGTH_MISMATCH: return "ds_gemv_x_length_mismatch";
        case DS_CACHE_CAPACITY_EXCEEDED: return "ds_cache_capacity_exceeded";
        case DS_BAD_DTYPE: return "ds_bad_dtype";
        case DS_CUDA_ERROR: return "ds_cuda_error";
        case DS_WORKSPACE_TOO_SMALL: return "ds_workspace_too_small";
        case DS_BAD_SAMPLING_PARAM: return "ds_bad_sampling_param";
        case DS_TOKEN_OUT_OF_RANGE: return "ds_token_out_of_range";
        case DS_BAD_ARGUMENT: return "ds_bad_argument";
        default: return "ds_code_out_of_range";
    }
}

extern "C" DS_API int ds_residual_dims_check(int64_t n, int64_t a_len, int64_t b_len) {
    if (n < 1) return DS_EMPTY_DIMENSION;
    if (n > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (a_len != n) return DS_A_LENGTH_MISMATCH;
    if (b_len != n) return DS_B_LENGTH_MISMATCH;
    return DS_OK;
}

extern "C" DS_API int ds_workspace_error(void *workspace, int32_t *host_word, ds_stream_t stream) {
    if (!workspace || !host_word) return DS_BAD_ARGUMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_word, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DS_CUDA_ERROR;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess) return DS_CUDA_ERROR;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DS_CUDA_ERROR;
    return DS_OK;
}

extern "C" DS_API int ds_device_sm_count(void) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 0;
    }
    return ds::sm_count();
}
