// Decode glue: residual add, add+RMSNorm, SiLU-gate, RoPE, reserved-capacity
// KV append, the embedding gather and the model's RoPE table.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace ds {

// out[i] = a[i] + b[i] ("LLM inference kernels", "Residual add").
__global__ void residual_add_kernel(const float *a, const float *b, float *out, long long n) {
    grid_dependency_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = a[i] + b[i];
}

// residual += x; h = residual * (mean(residual^2) + eps)^-1/2 * w, the square
// sum in fp32 ("decode-ops", "Usage" and "API — Method").  One CTA.
template <typename WT>
__global__ void add_rmsnorm_kernel(float *residual, const float *x, const WT *w, float eps, float *h, long long n) {
    __shared__ float red[32];
    __shared__ float s_scale;
    grid_dependency_wait();
    float ss = 0.0f;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
        float r = residual[i];
        if (x) {
            r = r + x[i];
            residual[i] = r;
        }
        ss = fmaf(r, r, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        s_scale = 1.0f / sqrtf(tot / (float)n + eps);
    }
    __syncthreads();
    const float s = s_scale;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) h[i] = residual[i] * s * to_f32(w[i]);
}

// out[i] = silu(gate[i]) * up[i] ("decode-ops", "Usage": silu_mul).
__global__ void silu_mul_kernel(const float *gate, const float *up, float *out, long long n) {
    grid_dependency_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float z = gate[i];
        out[i] = z / (1.0f + expf(-z)) * up[i];
    }
}

// The (cos, sin) of every rotation pair of one ds_rope call: the angles
// pos * base^(-2p/hd) are formed in fp64 on the host once per call
// ("decode-ops", "API — Method": the angle pairs are built once and reused
// for every head), rounded to fp32, and passed by value.
template <int P>
struct RopeAngles {
    float c[P], s[P];
};

// One thread per rotation pair of q (then k), the rotation in fp32.
template <int P>
__global__ void rope_kernel(float *q, int n_qh, float *k, int n_kh, int hd, int layout, const RopeAngles<P> ang) {
    grid_dependency_wait();
    const int half = hd >> 1;
    const int pair_id = blockIdx.x * blockDim.x + threadIdx.x;
    const int total = (n_qh + n_kh) * half;
    if (pair_id >= total) return;
    const int head = pair_id / half, pr = pair_id % half;
    float *v = head < n_qh ? q + (long long)head * hd : k + (long long)(head - n_qh) * hd;
    const float c = ang.c[pr], s = ang.s[pr];
    const int ia = layout == DS_ROPE_INTERLEAVED ? 2 * pr : pr;
    const int ib = layout == DS_ROPE_INTERLEAVED ? 2 * pr + 1 : pr + half;
    const float a = v[ia], b = v[ib];
    v[ia] = a * c - b * s;
    v[ib] = a * s + b * c;
}

template <int P>
static cudaError_t launch_rope(float *q, int n_qh, float *k, int n_kh, int64_t pos, int hd, double base, int layout,
                               cudaStream_t stream) {
    RopeAngles<P> ang;
    const int half = hd / 2;
    for (int p = 0; p < P; ++p) {
        ang.c[p] = 1.0f;
        ang.s[p] = 0.0f;
        if (p < half) {
            const double theta = (double)pos * std::pow(base, -(double)(2 * p) / (double)hd);
            ang.c[p] = (float)std::cos(theta);
            ang.s[p] = (float)std::sin(theta);
        }
    }
    const int pairs = (n_qh + n_kh) * half;
    return launch_ex(rope_kernel<P>, dim3((pairs + 255) / 256), dim3(256), 0, stream, false, q, n_qh, k, n_kh, hd,
                     layout, ang);
}

// cos/sin of pos * base^(-2p/hd) for every position row and pair, fp64
// angles rounded to fp32 once (the shared RoPE table of "LLM inference
// kernels", "The hot loop doesn't call kv_cache_append_flat").
__global__ void rope_table_kernel(float *cos_t, float *sin_t, int rows, int hd, double base, RopeScaling sc) {
    const int half = hd >> 1;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)rows * half) return;
    const int pos = (int)(i / half), pr = (int)(i % half);
    double f = pow(base, -(double)(2 * pr) / (double)hd);
    if (sc.factor != 0.0) {
        // long-context scaling by the pair's wavelength (Llama 3.1's remap):
        // fast pairs keep f, slow pairs turn factor times slower, the band
        // between blends the two linearly in orig_max_pos / wavelength
        const double w = 6.283185307179586476925286766559 / f;
        if (w > sc.orig_max_pos / sc.low_freq_factor) {
            f = f / sc.factor;
        } else if (!(w < sc.orig_max_pos / sc.high_freq_factor)) {
            const double s = (sc.orig_max_pos / w - sc.low_freq_factor) / (sc.high_freq_factor - sc.low_freq_factor);
            f = (1.0 - s) * (f / sc.factor) + s * f;
        }
    }
    const double theta = (double)pos * f;
    cos_t[i] = (float)cos(theta);
    sin_t[i] = (float)sin(theta);
}

// cache[cache_len + i] = new_vals[i] in the cache dtype.
__global__ void kv_append_kernel(void *cache, int dtype, long long cache_len, const float *nv, long long n_new) {
    grid_dependency_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_new; i += stride)
        store_as(cache, cache_len + i, dtype, nv[i]);
}

// h[s][:] = x[s][:] * (mean(x[s]^2) + eps)^-1/2 * w, square sum in fp32
// ("The forward pass end to end", "The code": rmsnorm), one CTA per row: the
// normalised input of a batched projection, written for the tensor cores as
// the bf16 pair hi (at h) + lo (lo_off elements further; 0: hi only).
__global__ void rmsnorm_rows_bf16_kernel(const float *x, const float *w, float eps, __nv_bfloat16 *h, int d,
                                         long long lo_off) {
    __shared__ float red[32];
    __shared__ float s_scale;
    allow_dependent_launch();
    grid_dependency_wait();
    const float *xr = x + (long long)blockIdx.x * d;
    float ss = 0.0f;
    if ((d & 3) == 0) {  // 16-byte loads, several in flight per thread
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
#pragma unroll 4
        for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
            const float4 v = x4[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
    } else {
        for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
        s_scale = 1.0f / sqrtf(tot / (float)d + eps);
    }
    __syncthreads();
    const float sc = s_scale;
    __nv_bfloat16 *hr = h + (long long)blockIdx.x * d;
#pragma unroll 4
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const float v = xr[i] * sc * w[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        hr[i] = hi;
        if (lo_off) hr[i + lo_off] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

cudaError_t launch_rmsnorm_rows_bf16(const float *x, const float *w, float eps, void *h, long long lo_off,
                                     int n_rows, int d, cudaStream_t stream, bool pdl) {
    return launch_ex(rmsnorm_rows_bf16_kernel, dim3(n_rows), dim3(256), 0, stream, pdl, x, w, eps,
                     static_cast<__nv_bfloat16 *>(h), d, lo_off);
}

// x[s][:] = emb[tokens[s]][:] widened to fp32; a token outside [0, vocab)
// is clamped and flagged.  grid.y = sequence.
template <typename WT>
__global__ void embed_kernel(const WT *emb, int vocab, int d, const int *tokens, float *x, int *err) {
    allow_dependent_launch();
    grid_dependency_wait();
    const int s = blockIdx.y;
    int tok = tokens[s];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, DS_ERR_TOKEN_RANGE);
        tok = min(max(tok, 0), vocab - 1);
    }
    const WT *row = emb + (long long)tok * d;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x)
        x[(long long)s * d + i] = to_f32(row[i]);
}

cudaError_t launch_embed(const void *emb, int w_dtype, int vocab, int d, const int *tokens, float *x, int *err,
                         int n_seqs, cudaStream_t stream, bool pdl) {
    const dim3 grid((d + 255) / 256, n_seqs);
    if (w_dtype == DS_BF16)
        return launch_ex(embed_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream, pdl,
                         static_cast<const __nv_bfloat16 *>(emb), vocab, d, tokens, x, err);
    return launch_ex(embed_kernel<float>, grid, dim3(256), 0, stream, pdl, static_cast<const float *>(emb), vocab, d,
                     tokens, x, err);
}

// Rows of a prompt chunk: row j is the token at position pos0 + j of
// sequence seq.
__global__ void chunk_rows_kernel(int *pos, int *row_seq, int pos0, int seq, int n) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < n) {
        pos[j] = pos0 + j;
        row_seq[j] = seq;
    }
}

cudaError_t launch_chunk_rows(int *pos, int *row_seq, int pos0, int seq, int n, cudaStream_t stream) {
    return launch_ex(chunk_rows_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, false, pos, row_seq, pos0, seq,
                     n);
}

cudaError_t launch_rope_table(float *cos_t, float *sin_t, int rows, int hd, double base, RopeScaling sc,
                              cudaStream_t stream) {
    const long long n = (long long)rows * (hd / 2);
    const int blocks = (int)((n + 255) / 256);
    return launch_ex(rope_table_kernel, dim3(blocks), dim3(256), 0, stream, false, cos_t, sin_t, rows, hd, base,
                     sc);
}

static int blocks_for(long long n, int threads) {
    long long b = (n + threads - 1) / threads;
    const long long cap = 8LL * std::max(1, sm_count());
    return (int)std::max(1LL, std::min(b, cap));
}

}  // namespace ds

using namespace ds;

static int dims_ok(int64_t n) {
    if (n < 1) return DS_EMPTY_DIMENSION;
    if (n > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    return DS_OK;
}

extern "C" DS_API int ds_residual_add(const float *a, int64_t a_len, const float *b, int64_t b_len, float *out,
                                      int64_t n, ds_stream_t stream) {
    int st = ds_residual_dims_check(n, a_len, b_len);
    if (st != DS_OK) return st;
    if (!a || !b || !out) return DS_BAD_ARGUMENT;
    cudaError_t e = launch_ex(residual_add_kernel, dim3(blocks_for(n, 256)), dim3(256), 0,
                              reinterpret_cast<cudaStream_t>(stream), false, a, b, out, (long long)n);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API int ds_add_rmsnorm(float *residual, int64_t residual_len, const float *x, int64_t x_len,
                                     const void *w, int64_t w_len, int w_dtype, float eps, float *h, int64_t h_len,
                                     int64_t n, ds_stream_t stream) {
    int st = dims_ok(n);
    if (st != DS_OK) return st;
    if (residual_len != n) return DS_A_LENGTH_MISMATCH;
    if (x && x_len != n) return DS_B_LENGTH_MISMATCH;
    if (w_len != n || h_len != n) return DS_A_LENGTH_MISMATCH;
    if (w_dtype != DS_F32 && w_dtype != DS_BF16) return DS_BAD_DTYPE;
    if (!residual || !w || !h || !(eps >= 0.0f)) return DS_BAD_ARGUMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (w_dtype == DS_BF16)
        e = launch_ex(add_rmsnorm_kernel<__nv_bfloat16>, dim3(1), dim3(1024), 0, s, false, residual, x,
                      static_cast<const __nv_bfloat16 *>(w), eps, h, (long long)n);
    else
        e = launch_ex(add_rmsnorm_kernel<float>, dim3(1), dim3(1024), 0, s, false, residual, x,
                      static_cast<const float *>(w), eps, h, (long long)n);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API int ds_silu_mul(const float *gate, int64_t gate_len, const float *up, int64_t up_len, float *out,
                                  int64_t n, ds_stream_t stream) {
    int st = ds_residual_dims_check(n, gate_len, up_len);
    if (st != DS_OK) return st;
    if (!gate || !up || !out) return DS_BAD_ARGUMENT;
    cudaError_t e = launch_ex(silu_mul_kernel, dim3(blocks_for(n, 256)), dim3(256), 0,
                              reinterpret_cast<cudaStream_t>(stream), false, gate, up, out, (long long)n);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API int ds_rope(float *q, int64_t q_len, float *k, int64_t k_len, int64_t pos, int n_qh, int n_kh,
                              int head_dim, double base, int layout, ds_stream_t stream) {
    if (n_qh < 1 || head_dim < 1 || n_kh < 0) return DS_EMPTY_DIMENSION;
    if ((int64_t)n_qh * head_dim > DS_MAX_DIM || (int64_t)n_kh * head_dim > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (q_len != (int64_t)n_qh * head_dim) return DS_A_LENGTH_MISMATCH;
    if (n_kh > 0 && k_len != (int64_t)n_kh * head_dim) return DS_B_LENGTH_MISMATCH;
    if (layout != DS_ROPE_HALF_SPLIT && layout != DS_ROPE_INTERLEAVED) return DS_BAD_DTYPE;
    if (head_dim % 2 || head_dim > 1024 || !q || (n_kh > 0 && !k) || !(base > 0.0)) return DS_BAD_ARGUMENT;
    if (pos < 0 || pos > DS_MAX_DIM) return DS_CACHE_LENGTH_MISMATCH;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the angle table rides in the launch's parameters: 512 bytes up to
    // head_dim 128, 4 KB up to head_dim 1024
    const cudaError_t e = head_dim <= 128 ? launch_rope<64>(q, n_qh, k, n_kh, pos, head_dim, base, layout, s)
                                          : launch_rope<512>(q, n_qh, k, n_kh, pos, head_dim, base, layout, s);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API int ds_kv_cache_append(void *cache, int cache_dtype, int64_t capacity, int64_t cache_len,
                                         const float *new_vals, int64_t new_len, int64_t n_new, ds_stream_t stream) {
    if (n_new < 1 || capacity < 1) return DS_EMPTY_DIMENSION;
    if (n_new > DS_MAX_DIM || capacity > DS_MAX_DIM || cache_len > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (cache_len < 0) return DS_CACHE_LENGTH_MISMATCH;
    if (new_len != n_new) return DS_NEW_LENGTH_MISMATCH;
    if (cache_len + n_new > capacity) return DS_CACHE_CAPACITY_EXCEEDED;
    if (cache_dtype != DS_F32 && cache_dtype != DS_BF16) return DS_BAD_DTYPE;
    if (!cache || !new_vals) return DS_BAD_ARGUMENT;
    cudaError_t e = launch_ex(kv_append_kernel, dim3(blocks_for(n_new, 256)), dim3(256), 0,
                              reinterpret_cast<cudaStream_t>(stream), false, cache, cache_dtype, (long long)cache_len,
                              new_vals, (long long)n_new);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}
