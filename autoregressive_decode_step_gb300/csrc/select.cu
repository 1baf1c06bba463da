// Picking the next token: full-vocabulary greedy argmax and the
// temperature / top-k / top-p sampler.
//
// Argmax ("LLM inference kernels", "KV-cache growth and greedy argmax";
// "decode-ops", "Correctness"): blocks scan contiguous slices of a row, the
// last block of the row (an atomic counter) reduces their candidates.  The
// ranking — NaN above every number, equal values to the lower index — is a
// total order, so the result does not depend on reduction order.
//
// Sampler ("decode-ops", "API — Method"): one CTA per row, no heap and no
// global sort.  The top_k-th largest scaled logit is found by a 4-pass radix
// select over order-preserving 32-bit keys (per-warp histograms, warp-
// aggregated increments); the survivors — every key above the threshold and
// the lowest-index keys equal to it — are bitonic-sorted into (key desc,
// index asc) order, the order the page's heap pops them in.  Softmax, top-p
// and the inverse CDF then run in fp32 in exactly the sequence the header
// documents.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kAmThreads = 256;

__device__ __forceinline__ void block_best(float &bv, int &bi, float *sv, int *si) {
    const int t = threadIdx.x;
    sv[t] = bv;
    si[t] = bi;
    __syncthreads();
    for (int s = blockDim.x >> 1; s > 0; s >>= 1) {
        if (t < s && ranks_above(sv[t + s], si[t + s], sv[t], si[t])) {
            sv[t] = sv[t + s];
            si[t] = si[t + s];
        }
        __syncthreads();
    }
    bv = sv[0];
    bi = si[0];
}

__global__ void __launch_bounds__(kAmThreads) argmax_kernel(const __grid_constant__ ArgmaxArgs p) {
    __shared__ float sv[kAmThreads];
    __shared__ int si[kAmThreads];
    __shared__ int s_last;
    allow_dependent_launch();
    grid_dependency_wait();
    const int row = blockIdx.y, b = blockIdx.x, B = gridDim.x;
    const float *l = p.logits + (long long)row * p.n;
    const long long i0 = p.n * b / B, i1 = p.n * (b + 1) / B;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (long long i = i0 + threadIdx.x; i < i1; i += kAmThreads) {
        const float v = l[i];
        if (ranks_above(v, (int)i, bv, bi)) {
            bv = v;
            bi = (int)i;
        }
    }
    block_best(bv, bi, sv, si);
    if (threadIdx.x == 0) {
        p.part_val[(long long)row * B + b] = bv;
        p.part_idx[(long long)row * B + b] = bi;
        __threadfence();
        s_last = atomicAdd(&p.counters[row], 1) == B - 1;
    }
    __syncthreads();
    if (!s_last || threadIdx.x != 0) return;
    __threadfence();
    bv = __ldcg(&p.part_val[(long long)row * B]);
    bi = __ldcg(&p.part_idx[(long long)row * B]);
    for (int j = 1; j < B; ++j) {
        const float v = __ldcg(&p.part_val[(long long)row * B + j]);
        const int ix = __ldcg(&p.part_idx[(long long)row * B + j]);
        if (ranks_above(v, ix, bv, bi)) {
            bv = v;
            bi = ix;
        }
    }
    p.counters[row] = 0;
    p.ids[row] = bi;
    if (p.max_logit) p.max_logit[row] = bv;
    if (p.tokens_adv) p.tokens_adv[row] = bi;
    if (p.pos_adv) p.pos_adv[row] += 1;
}

int argmax_blocks_per_row(long long n) {
    long long b = (n + 4095) / 4096;
    return (int)std::max(1LL, std::min(b, 64LL));
}

cudaError_t launch_argmax(const ArgmaxArgs &a, cudaStream_t stream, bool pdl) {
    return launch_ex(argmax_kernel, dim3(a.blocks_per_row, a.n_rows), dim3(kAmThreads), 0, stream, pdl, a);
}

// ------------------------------------------------------------------ sampler
constexpr int kSmThreads = 1024;
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kSmMaxK = DS_SAMPLE_MAX_TOP_K;
constexpr size_t kSmSmem = (size_t)kSmWarps * 256 * 4 + (size_t)kSmMaxK * 12 + kSmThreads * 4 + 256;

// Order-preserving map of an fp32 value to an unsigned key and back.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ bool sorts_before(uint32_t ka, int ia, uint32_t kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kSmThreads, 1) sample_kernel(const __grid_constant__ SampleArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem);                  // [warps][256]
    uint32_t *keys = hist + kSmWarps * 256;                               // [kSmMaxK]
    int *idx = reinterpret_cast<int *>(keys + kSmMaxK);                   // [kSmMaxK]
    float *pr = reinterpret_cast<float *>(idx + kSmMaxK);                 // [kSmMaxK]
    int *scan = reinterpret_cast<int *>(pr + kSmMaxK);                    // [threads]
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_need, s_count, s_warp_tot[kSmWarps];
    __shared__ float s_sum;

    allow_dependent_launch();
    grid_dependency_wait();
    const int row = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long n = p.n;
    const float *l = p.logits + (long long)row * n;
    const float T = p.temperature;

    if (!(T > 0.0f)) {  // greedy
        float *sv = reinterpret_cast<float *>(hist);
        int *si = reinterpret_cast<int *>(hist) + kSmThreads;
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (long long i = tid; i < n; i += kSmThreads)
            if (ranks_above(l[i], (int)i, bv, bi)) {
                bv = l[i];
                bi = (int)i;
            }
        block_best(bv, bi, sv, si);
        if (tid == 0) {
            p.ids[row] = bi;
            if (p.tokens_adv) p.tokens_adv[row] = bi;
            if (p.pos_adv) p.pos_adv[row] += 1;
        }
        return;
    }

    const long long k_eff = (p.top_k <= 0 || p.top_k >= n) ? n : p.top_k;
    if (tid == 0) {
        s_prefix = 0;
        s_mask = 0;
        s_need = (int)k_eff;
        s_count = 0;
    }
    __syncthreads();

    if (k_eff < n) {
        // radix select of the k_eff-th largest key, 8 bits per pass, MSB first
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int d = lane; d < 256; d += 32) hist[warp * 256 + d] = 0;
            __syncthreads();
            const uint32_t prefix = s_prefix, mask = s_mask;
            for (long long base = 0; base < n; base += kSmThreads) {
                const long long i = base + tid;
                uint32_t key = 0;
                bool m = false;
                if (i < n) {
                    key = order_key(l[i] / T);
                    m = (key & mask) == prefix;
                }
                const unsigned act = __ballot_sync(0xffffffffu, m);
                if (m) {
                    const uint32_t digit = (key >> shift) & 255u;
                    const unsigned peers = __match_any_sync(act, digit);
                    if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[warp * 256 + digit], (uint32_t)__popc(peers));
                }
            }
            __syncthreads();
            if (tid < 256) {
                uint32_t tot = 0;
                for (int w = 0; w < kSmWarps; ++w) tot += hist[w * 256 + tid];
                scan[tid] = (int)tot;
            }
            __syncthreads();
            if (tid == 0) {
                int kk = s_need, cum = 0, sel = 0;
                for (int d = 255; d >= 0; --d) {
                    if (cum + scan[d] >= kk) {
                        sel = d;
                        break;
                    }
                    cum += scan[d];
                }
                s_need = kk - cum;
                s_prefix = prefix | ((uint32_t)sel << shift);
                s_mask = mask | (0xffu << shift);
            }
            __syncthreads();
        }
        // survivors: keys above the threshold, and the lowest-index keys equal to it
        const uint32_t thr = s_prefix;
        const int need_eq = s_need;
        const long long chunk = (n + kSmThreads - 1) / kSmThreads;
        const long long c0 = min(n, chunk * tid), c1 = min(n, c0 + chunk);
        int eq = 0;
        for (long long i = c0; i < c1; ++i) eq += order_key(l[i] / T) == thr;
        int v = eq;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nb = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += nb;
        }
        if (lane == 31) s_warp_tot[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int w = s_warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += nb;
            }
            s_warp_tot[lane] = w;
        }
        __syncthreads();
        int rank = v - eq + (warp > 0 ? s_warp_tot[warp - 1] : 0);
        for (long long i = c0; i < c1; ++i) {
            const uint32_t key = order_key(l[i] / T);
            bool take = key > thr;
            if (key == thr) take = rank++ < need_eq;
            if (take) {
                const int slot = atomicAdd(&s_count, 1);
                if (slot < kSmMaxK) {
                    keys[slot] = key;
                    idx[slot] = (int)i;
                }
            }
        }
    } else {
        for (long long i = tid; i < n; i += kSmThreads) {
            keys[i] = order_key(l[i] / T);
            idx[i] = (int)i;
        }
    }
    __syncthreads();

    const int K = (int)k_eff;
    int P = 1;
    while (P < K) P <<= 1;
    for (int i = K + tid; i < P; i += kSmThreads) {
        keys[i] = 0;
        idx[i] = INT_MAX;
    }
    __syncthreads();
    // bitonic sort into (key desc, index asc)
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < P; i += kSmThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const bool sw = up ? sorts_before(keys[j], idx[j], keys[i], idx[i])
                                       : sorts_before(keys[i], idx[i], keys[j], idx[j]);
                    if (sw) {
                        const uint32_t tk = keys[i];
                        keys[i] = keys[j];
                        keys[j] = tk;
                        const int ti = idx[i];
                        idx[i] = idx[j];
                        idx[j] = ti;
                    }
                }
            }
            __syncthreads();
        }
    }

    const float lmax = key_value(keys[0]);
    for (int i = tid; i < K; i += kSmThreads) pr[i] = expf(key_value(keys[i]) - lmax);
    __syncthreads();
    if (tid == 0) {
        float S = 0.0f;
        for (int i = 0; i < K; ++i) S += pr[i];
        s_sum = S;
        if (!(lmax == lmax) || !(S > 0.0f)) flag_error(p.err, DS_ERR_SAMPLING);
    }
    __syncthreads();
    const float S = s_sum;
    for (int i = tid; i < K; i += kSmThreads) pr[i] = pr[i] / S;
    __syncthreads();
    if (tid == 0) {
        int kept = K;
        if (p.top_p < 1.0f) {
            float excl = 0.0f;
            kept = 0;
            while (kept < K && (kept == 0 || excl < p.top_p)) {
                excl += pr[kept];
                ++kept;
            }
        }
        float S2 = 0.0f;
        for (int i = 0; i < kept; ++i) S2 += pr[i];
        const float target = p.u[row] * S2;
        float incl = 0.0f;
        int chosen = -1;
        for (int i = 0; i < kept; ++i) {
            incl += pr[i];
            if (incl > target) {
                chosen = i;
                break;
            }
        }
        if (chosen < 0) chosen = kept - 1;
        const int id = idx[chosen];
        p.ids[row] = id;
        if (p.tokens_adv) p.tokens_adv[row] = id;
        if (p.pos_adv) p.pos_adv[row] += 1;
    }
}

static bool g_sample_ready = false;

cudaError_t prepare_sample_kernel() {
    cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmSmem);
    if (e == cudaSuccess) g_sample_ready = true;
    return e;
}

cudaError_t launch_sample(const SampleArgs &a, cudaStream_t stream, bool pdl) {
    if (!g_sample_ready) {
        cudaError_t e = prepare_sample_kernel();
        if (e != cudaSuccess) return e;
    }
    return launch_ex(sample_kernel, dim3(a.n_rows), dim3(kSmThreads), kSmSmem, stream, pdl, a);
}

}  // namespace ds

using namespace ds;

extern "C" DS_API size_t ds_argmax_workspace_bytes(int n_rows, int64_t n) {
    if (n_rows < 1 || n < 1) return 0;
    const int B = argmax_blocks_per_row(n);
    return kWsHeader + align_up((size_t)n_rows * 4, 256) + align_up((size_t)n_rows * B * 4, 256) * 2;
}

extern "C" DS_API int ds_greedy_argmax(const float *logits, int64_t logits_len, int n_rows, int64_t n, int32_t *ids,
                                       float *max_logit, void *workspace, size_t workspace_bytes, ds_stream_t stream) {
    if (n_rows < 1 || n < 1) return DS_EMPTY_DIMENSION;
    if (n_rows > 65535 || n > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (logits_len != (int64_t)n_rows * n) return DS_LOGITS_LENGTH_MISMATCH;
    if (!logits || !ids) return DS_BAD_ARGUMENT;
    const size_t need = ds_argmax_workspace_bytes(n_rows, n);
    if (!workspace || workspace_bytes < need) return DS_WORKSPACE_TOO_SMALL;
    if ((uintptr_t)workspace & 255) return DS_BAD_ARGUMENT;
    const int B = argmax_blocks_per_row(n);
    char *ws = static_cast<char *>(workspace);
    ArgmaxArgs a = {};
    a.logits = logits;
    a.n_rows = n_rows;
    a.n = n;
    a.ids = ids;
    a.max_logit = max_logit;
    a.err = reinterpret_cast<int *>(ws);
    a.counters = reinterpret_cast<int *>(ws + kWsHeader);
    char *pv = ws + kWsHeader + align_up((size_t)n_rows * 4, 256);
    a.part_val = reinterpret_cast<float *>(pv);
    a.part_idx = reinterpret_cast<int *>(pv + align_up((size_t)n_rows * B * 4, 256));
    a.blocks_per_row = B;
    cudaError_t e = launch_argmax(a, reinterpret_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

extern "C" DS_API size_t ds_sample_workspace_bytes(int n_rows, int64_t n) {
    if (n_rows < 1 || n < 1) return 0;
    return kWsHeader;
}

extern "C" DS_API int ds_sample(const float *logits, int64_t logits_len, int n_rows, int64_t n, float temperature,
                                int top_k, float top_p, const float *u, int32_t *ids, void *workspace,
                                size_t workspace_bytes, ds_stream_t stream) {
    if (n_rows < 1 || n < 1) return DS_EMPTY_DIMENSION;
    if (n_rows > 65535 || n > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (logits_len != (int64_t)n_rows * n) return DS_LOGITS_LENGTH_MISMATCH;
    if (temperature > 0.0f) {
        const int64_t k_eff = (top_k <= 0 || top_k >= n) ? n : top_k;
        if (k_eff > DS_SAMPLE_MAX_TOP_K) return DS_BAD_SAMPLING_PARAM;
        if (!(top_p > 0.0f) || top_p > 1.0f) return DS_BAD_SAMPLING_PARAM;
        if (!u) return DS_BAD_ARGUMENT;
    } else if (temperature != temperature) {
        return DS_BAD_SAMPLING_PARAM;
    }
    if (!logits || !ids) return DS_BAD_ARGUMENT;
    const size_t need = ds_sample_workspace_bytes(n_rows, n);
    if (!workspace || workspace_bytes < need) return DS_WORKSPACE_TOO_SMALL;
    SampleArgs a = {};
    a.logits = logits;
    a.n_rows = n_rows;
    a.n = n;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.u = u;
    a.ids = ids;
    a.err = static_cast<int *>(workspace);
    cudaError_t e = launch_sample(a, reinterpret_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}
