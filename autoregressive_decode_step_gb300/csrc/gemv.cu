// Weight-streaming mat-vecs for the decode step.
//
// gemv_t: y = A^T x with A [K rows][N cols] row-major — the transposed
// mat-vec of the "LLM inference kernels" page ("A parallel path for one
// frozen kernel's known-slow shape").  The page hands disjoint column bands
// to workers, each running an i-outer / j-inner loop.  Here a band is 512
// bytes of every row (256 bf16 or 128 fp32 columns): a warp covers a band row
// with one 16-byte load per lane, so every weight byte is read exactly once,
// coalesced.  The (band, row) space is flattened and cut into equal
// contiguous ranges, one per CTA (one CTA per SM), so the grid is balanced to
// one row whatever the matrix shape ("split-K where rows are few").  A
// producer warp streams each range's rows into a 6-stage shared-memory ring
// with bulk asynchronous copies (cp.async.bulk, the TMA engine) tracked by
// mbarriers; eight consumer warps accumulate in fp32 registers.  Partial sums
// of a band split across CTAs meet in a workspace; the last CTA to finish a
// band (an atomic counter, never a wait) adds them in CTA order — a fixed
// order, so results are bit-stable — and runs the fused epilogue: store,
// residual add, SiLU-gate, or RoPE + K/V cache write.
//
// gemv_n: y = W x with W [rows][cols] row-major (the output head).  Each CTA
// streams a contiguous run of whole rows; the greedy argmax over the rows is
// fused in ("Inside the engine", section 1: the fused tail keeps the final
// norm, the output head and the argmax on the same stream).
//
// Both kernels fetch weights before waiting on the previous kernel
// (programmatic dependent launch): weights never depend on it.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "internal.h"
#include "tc.h"

namespace ds {

constexpr int kGtThreads = (kGtConsumerWarps + 1) * 32;
constexpr int kGtConsumers = kGtConsumerWarps * 32;
constexpr int kGtStageBytes = kGtBandBytes * kGtRows;
constexpr int kGtBoxesPerStage = kGtRows / kGtBoxRows;
constexpr int kGtRedFloats = kGtConsumerWarps * 256;
// ring | red | vals | barriers and flags | x slice (xs_cap floats)
constexpr size_t kGtSmemBase = (size_t)kGtStages * kGtStageBytes + kGtRedFloats * 4 + 256 * 4 + 256;
constexpr int kGtMaxXs = 16384;  // floats of x one CTA may stage (64 KB)
constexpr size_t kGtSmemMax = std::min<size_t>(kGtSmemBase + (size_t)kGtMaxXs * 4, 227 * 1024);
static_assert(kGtRows % kGtBoxRows == 0, "stage rows must be whole boxes");

// CTA whose range holds unit u when W units are cut into G ranges
// [W*c/G, W*(c+1)/G).
__device__ __forceinline__ int cta_of_unit(long long u, long long W, int G) {
    return (int)(((u + 1) * (long long)G - 1) / W);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }


template <typename T, int PRO, int EPI>
__global__ void __launch_bounds__(kGtThreads, 1) gemv_t_kernel(const __grid_constant__ GemvTArgs p) {
    constexpr int ES = sizeof(T);
    constexpr int LE = 16 / ES;                  // elements per lane per row
    constexpr int BAND_COLS = kGtBandBytes / ES; // partial columns per band
    constexpr bool PAIRED = (EPI == EPI_SILU);
    constexpr int SUB_BAND_COLS = PAIRED ? BAND_COLS / 2 : BAND_COLS;
    constexpr int SUB_ROW_BYTES = SUB_BAND_COLS * ES;          // bytes of one box row
    constexpr uint32_t BOX_BYTES = kGtBoxRows * SUB_ROW_BYTES;  // bytes of one box

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)kGtStages * kGtStageBytes);
    float *vals = red + kGtRedFloats;
    uint64_t *full = reinterpret_cast<uint64_t *>(vals + 256);
    uint64_t *empty = full + kGtStages;
    volatile int *s_flag = reinterpret_cast<volatile int *>(empty + kGtStages);
    volatile int *s_abort = s_flag + 1;
    float *s_scale = reinterpret_cast<float *>(const_cast<int *>(s_flag) + 2);
    float *xs = reinterpret_cast<float *>(smem + kGtSmemBase);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    // work units are boxes of kGtBoxRows rows of one band
    const int UB = (p.K + kGtBoxRows - 1) / kGtBoxRows;  // boxes per band
    const long long W = (long long)p.n_bands * UB;
    const long long u0 = W * blockIdx.x / G, u1 = W * (blockIdx.x + 1) / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kGtConsumerWarps);
        }
        *s_flag = 0;
        *s_abort = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    allow_dependent_launch();

    if (warp == kGtConsumerWarps) {
        // ---------------- producer: stream this CTA's boxes into the ring
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t fill = 0;
            bool ok = true;
            for (long long u = u0; u < u1 && ok;) {
                const int band = (int)(u / UB);
                const int j0 = (int)(u - (long long)band * UB);
                const int j1 = (int)min((long long)UB, j0 + (u1 - u));
                for (int j = j0; j < j1; j += kGtBoxesPerStage) {
                    const int nb = min(kGtBoxesPerStage, j1 - j);
                    const int s = fill % kGtStages;
                    const uint32_t use = fill / kGtStages;
                    if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, p.err)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], (uint32_t)nb * BOX_BYTES * (PAIRED ? 2 : 1));
                    unsigned char *dst = ring + (size_t)s * kGtStageBytes;
                    for (int b = 0; b < nb; ++b) {
                        const int r = (j + b) * kGtBoxRows;
                        tma_box_g2s(dst + b * BOX_BYTES, &p.tm0, band * SUB_BAND_COLS, r, &full[s], pol);
                        if (PAIRED)
                            tma_box_g2s(dst + kGtStageBytes / 2 + b * BOX_BYTES, &p.tm1, band * SUB_BAND_COLS, r,
                                        &full[s], pol);
                    }
                    ++fill;
                }
                u += j1 - j0;
            }
            // every copy this CTA issued must land before its shared memory
            // is released (bounded wait; already complete on the normal path)
            const uint32_t first = fill > (uint32_t)kGtStages ? fill - kGtStages : 0;
            for (uint32_t f = first; f < fill; ++f) mbar_wait(&full[f % kGtStages], (f / kGtStages) & 1, p.err);
        }
        return;
    }

    // ---------------- consumers
    const int t = threadIdx.x;  // 0 .. kGtConsumers-1
    grid_dependency_wait();

    float scale = 1.0f;
    if (PRO == PRO_RMSNORM) {
        // RMSNorm of the residual, square sum in fp32; every CTA computes the
        // same value in the same order.
        float ss = 0.0f;
        for (int i = t; i < p.K; i += kGtConsumers) {
            const float r = p.x[i];
            ss = fmaf(r, r, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        named_sync(1, kGtConsumers);
        if (t == 0) {
            float tot = 0.0f;
            for (int w = 0; w < kGtConsumerWarps; ++w) tot += red[w];
            *s_scale = 1.0f / sqrtf(tot / (float)p.K + p.eps);
        }
        named_sync(1, kGtConsumers);
        scale = *s_scale;
    }
    // this CTA's slice of x (normalised; zero past K) into shared memory
    {
        int off = 0;
        for (long long u = u0; u < u1;) {
            const int band = (int)(u / UB);
            const int j0 = (int)(u - (long long)band * UB);
            const int j1 = (int)min((long long)UB, j0 + (u1 - u));
            u += j1 - j0;
            const int k0 = j0 * kGtBoxRows, k1 = j1 * kGtBoxRows;
            for (int k = k0 + t; k < k1; k += kGtConsumers) {
                float v = 0.0f;
                if (k < p.K) {
                    v = p.x[k];
                    if (PRO == PRO_RMSNORM) v = v * scale * p.norm_w[k];
                }
                if (off + k - k0 < p.xs_cap) xs[off + k - k0] = v;
            }
            off += k1 - k0;
        }
        named_sync(1, kGtConsumers);
    }

    uint32_t fill = 0;
    int seg_off = 0;
    for (long long u = u0; u < u1;) {
        const int band = (int)(u / UB);
        const int j0 = (int)(u - (long long)band * UB);
        const int j1 = (int)min((long long)UB, j0 + (u1 - u));
        u += j1 - j0;
        const float *xseg = xs + seg_off - j0 * kGtBoxRows;  // xseg[k] for rows of this segment
        seg_off += (j1 - j0) * kGtBoxRows;

        float acc[LE];
#pragma unroll
        for (int e = 0; e < LE; ++e) acc[e] = 0.0f;
        for (int j = j0; j < j1; j += kGtBoxesPerStage) {
            const int nr = min(kGtBoxesPerStage, j1 - j) * kGtBoxRows;
            const int s = fill % kGtStages;
            const uint32_t use = fill / kGtStages;
            if (!*s_abort) {
                if (!mbar_wait(&full[s], use & 1, p.err)) *s_abort = 1;
            }
            if (!*s_abort) {
                const unsigned char *st = ring + (size_t)s * kGtStageBytes;
                // lane's 16 bytes of row r: one dense [rows][SUB_ROW_BYTES] array
                // per sub-tile, sub-tile 1 (lanes 16-31 when paired) in the upper half
                const unsigned char *lane_base =
                    PAIRED ? st + (lane >> 4) * (kGtStageBytes / 2) + (lane & 15) * 16 : st + lane * 16;
                const int kr = j * kGtBoxRows;
#pragma unroll 4
                for (int r = warp; r < nr; r += kGtConsumerWarps) {
                    const float xk = xseg[kr + r];
                    const uint4 w = *reinterpret_cast<const uint4 *>(lane_base + r * SUB_ROW_BYTES);
                    float f[LE];
                    widen16(w, f);
#pragma unroll
                    for (int e = 0; e < LE; ++e) acc[e] = fmaf(f[e], xk, acc[e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++fill;
        }

        // cross-warp reduction of the band's column sums, fixed order
#pragma unroll
        for (int e = 0; e < LE; ++e) red[warp * BAND_COLS + lane * LE + e] = acc[e];
        named_sync(1, kGtConsumers);
        float v = 0.0f;
        if (t < BAND_COLS)
            for (int w = 0; w < kGtConsumerWarps; ++w) v += red[w * BAND_COLS + t];

        const bool sole = (j0 == 0 && j1 == UB);
        if (!sole) {
            const int first = cta_of_unit((long long)band * UB, W, G);
            const int last = cta_of_unit((long long)(band + 1) * UB - 1, W, G);
            const int n_contrib = last - first + 1;
            if (t < BAND_COLS) p.partials[(size_t)(blockIdx.x + band) * BAND_COLS + t] = v;
            __threadfence();
            named_sync(1, kGtConsumers);
            if (t == 0) *s_flag = (atomicAdd(&p.counters[band], 1) == n_contrib - 1);
            named_sync(1, kGtConsumers);
            if (!*s_flag) continue;
            __threadfence();
            v = 0.0f;
            if (t < BAND_COLS)
                for (int c = 0; c < n_contrib; ++c)
                    v += __ldcg(&p.partials[(size_t)(first + c + band) * BAND_COLS + t]);
            if (t == 0) p.counters[band] = 0;
        }

        // ---------------- epilogue for this band
        if (EPI == EPI_STORE || EPI == EPI_ADD) {
            const int col = band * BAND_COLS + t;
            if (t < BAND_COLS && col < p.sub_cols) {
                if (EPI == EPI_STORE)
                    p.y[col] = v;
                else
                    p.y[col] += v;
            }
        } else if (EPI == EPI_SILU) {
            vals[t] = v;
            named_sync(1, kGtConsumers);
            const int col = band * SUB_BAND_COLS + t;
            if (t < SUB_BAND_COLS && col < p.sub_cols) p.y[col] = silu_f(vals[t]) * vals[t + SUB_BAND_COLS];
        } else {  // EPI_QKV
            vals[t] = v;
            named_sync(1, kGtConsumers);
            if (p.q_norm) {  // QK-norm: each q / k head of the band RMS-normalised before RoPE
                const int col = band * BAND_COLS + t;
                const bool normed = t < BAND_COLS && col < p.nq_cols + p.nkv_cols;
                const int hd = p.head_dim;
                const float x = normed ? v : 0.0f;
                float s2 = x * x;
                if (hd >= 32) {  // a head spans hd / 32 whole warps; red is free here
                    s2 = warp_sum(s2);
                    if (lane == 0) red[warp] = s2;
                    named_sync(1, kGtConsumers);
                    const int w0 = (t / hd) * (hd >> 5);
                    s2 = 0.0f;
                    for (int w = w0; w < w0 + (hd >> 5); ++w) s2 += red[w];
                } else {
                    for (int o = hd >> 1; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                }
                if (normed) {
                    const bool is_q = col < p.nq_cols;
                    const int i = (is_q ? col : col - p.nq_cols) % hd;
                    v = x * (1.0f / sqrtf(s2 / (float)hd + p.eps)) * __ldg((is_q ? p.q_norm : p.k_norm) + i);
                    vals[t] = v;
                }
                named_sync(1, kGtConsumers);
            }
            const int col = band * BAND_COLS + t;
            const int total = p.nq_cols + 2 * p.nkv_cols;
            const int pos = *p.pos;
            const int cap = p.max_blocks * p.block_tokens;
            const bool pos_ok = pos >= 0 && pos < p.rope_rows && pos < cap;
            if (!pos_ok && t == 0) flag_error(p.err, DS_ERR_POSITION);
            if (t < BAND_COLS && col < total) {
                float out = v;
                if (col < p.nq_cols + p.nkv_cols) {
                    const int hd = p.head_dim, half = hd >> 1;
                    const int region = col < p.nq_cols ? 0 : p.nq_cols;
                    const int i = (col - region) % hd;
                    int pair;
                    float a, b;
                    bool first_of_pair;
                    if (p.rope_layout == DS_ROPE_HALF_SPLIT) {
                        first_of_pair = i < half;
                        pair = first_of_pair ? i : i - half;
                        a = first_of_pair ? vals[t] : vals[t - half];
                        b = first_of_pair ? vals[t + half] : vals[t];
                    } else {
                        first_of_pair = (i & 1) == 0;
                        pair = i >> 1;
                        a = first_of_pair ? vals[t] : vals[t - 1];
                        b = first_of_pair ? vals[t + 1] : vals[t];
                    }
                    float c = 1.0f, sn = 0.0f;
                    if (pos_ok) {
                        c = p.rope_cos[(size_t)pos * half + pair];
                        sn = p.rope_sin[(size_t)pos * half + pair];
                    }
                    out = first_of_pair ? a * c - b * sn : a * sn + b * c;
                }
                if (col < p.nq_cols) {
                    p.y[col] = out;
                } else if (pos_ok) {
                    const int blk = p.block_table ? p.block_table[pos / p.block_tokens] : pos / p.block_tokens;
                    const long long row = (long long)blk * p.block_tokens + pos % p.block_tokens;
                    if (col < p.nq_cols + p.nkv_cols)
                        store_as(p.k_cache, row * p.nkv_cols + (col - p.nq_cols), p.kv_dtype, out);
                    else
                        store_as(p.v_cache, row * p.nkv_cols + (col - p.nq_cols - p.nkv_cols), p.kv_dtype, out);
                }
            }
        }
        named_sync(1, kGtConsumers);  // red / vals free for the next band
    }
}

// Plain-load fallback for shapes the tensor-map path cannot stream (rows not a
// multiple of 16 bytes or a misaligned base): one thread per output column,
// rows summed in order.
template <typename T>
__global__ void gemv_t_plain_kernel(const T *A, const float *x, int K, int N, float *y) {
    grid_dependency_wait();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) acc = fmaf(to_f32(A[(long long)k * N + j]), __ldg(x + k), acc);
    y[j] = acc;
}

int gemv_t_grid(int K, int n_bands) {
    const long long UB = (K + kGtBoxRows - 1) / kGtBoxRows;
    const long long W = UB * n_bands;
    long long g = (W + 7) / 8;  // at least 8 boxes per CTA
    g = std::min<long long>(g, sm_count());
    // enough CTAs that each one's slice of x fits in shared memory
    const long long per = kGtMaxXs / kGtBoxRows - 1;
    g = std::max(g, (W + per - 1) / per);
    return (int)std::max(1LL, g);
}

static int gemv_t_xs_cap(int K, int n_bands, int grid) {
    const long long UB = (K + kGtBoxRows - 1) / kGtBoxRows;
    const long long W = UB * n_bands;
    return (int)(((W + grid - 1) / grid + 1) * kGtBoxRows);
}

size_t gemv_t_partial_floats(int grid, int n_bands, int es) {
    return (size_t)(grid + n_bands) * gemv_t_band_cols(es);
}

bool gemv_t_streamable(const void *a0, const void *a1, long long row_stride, int sub_cols, int es) {
    if (((uintptr_t)a0 & 15) || (a1 && ((uintptr_t)a1 & 15))) return false;
    if (row_stride % 16 || row_stride >= (1LL << 40)) return false;
    if (((long long)sub_cols * es) % 16) return false;
    return true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
        else
            cudaGetLastError();
    }
    return fn;
}

static bool encode_band_map(CUtensorMap *m, const void *base, int dtype, long long cols, long long rows,
                            long long row_stride, int box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kGtBoxRows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = dtype == DS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_2d(CUtensorMap *m, const void *base, int dtype, long long cols, long long rows,
                     long long row_stride, int box_cols, int box_rows, bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = dtype == DS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_3d(CUtensorMap *m, const void *base, int dtype, const long long dims[3], const long long strides[2],
                     const int box[3], bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t d[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
    const cuuint64_t st[2] = {(cuuint64_t)strides[0], (cuuint64_t)strides[1]};
    const cuuint32_t bx[3] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = dtype == DS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(m, dt, 3, const_cast<void *>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemv_t_make_maps(GemvTArgs &a, int dtype) {
    const int es = dtype == DS_BF16 ? 2 : 4;
    const int band_cols = gemv_t_band_cols(es);
    const int box_cols = a.a1 ? band_cols / 2 : band_cols;
    if (!encode_band_map(&a.tm0, a.a0, dtype, a.sub_cols, a.K, a.row_stride, box_cols)) return false;
    if (a.a1 && !encode_band_map(&a.tm1, a.a1, dtype, a.sub_cols, a.K, a.row_stride, box_cols)) return false;
    return true;
}

// Opt each instantiation into its dynamic shared memory once (the model
// calls prepare_kernels() before any capture; op calls do it lazily).
template <typename T, int PRO, int EPI>
static cudaError_t ensure_gt(bool force = false) {
    static bool done = false;
    if (done && !force) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemv_t_kernel<T, PRO, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kGtSmemMax);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int PRO, int EPI>
static cudaError_t launch_gt(const GemvTArgs &a, int grid, cudaStream_t stream, bool pdl) {
    cudaError_t e = ensure_gt<T, PRO, EPI>();
    if (e != cudaSuccess) return e;
    GemvTArgs b = a;
    b.xs_cap = gemv_t_xs_cap(a.K, a.n_bands, grid);
    if (b.xs_cap > kGtMaxXs) return cudaErrorInvalidValue;
    const size_t smem = kGtSmemBase + align_up((size_t)b.xs_cap * 4, 16);
    return launch_ex(gemv_t_kernel<T, PRO, EPI>, dim3(grid), dim3(kGtThreads), smem, stream, pdl, b);
}

template <typename T>
static cudaError_t launch_gt_dtype(const GemvTArgs &a, int pro, int epi, int grid,
                                   cudaStream_t stream, bool pdl) {
    if (pro == PRO_PLAIN && epi == EPI_STORE) return launch_gt<T, PRO_PLAIN, EPI_STORE>(a, grid, stream, pdl);
    if (pro == PRO_PLAIN && epi == EPI_ADD) return launch_gt<T, PRO_PLAIN, EPI_ADD>(a, grid, stream, pdl);
    if (pro == PRO_RMSNORM && epi == EPI_QKV) return launch_gt<T, PRO_RMSNORM, EPI_QKV>(a, grid, stream, pdl);
    if (pro == PRO_RMSNORM && epi == EPI_SILU) return launch_gt<T, PRO_RMSNORM, EPI_SILU>(a, grid, stream, pdl);
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return launch_gt<T, PRO_RMSNORM, EPI_STORE>(a, grid, stream, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_t(const GemvTArgs &a, int dtype, int pro, int epi, int grid,
                          cudaStream_t stream, bool pdl) {
    if (dtype == DS_BF16) return launch_gt_dtype<__nv_bfloat16>(a, pro, epi, grid, stream, pdl);
    return launch_gt_dtype<float>(a, pro, epi, grid, stream, pdl);
}

// =====================================================================
// gemv_n: whole rows per CTA, fused greedy argmax
// =====================================================================
#ifndef DS_GN_STAGE_BYTES
#define DS_GN_STAGE_BYTES 65536
#endif
#ifndef DS_GN_STAGES
#define DS_GN_STAGES 3
#endif
constexpr int kGnStageBytes = DS_GN_STAGE_BYTES;
constexpr int kGnStages = DS_GN_STAGES;
constexpr int kGnConsumerWarps = 8;
constexpr int kGnThreads = (kGnConsumerWarps + 1) * 32;
constexpr int kGnConsumers = kGnConsumerWarps * 32;
constexpr int kGnMaxCols = 8192;
constexpr int kGnMaxRowsPerStage = 256;
// ring | barriers and flags | best value/index per consumer | x | row partials
constexpr size_t kGnSmemBase = (size_t)kGnStages * kGnStageBytes + 256 + (size_t)kGnConsumers * 8;
constexpr size_t kGnSmemMax = 227 * 1024;

__host__ __device__ inline int gn_rows_per_stage(long long row_bytes) {
    long long r = kGnStageBytes / row_bytes;
    return (int)(r < 1 ? 1 : (r > kGnMaxRowsPerStage ? kGnMaxRowsPerStage : r));
}
__host__ __device__ inline int gn_parts(int rps) { return rps >= kGnConsumerWarps ? 1 : kGnConsumerWarps / rps; }

template <typename T, int PRO>
__global__ void __launch_bounds__(kGnThreads, 1) gemv_n_kernel(const __grid_constant__ GemvNArgs p) {
    constexpr int ES = sizeof(T);
    constexpr int LE = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kGnStages * kGnStageBytes);
    uint64_t *empty = full + kGnStages;
    volatile int *s_flag = reinterpret_cast<volatile int *>(empty + kGnStages);
    volatile int *s_abort = s_flag + 1;
    float *s_scale = reinterpret_cast<float *>(const_cast<int *>(s_flag) + 2);
    float *bestv = reinterpret_cast<float *>(smem + (size_t)kGnStages * kGnStageBytes + 256);
    int *besti = reinterpret_cast<int *>(bestv + kGnConsumers);
    float *xs = reinterpret_cast<float *>(besti + kGnConsumers);
    float *rowpart = xs + p.cols;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long row_bytes = (long long)p.cols * ES;
    const int rps = gn_rows_per_stage(row_bytes);
    const int parts = gn_parts(rps);
    const int r0 = (int)((long long)p.rows * blockIdx.x / G);
    const int r1 = (int)((long long)p.rows * (blockIdx.x + 1) / G);
    const int n_stages = (r1 - r0 + rps - 1) / rps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGnStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kGnConsumerWarps);
        }
        *s_flag = 0;
        *s_abort = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    allow_dependent_launch();

    if (warp == kGnConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int i = 0;
            for (; i < n_stages; ++i) {
                const int s = i % kGnStages;
                const uint32_t use = i / kGnStages;
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, p.err)) {
                    *s_abort = 1;
                    break;
                }
                const int rr = r0 + i * rps;
                const int nr = min(rps, r1 - rr);
                const uint32_t bytes = (uint32_t)(nr * row_bytes);
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_g2s(ring + (size_t)s * kGnStageBytes, p.W + (long long)rr * row_bytes, bytes, &full[s], pol);
            }
            const int first = i > kGnStages ? i - kGnStages : 0;
            for (int f = first; f < i; ++f) mbar_wait(&full[f % kGnStages], (f / kGnStages) & 1, p.err);
        }
        return;
    }

    const int t = threadIdx.x;
    grid_dependency_wait();

    // x (optionally RMS-normalised) into shared memory
    float scale = 1.0f;
    if (PRO == PRO_RMSNORM) {
        float ss = 0.0f;
        for (int i = t; i < p.cols; i += kGnConsumers) {
            const float r = p.x[i];
            ss = fmaf(r, r, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) bestv[warp] = ss;
        named_sync(1, kGnConsumers);
        if (t == 0) {
            float tot = 0.0f;
            for (int w = 0; w < kGnConsumerWarps; ++w) tot += bestv[w];
            *s_scale = 1.0f / sqrtf(tot / (float)p.cols + p.eps);
        }
        named_sync(1, kGnConsumers);
        scale = *s_scale;
    }
    for (int i = t; i < p.cols; i += kGnConsumers) {
        float v = p.x[i];
        if (PRO == PRO_RMSNORM) v = v * scale * p.norm_w[i];
        xs[i] = v;
    }
    named_sync(1, kGnConsumers);

    // dot products: each warp owns one (row, part) of every stage; the part
    // sums wait in shared memory until the CTA's rows are all done
    const int chunks = (int)(row_bytes / 16);
    for (int i = 0; i < n_stages; ++i) {
        const int s = i % kGnStages;
        const uint32_t use = i / kGnStages;
        const int rr = r0 + i * rps;
        const int nr = min(rps, r1 - rr);
        if (!*s_abort) {
            if (!mbar_wait(&full[s], use & 1, p.err)) *s_abort = 1;
        }
        if (!*s_abort) {
            const unsigned char *st = ring + (size_t)s * kGnStageBytes;
            if (parts == 1) {
                for (int r = warp; r < nr; r += kGnConsumerWarps) {
                    const unsigned char *row = st + (size_t)r * row_bytes;
                    float acc = 0.0f;
                    for (int c = lane; c < chunks; c += 32) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + c * 16);
                        float f[LE];
                        widen16(w, f);
#pragma unroll
                        for (int e = 0; e < LE; ++e) acc = fmaf(f[e], xs[c * LE + e], acc);
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) rowpart[rr - r0 + r] = acc;
                }
            } else {
                const int r = warp / parts, part = warp % parts;
                if (r < nr) {
                    const unsigned char *row = st + (size_t)r * row_bytes;
                    const int c0 = chunks * part / parts, c1 = chunks * (part + 1) / parts;
                    float acc = 0.0f;
#pragma unroll 4
                    for (int c = c0 + lane; c < c1; c += 32) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + c * 16);
                        float f[LE];
                        widen16(w, f);
#pragma unroll
                        for (int e = 0; e < LE; ++e) acc = fmaf(f[e], xs[c * LE + e], acc);
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) rowpart[(rr - r0 + r) * parts + part] = acc;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    named_sync(1, kGnConsumers);

    // logits in row order, and this CTA's greedy candidate
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    for (int r = t; r < r1 - r0; r += kGnConsumers) {
        float logit = 0.0f;
        for (int q = 0; q < parts; ++q) logit += rowpart[r * parts + q];
        p.y[r0 + r] = logit;
        if (ranks_above(logit, r0 + r, best_v, best_i)) {
            best_v = logit;
            best_i = r0 + r;
        }
    }

    if (!p.do_argmax) return;
    bestv[t] = best_v;
    besti[t] = best_i;
    named_sync(1, kGnConsumers);
    if (t == 0) {
        float bv = bestv[0];
        int bi = besti[0];
        for (int j = 1; j < kGnConsumers; ++j)
            if (ranks_above(bestv[j], besti[j], bv, bi)) {
                bv = bestv[j];
                bi = besti[j];
            }
        p.part_val[blockIdx.x] = bv;
        p.part_idx[blockIdx.x] = bi;
        __threadfence();
        const bool last = atomicAdd(p.counter, 1) == G - 1;
        if (last) {
            __threadfence();
            bv = __ldcg(&p.part_val[0]);
            bi = __ldcg(&p.part_idx[0]);
            for (int j = 1; j < G; ++j) {
                const float v = __ldcg(&p.part_val[j]);
                const int ix = __ldcg(&p.part_idx[j]);
                if (ranks_above(v, ix, bv, bi)) {
                    bv = v;
                    bi = ix;
                }
            }
            *p.counter = 0;
            p.ids_out[0] = bi;
            if (p.max_out) p.max_out[0] = bv;
            if (p.tokens_adv) p.tokens_adv[0] = bi;
            if (p.pos_adv) p.pos_adv[0] += 1;
        }
    }
}

template <typename T>
__global__ void gemv_n_plain_kernel(const T *W, const float *x, int rows, int cols, float *y) {
    grid_dependency_wait();
    const int warps = blockDim.x >> 5;
    const int r = blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    float acc = 0.0f;
    for (int c = lane; c < cols; c += 32) acc = fmaf(to_f32(W[(long long)r * cols + c]), __ldg(x + c), acc);
    acc = warp_sum(acc);
    if (lane == 0) y[r] = acc;
}

// Floats of shared memory left for per-row partial sums once the ring and x
// are placed.
static long long gn_rowpart_budget(int cols) {
    return ((long long)kGnSmemMax - (long long)kGnSmemBase - (long long)cols * 4 - 16) / 4;
}

int gemv_n_grid(int rows, int cols, int es) {
    const long long row_bytes = (long long)cols * es;
    const int rps = gn_rows_per_stage(row_bytes);
    const int parts = gn_parts(rps);
    long long g = (rows + rps - 1) / rps;
    g = std::min<long long>(g, sm_count());
    // enough CTAs that each one's row partials fit in shared memory
    const long long per = std::max(1LL, gn_rowpart_budget(cols) / parts - 1);
    g = std::max(g, (rows + per - 1) / per);
    return (int)std::max(1LL, g);
}

static size_t gemv_n_smem(int rows, int cols, int es, int grid) {
    const int rps = gn_rows_per_stage((long long)cols * es);
    const long long rows_cap = ((long long)rows + grid - 1) / grid + 1;
    return kGnSmemBase + (size_t)cols * 4 + align_up((size_t)rows_cap * gn_parts(rps) * 4, 16);
}

bool gemv_n_streamable(const void *W, int rows, int cols, int es) {
    if ((uintptr_t)W & 15) return false;
    const long long row_bytes = (long long)cols * es;
    if (row_bytes % 16 || row_bytes > kGnStageBytes || cols > kGnMaxCols) return false;
    (void)rows;
    return gn_rowpart_budget(cols) >= 4LL * gn_parts(gn_rows_per_stage(row_bytes));
}

template <typename T, int PRO>
static cudaError_t ensure_gn(bool force = false) {
    static bool done = false;
    if (done && !force) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(gemv_n_kernel<T, PRO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGnSmemMax);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int PRO>
static cudaError_t launch_gn(const GemvNArgs &a, int grid, cudaStream_t stream, bool pdl) {
    cudaError_t e = ensure_gn<T, PRO>();
    if (e != cudaSuccess) return e;
    const size_t smem = gemv_n_smem(a.rows, a.cols, (int)sizeof(T), grid);
    return launch_ex(gemv_n_kernel<T, PRO>, dim3(grid), dim3(kGnThreads), smem, stream, pdl, a);
}

template <typename T>
static cudaError_t prepare_dtype() {
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = ensure_gt<T, PRO_PLAIN, EPI_STORE>(true);
    if (e == cudaSuccess) e = ensure_gt<T, PRO_PLAIN, EPI_ADD>(true);
    if (e == cudaSuccess) e = ensure_gt<T, PRO_RMSNORM, EPI_QKV>(true);
    if (e == cudaSuccess) e = ensure_gt<T, PRO_RMSNORM, EPI_SILU>(true);
    if (e == cudaSuccess) e = ensure_gt<T, PRO_RMSNORM, EPI_STORE>(true);
    if (e == cudaSuccess) e = ensure_gn<T, PRO_PLAIN>(true);
    if (e == cudaSuccess) e = ensure_gn<T, PRO_RMSNORM>(true);
    return e;
}

cudaError_t prepare_sample_kernel();

// Set every kernel's shared-memory attribute on the current device.
cudaError_t prepare_kernels() {
    cudaError_t e = prepare_dtype<float>();
    if (e == cudaSuccess) e = prepare_dtype<__nv_bfloat16>();
    if (e == cudaSuccess) e = prepare_sample_kernel();
    return e;
}

cudaError_t launch_gemv_n(const GemvNArgs &a, int dtype, int pro, int grid, cudaStream_t stream, bool pdl) {
    if (dtype == DS_BF16)
        return pro == PRO_RMSNORM ? launch_gn<__nv_bfloat16, PRO_RMSNORM>(a, grid, stream, pdl)
                                  : launch_gn<__nv_bfloat16, PRO_PLAIN>(a, grid, stream, pdl);
    return pro == PRO_RMSNORM ? launch_gn<float, PRO_RMSNORM>(a, grid, stream, pdl)
                              : launch_gn<float, PRO_PLAIN>(a, grid, stream, pdl);
}

}  // namespace ds

// =====================================================================
// C ABI
// =====================================================================
using namespace ds;

static int check_matvec(const void *A, int64_t a_len, int dtype, const float *x, int64_t x_len,
                        int64_t rows, int64_t cols, const float *y, int64_t y_len, int64_t x_need,
                        int64_t y_need) {
    if (rows < 1 || cols < 1) return DS_EMPTY_DIMENSION;
    if (rows > DS_MAX_DIM || cols > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (dtype != DS_F32 && dtype != DS_BF16) return DS_BAD_DTYPE;
    if (a_len != rows * cols) return DS_GEMV_A_LENGTH_MISMATCH;
    if (x_len != x_need) return DS_GEMV_X_LENGTH_MISMATCH;
    if (y_len != y_need) return DS_A_LENGTH_MISMATCH;
    if (!A || !x || !y) return DS_BAD_ARGUMENT;
    return DS_OK;
}

extern "C" DS_API size_t ds_gemv_workspace_bytes(int64_t rows, int64_t cols, int a_dtype) {
    if (rows < 1 || cols < 1 || rows > DS_MAX_DIM || cols > DS_MAX_DIM) return 0;
    const int es = a_dtype == DS_BF16 ? 2 : 4;
    const int band_cols = gemv_t_band_cols(es);
    const int n_bands = (int)((cols + band_cols - 1) / band_cols);
    const int grid = gemv_t_grid((int)rows, n_bands);
    return kWsHeader + align_up((size_t)n_bands * 4, 256) + gemv_t_partial_floats(grid, n_bands, es) * 4;
}

namespace ds {

bool gemv_t_uses_workspace(const void *A, int64_t cols, int a_dtype) {
    const int es = a_dtype == DS_BF16 ? 2 : 4;
    return gemv_t_streamable(A, nullptr, cols * es, (int)cols, es);
}

size_t gemv_t_zeroed_bytes(int64_t cols, int a_dtype) {
    const int es = a_dtype == DS_BF16 ? 2 : 4;
    const int band_cols = gemv_t_band_cols(es);
    const int64_t n_bands = (cols + band_cols - 1) / band_cols;
    return kWsHeader + align_up((size_t)n_bands * 4, 256);
}

int gemv_transposed_run(const void *A, int a_dtype, const float *x, int64_t rows, int64_t cols, float *y,
                        char *ws, cudaStream_t s) {
    const int es = a_dtype == DS_BF16 ? 2 : 4;
    cudaError_t e;
    if (!gemv_t_uses_workspace(A, cols, a_dtype)) {
        const int threads = 256;
        const int blocks = (int)((cols + threads - 1) / threads);
        if (a_dtype == DS_BF16)
            e = launch_ex(gemv_t_plain_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, s, false,
                          (const __nv_bfloat16 *)A, x, (int)rows, (int)cols, y);
        else
            e = launch_ex(gemv_t_plain_kernel<float>, dim3(blocks), dim3(threads), 0, s, false,
                          (const float *)A, x, (int)rows, (int)cols, y);
        return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
    }
    const int band_cols = gemv_t_band_cols(es);
    const int n_bands = (int)((cols + band_cols - 1) / band_cols);
    const int grid = gemv_t_grid((int)rows, n_bands);
    GemvTArgs a = {};
    a.a0 = static_cast<const char *>(A);
    a.row_stride = cols * es;
    a.K = (int)rows;
    a.sub_cols = (int)cols;
    a.n_bands = n_bands;
    a.x = x;
    a.err = reinterpret_cast<int *>(ws);
    a.counters = reinterpret_cast<int *>(ws + kWsHeader);
    a.partials = reinterpret_cast<float *>(ws + kWsHeader + align_up((size_t)n_bands * 4, 256));
    a.y = y;
    if (!gemv_t_make_maps(a, a_dtype)) return DS_CUDA_ERROR;
    e = launch_gemv_t(a, a_dtype, PRO_PLAIN, EPI_STORE, grid, s, false);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

}  // namespace ds

extern "C" DS_API int ds_gemv_transposed(const void *A, int64_t a_len, int a_dtype, const float *x,
                                         int64_t x_len, int64_t rows, int64_t cols, float *y,
                                         int64_t y_len, void *workspace, size_t workspace_bytes,
                                         ds_stream_t stream) {
    int st = check_matvec(A, a_len, a_dtype, x, x_len, rows, cols, y, y_len, rows, cols);
    if (st != DS_OK) return st;
    const size_t need = ds_gemv_workspace_bytes(rows, cols, a_dtype);
    if (!workspace || workspace_bytes < need) return DS_WORKSPACE_TOO_SMALL;
    if ((uintptr_t)workspace & 255) return DS_BAD_ARGUMENT;
    return gemv_transposed_run(A, a_dtype, x, rows, cols, y, static_cast<char *>(workspace),
                               reinterpret_cast<cudaStream_t>(stream));
}

extern "C" DS_API int ds_gemv(const void *W, int64_t w_len, int w_dtype, const float *x, int64_t x_len,
                              int64_t rows, int64_t cols, float *y, int64_t y_len, ds_stream_t stream) {
    int st = check_matvec(W, w_len, w_dtype, x, x_len, rows, cols, y, y_len, cols, rows);
    if (st != DS_OK) return st;
    const int es = w_dtype == DS_BF16 ? 2 : 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!gemv_n_streamable(W, (int)rows, (int)cols, es)) {
        const int threads = 256, warps = threads / 32;
        const int blocks = (int)((rows + warps - 1) / warps);
        if (w_dtype == DS_BF16)
            e = launch_ex(gemv_n_plain_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, s, false,
                          (const __nv_bfloat16 *)W, x, (int)rows, (int)cols, y);
        else
            e = launch_ex(gemv_n_plain_kernel<float>, dim3(blocks), dim3(threads), 0, s, false,
                          (const float *)W, x, (int)rows, (int)cols, y);
        return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
    }
    GemvNArgs a = {};
    a.W = static_cast<const char *>(W);
    a.rows = (int)rows;
    a.cols = (int)cols;
    a.x = x;
    a.y = y;
    a.do_argmax = 0;
    e = launch_gemv_n(a, w_dtype, PRO_PLAIN, gemv_n_grid((int)rows, (int)cols, es), s, false);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}
