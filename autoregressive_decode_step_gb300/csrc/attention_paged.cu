// Grouped-query decode attention over a paged K/V pool, streamed a block at
// a time ("Inside the engine", section 1: flash attention over each
// sequence's K/V, split across the context and reduced; section 3: the K/V
// pool of blocks, one K and one V buffer per layer; "The forward pass end to
// end", "The code": forward_token's attention).
//
// The work is the list of every sequence's cache blocks (block_tokens = 16
// positions), cut into equal contiguous ranges, one per CTA, so every CTA
// streams the same number of K/V bytes whatever the mix of context lengths.
// A block's K rows (16 positions x n_kvh heads x 128 dims) are contiguous in
// the layer's K buffer, as are its V rows; a producer warp moves each with
// one bulk asynchronous copy into a ring of shared-memory stages (K stage,
// then V stage).  Consumer warp g serves KV head g and its GQ query heads:
// lane (s, half) owns dims 8s..8s+7 of all GQ heads and positions 8 half ..
// 8 half + 7 of the block.  Scores are summed over the 16 lanes of a half by
// a halving butterfly (each step trades half of the partial sums with the
// partner lane), leaving every lane two finished dot products; the block's
// softmax weights go through a small per-warp table to the lanes that apply
// them to V.  Each warp keeps an online softmax (running max, sum,
// rescaled accumulator) per query head.
//
// When a CTA's range leaves a sequence it publishes, per KV head, its
// (max, sum, accumulator) record; the last contributor of a (sequence, KV
// head) — an atomic counter, never a wait — merges the records of the CTAs
// that covered the sequence in CTA order and writes the output rows (fp32,
// and the bf16 pair hi + lo for the tensor-core output projection).  Every
// mbarrier wait is bounded.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kPaBt = 16;            // positions per block
constexpr int kPaHd = 128;           // head dimension this kernel serves
constexpr int kPaMaxKvh = 8;
constexpr int kPaMaxSeqs = 256;
constexpr size_t kPaSmemLimit = 227 * 1024 - 4096;  // dynamic part: the kernel has 3 KB of static shared memory
constexpr int kPaRingBytes = 192 * 1024;

struct PaSeqs {
    int n_ctx[kPaMaxSeqs];
    int first[kPaMaxSeqs + 1];  // first unit (block) of each sequence in the flattened list
};

// Butterfly step: of the 2N values v, this lane keeps the half selected by
// `upper` and adds the partner's copy of it.
template <int N>
__device__ __forceinline__ void fold(float (&v)[2 * N], float (&out)[N], int dist, bool upper) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float send = upper ? v[i] : v[i + N];
        const float keep = upper ? v[i + N] : v[i];
        out[i] = keep + __shfl_xor_sync(0xffffffffu, send, dist);
    }
}

template <typename KT, int GQ>
__global__ void __launch_bounds__(kPaMaxKvh * 32 + 32, 1) paged_attention_kernel(const __grid_constant__ PagedAttnArgs p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    constexpr int ES = sizeof(KT);
    const int n_kvh = p.n_kvh;
    const int row_bytes = n_kvh * kPaHd * ES;
    const int stage_bytes = kPaBt * row_bytes;  // one block of K (or V)
    const int stages = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + 16;
    __shared__ PaSeqs sq;
    __shared__ int s_abort_raw;
    volatile int &s_abort = s_abort_raw;
    // per consumer warp: the block's softmax weights [16 positions][GQ]
    float *ptab = reinterpret_cast<float *>(empty + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int consumer_warps = n_kvh;
    const int G = gridDim.x;

    allow_dependent_launch();
    grid_dependency_wait();

    // every thread block derives the flattened block list from the lengths
    if (warp == 0) {
        const int cap = p.max_blocks * kPaBt;
        int carry = 0;
        for (int s0 = 0; s0 < p.n_seqs; s0 += 32) {
            const int s = s0 + lane;
            int n_ctx = 0, nb = 0;
            if (s < p.n_seqs) {
                n_ctx = p.seq_lens ? p.seq_lens[s] : p.pos[s] + 1;
                if (n_ctx < 1 || n_ctx > cap) {
                    if (blockIdx.x == 0) flag_error(p.err, DS_ERR_POSITION);
                    n_ctx = min(max(n_ctx, 1), cap);
                }
                nb = (n_ctx + kPaBt - 1) / kPaBt;
                sq.n_ctx[s] = n_ctx;
            }
            int incl = nb;  // inclusive scan over the warp
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (s < p.n_seqs) sq.first[s] = carry + incl - nb;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sq.first[p.n_seqs] = carry;
            s_abort = 0;
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], consumer_warps);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    const long long T = sq.first[p.n_seqs];
    // only min(grid, blocks) CTAs take part, so that every one has a non-empty
    // range and the contributors to a sequence are consecutive CTAs
    const int Ge = (int)min((long long)G, T);
    const bool in = (int)blockIdx.x < Ge;
    const long long u0 = in ? T * blockIdx.x / Ge : 0, u1 = in ? T * (blockIdx.x + 1) / Ge : 0;
    // the sequence holding unit u (sequences are in unit order)
    auto seq_of = [&](long long u) {
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sq.first[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };

    if (warp == consumer_warps) {
        // ------------------------------------------------ producer
        if (lane == 0 && u0 < u1) {
            const uint64_t pol = policy_evict_first();
            uint32_t fill = 0;
            int s = seq_of(u0);
            for (long long u = u0; u < u1; ++u) {
                while (u >= sq.first[s + 1]) ++s;
                const int b = (int)(u - sq.first[s]);
                const long long blk = p.block_table ? (long long)__ldg(p.block_table + (long long)s * p.max_blocks + b)
                                                    : (long long)s * p.max_blocks + b;
                bool ok = blk >= 0 && (blk + 1) * kPaBt <= p.cache_rows;
                if (!ok) flag_error(p.err, DS_ERR_POSITION);
                const char *src[2] = {static_cast<const char *>(p.k_cache), static_cast<const char *>(p.v_cache)};
                for (int kv = 0; kv < 2; ++kv, ++fill) {
                    const int st = fill % stages;
                    const uint32_t use = fill / stages;
                    if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1, p.err)) {
                        s_abort = 1;
                        goto drain;
                    }
                    mbar_arrive_expect_tx(&full[st], (uint32_t)stage_bytes);
                    // a block outside the pool is not copied: block 0 stands in (its
                    // values are never used: the flag above marks the step bad)
                    bulk_g2s(smem + (size_t)st * stage_bytes, src[kv] + (ok ? blk : 0) * (long long)stage_bytes,
                             (uint32_t)stage_bytes, &full[st], pol);
                }
            }
        drain:
            // every copy issued has landed before the CTA may exit
            const uint32_t first = fill > (uint32_t)stages ? fill - stages : 0;
            for (uint32_t f = first; f < fill; ++f)
                if (!mbar_wait(&full[f % stages], (f / stages) & 1, p.err)) break;
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int g = warp;             // KV head of this warp
    const int sl = lane & 15;       // dims 8 sl .. 8 sl + 7
    const int half = lane >> 4;     // positions 8 half .. 8 half + 7 of a block
    const float scale = p.scale;
    const int rec = kPaHd + 2;      // per query head: m, l, acc[128]
    float *my_ptab = ptab + warp * kPaBt * GQ;
    uint32_t fill = 0;
    float q[GQ][8], acc[GQ][8], m[GQ], l[GQ];
    int s = u0 < u1 ? seq_of(u0) : 0;
    long long u = u0;
    while (u < u1) {
        while (u >= sq.first[s + 1]) ++s;
        const long long seg_end = min(u1, (long long)sq.first[s + 1]);
        const int n_ctx = sq.n_ctx[s];
        // this sequence's query rows of KV head g, dims 8 sl ..
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            const float *qr = p.q + ((long long)s * p.n_qh + g * GQ + j) * kPaHd + sl * 8;
            const float4 a = __ldg(reinterpret_cast<const float4 *>(qr));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(qr + 4));
            q[j][0] = a.x; q[j][1] = a.y; q[j][2] = a.z; q[j][3] = a.w;
            q[j][4] = b.x; q[j][5] = b.y; q[j][6] = b.z; q[j][7] = b.w;
            m[j] = -INFINITY;
            l[j] = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
        }
        for (; u < seg_end; ++u) {
            const int b = (int)(u - sq.first[s]);
            const int valid = min(kPaBt, n_ctx - b * kPaBt);  // positions of this block in the context
            // ---- K stage: scores of this lane's 8 positions for the GQ heads
            int st = fill % stages;
            bool ok = !s_abort && mbar_wait(&full[st], (fill / stages) & 1, p.err);
            if (!ok) s_abort = 1;
            float part[GQ * 8];
            {
                const unsigned char *base = smem + (size_t)st * stage_bytes + (size_t)g * kPaHd * ES + sl * 8 * ES;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const unsigned char *rowp = base + (size_t)(half * 8 + i) * row_bytes;
                    float k[8];
                    if (ES == 2) {
                        widen16(*reinterpret_cast<const uint4 *>(rowp), k);
                    } else {
                        const float4 a = *reinterpret_cast<const float4 *>(rowp);
                        const float4 c = *reinterpret_cast<const float4 *>(rowp + 16);
                        k[0] = a.x; k[1] = a.y; k[2] = a.z; k[3] = a.w;
                        k[4] = c.x; k[5] = c.y; k[6] = c.z; k[7] = c.w;
                    }
#pragma unroll
                    for (int j = 0; j < GQ; ++j) {
                        float d = 0.0f;
#pragma unroll
                        for (int e = 0; e < 8; ++e) d = fmaf(q[j][e], k[e], d);
                        part[j * 8 + i] = d;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            ++fill;
            // halving butterfly over the 16 lanes of this half: lane sl ends
            // with the dot products v = (GQ / 2) sl .. (GQ / 2) sl + GQ/2 - 1
            // of the GQ x 8 (head j = v / 8, position i = v % 8)
            constexpr int NV = GQ * 8;
            float r[NV / 16];
            {
                float a8[NV / 2], a4[NV / 4], a2[NV / 8];
                fold<NV / 2>(part, a8, 8, (sl & 8) != 0);
                fold<NV / 4>(a8, a4, 4, (sl & 4) != 0);
                fold<NV / 8>(a4, a2, 2, (sl & 2) != 0);
                fold<NV / 16>(a2, r, 1, (sl & 1) != 0);
            }
            // scores (masked past the context), block max per head
            constexpr int R = NV / 16;
            const int v0 = R * sl;
            float sc[R];
            float bmax[GQ];
#pragma unroll
            for (int j = 0; j < GQ; ++j) bmax[j] = -INFINITY;
#pragma unroll
            for (int t = 0; t < R; ++t) {
                const int v = v0 + t, j = v / 8, i = v % 8;
                const bool in = half * 8 + i < valid;
                sc[t] = in ? r[t] * scale : -INFINITY;
#pragma unroll
                for (int jj = 0; jj < GQ; ++jj)
                    if (jj == j) bmax[jj] = fmaxf(bmax[jj], sc[t]);
            }
            // a head's 16 scores sit in 8 / R lanes of each half: max over them
#pragma unroll
            for (int jj = 0; jj < GQ; ++jj) {
                float x = bmax[jj];
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
                bmax[jj] = x;
            }
            float corr[GQ], bsum[GQ];
#pragma unroll
            for (int jj = 0; jj < GQ; ++jj) {
                const float mn = fmaxf(m[jj], bmax[jj]);
                corr[jj] = mn == -INFINITY ? 1.0f : expf(m[jj] - mn);
                m[jj] = mn;
                bsum[jj] = 0.0f;
            }
#pragma unroll
            for (int t = 0; t < R; ++t) {
                const int v = v0 + t, j = v / 8, i = v % 8;
                float w = 0.0f;
#pragma unroll
                for (int jj = 0; jj < GQ; ++jj)
                    if (jj == j) w = sc[t] == -INFINITY ? 0.0f : expf(sc[t] - m[jj]);
#pragma unroll
                for (int jj = 0; jj < GQ; ++jj)
                    if (jj == j) bsum[jj] += w;
                my_ptab[(half * 8 + i) * GQ + j] = w;
            }
#pragma unroll
            for (int jj = 0; jj < GQ; ++jj) {
                float x = bsum[jj];
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                l[jj] = l[jj] * corr[jj] + x;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[jj][e] *= corr[jj];
            }
            __syncwarp();
            // ---- V stage: acc += w * V over this lane's 8 positions
            st = fill % stages;
            ok = !s_abort && mbar_wait(&full[st], (fill / stages) & 1, p.err);
            if (!ok) s_abort = 1;
            {
                const unsigned char *base = smem + (size_t)st * stage_bytes + (size_t)g * kPaHd * ES + sl * 8 * ES;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int pos = half * 8 + i;
                    if (pos < valid) {  // rows past the context may hold anything
                        const unsigned char *rowp = base + (size_t)pos * row_bytes;
                        float vv[8];
                        if (ES == 2) {
                            widen16(*reinterpret_cast<const uint4 *>(rowp), vv);
                        } else {
                            const float4 a = *reinterpret_cast<const float4 *>(rowp);
                            const float4 c = *reinterpret_cast<const float4 *>(rowp + 16);
                            vv[0] = a.x; vv[1] = a.y; vv[2] = a.z; vv[3] = a.w;
                            vv[4] = c.x; vv[5] = c.y; vv[6] = c.z; vv[7] = c.w;
                        }
#pragma unroll
                        for (int j = 0; j < GQ; ++j) {
                            const float w = my_ptab[pos * GQ + j];
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(w, vv[e], acc[j][e]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            ++fill;
        }
        // ---- the two halves hold disjoint positions under one running max
#pragma unroll
        for (int j = 0; j < GQ; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], 16);
        // this CTA's record for (sequence s, KV head g), slot CTA + sequence
        float *slot = p.partials + ((size_t)blockIdx.x + s) * p.n_qh * rec;
        if (half == 0) {
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                float *rr = slot + (size_t)(g * GQ + j) * rec;
                if (sl == 0) {
                    rr[0] = m[j];
                    rr[1] = l[j];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) rr[2 + sl * 8 + e] = acc[j][e];
            }
        }
        // the CTAs holding this sequence's first and last block
        const long long f0 = sq.first[s], f1 = sq.first[s + 1] - 1;
        const int c_first = (int)(((f0 + 1) * Ge - 1) / T), c_last = (int)(((f1 + 1) * Ge - 1) / T);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            int *ctr = p.counters + (size_t)s * n_kvh + g;
            last = atomicAdd(ctr, 1) == c_last - c_first;
            if (last) *ctr = 0;  // ready for the next launch
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            // merge in CTA order: out = sum_c w_c acc_c / sum_c w_c l_c, w_c = exp(m_c - max m)
            for (int j = 0; j < GQ; ++j) {
                const int h = g * GQ + j;
                float M = -INFINITY;
                for (int c = c_first; c <= c_last; ++c)
                    M = fmaxf(M, __ldcg(p.partials + ((size_t)c + s) * p.n_qh * rec + (size_t)h * rec));
                float L = 0.0f, A[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int c = c_first; c <= c_last; ++c) {
                    const float *rr = p.partials + ((size_t)c + s) * p.n_qh * rec + (size_t)h * rec;
                    const float mc = __ldcg(rr);
                    const float w = mc == -INFINITY ? 0.0f : expf(mc - M);
                    L = fmaf(__ldcg(rr + 1), w, L);
#pragma unroll
                    for (int e = 0; e < 4; ++e) A[e] = fmaf(__ldcg(rr + 2 + lane * 4 + e), w, A[e]);
                }
                const long long o = ((long long)s * p.n_qh + h) * kPaHd + lane * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float r1 = A[e] / L;
                    p.out[o + e] = r1;
                    if (p.out_bf16) {
                        __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(p.out_bf16);
                        const __nv_bfloat16 hi = __float2bfloat16_rn(r1);
                        ob[o + e] = hi;
                        if (p.out_bf16_lo) ob[o + e + p.out_bf16_lo] = __float2bfloat16_rn(r1 - __bfloat162float(hi));
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- host
bool paged_attention_supported(int n_qh, int n_kvh, int hd, int block_tokens, int n_seqs, int kv_dtype) {
    const int gq = n_qh / n_kvh;
    if (hd != kPaHd || block_tokens != kPaBt || n_kvh > kPaMaxKvh || n_seqs > kPaMaxSeqs) return false;
    if (gq != 2 && gq != 4) return false;  // 8 heads per lane would not fit the register file
    const int es = kv_dtype == DS_BF16 ? 2 : 4;
    return kPaBt * n_kvh * kPaHd * es <= kPaRingBytes / 2;  // at least two stages
}

size_t paged_attention_partial_floats(int n_seqs, int n_qh) {
    return (size_t)(sm_count() + n_seqs) * n_qh * (kPaHd + 2);
}

template <typename KT, int GQ>
static cudaError_t launch_pa(PagedAttnArgs a, cudaStream_t stream, bool pdl) {
    const int es = sizeof(KT);
    const int stage_bytes = kPaBt * a.n_kvh * kPaHd * es;
    a.stages = std::min(16, kPaRingBytes / stage_bytes);
    const size_t smem = (size_t)a.stages * stage_bytes + 256 + (size_t)a.n_kvh * kPaBt * GQ * 4;
    if (smem > kPaSmemLimit) return cudaErrorInvalidValue;
    return launch_ex(paged_attention_kernel<KT, GQ>, dim3(sm_count()), dim3(a.n_kvh * 32 + 32), smem, stream, pdl, a);
}

static bool g_pa_ready = false;

cudaError_t prepare_paged_attention() {
    const void *fns[] = {(const void *)paged_attention_kernel<__nv_bfloat16, 2>,
                         (const void *)paged_attention_kernel<__nv_bfloat16, 4>,
                         (const void *)paged_attention_kernel<float, 2>, (const void *)paged_attention_kernel<float, 4>};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPaSmemLimit);
        if (e != cudaSuccess) return e;
    }
    g_pa_ready = true;
    return cudaSuccess;
}

cudaError_t launch_paged_attention(const PagedAttnArgs &a, cudaStream_t stream, bool pdl) {
    if (!g_pa_ready) {
        cudaError_t e = prepare_paged_attention();
        if (e != cudaSuccess) return e;
    }
    const int gq = a.n_qh / a.n_kvh;
    if (a.kv_dtype == DS_BF16) {
        switch (gq) {
            case 2: return launch_pa<__nv_bfloat16, 2>(a, stream, pdl);
            case 4: return launch_pa<__nv_bfloat16, 4>(a, stream, pdl);
        }
    } else {
        switch (gq) {
            case 2: return launch_pa<float, 2>(a, stream, pdl);
            case 4: return launch_pa<float, 4>(a, stream, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace ds
