// Grouped-query decode attention, split across the context and reduced
// ("Inside the engine", section 1: the flash attention over the sequence's
// K/V, split across the context and reduced; "The forward pass end to end",
// "The code": forward_token's attention).
//
// One CTA per (context split, KV head, sequence).  A CTA serves every query
// head of its KV head's group, so each K/V row is fetched once for the whole
// group.  Within a CTA, four warps take interleaved runs of eight positions;
// a lane owns 4 (or 8) consecutive head dimensions, so one K row of a KV head
// is one coalesced 256- or 512-byte read by the warp.  Each warp runs an online
// softmax (running max, running sum, rescaled accumulator) per query head;
// the warps are merged in shared memory and the CTA's partial result goes to
// the workspace.  The last CTA of a (sequence, KV head) — an atomic counter,
// never a wait — merges the splits in split order, so the result does not
// depend on which CTA finishes first.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kAttnWarps = 8;
constexpr int kAttnMaxSplits = 64;
constexpr int kAttnMinPerSplit = 64;  // positions: one run of eight per warp
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnRun = 8;  // positions a warp fetches together

__device__ __forceinline__ long long kv_row(int seq, int t, const int *table, int max_blocks, int bt) {
    const int b = t / bt;
    const long long blk = table ? (long long)table[(long long)seq * max_blocks + b]
                                : (long long)seq * max_blocks + b;
    return blk * bt + t % bt;
}

template <typename KT, int DPL>
__device__ __forceinline__ void load_dims(const KT *base, long long off, bool active, float (&f)[DPL]) {
    if (!active) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) f[e] = 0.0f;
        return;
    }
    if (sizeof(KT) == 2) {
        if (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(base + off);
            f[0] = __uint_as_float(w.x << 16);
            f[1] = __uint_as_float(w.x & 0xffff0000u);
            f[2] = __uint_as_float(w.y << 16);
            f[3] = __uint_as_float(w.y & 0xffff0000u);
        } else {
            const uint4 w = *reinterpret_cast<const uint4 *>(base + off);
            float g[8];
            widen16(w, g);
#pragma unroll
            for (int e = 0; e < DPL; ++e) f[e] = g[e];
        }
    } else {
#pragma unroll
        for (int e = 0; e < DPL; e += 4) {
            const float4 w = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + off + e);
            f[e] = w.x;
            f[e + 1] = w.y;
            f[e + 2] = w.z;
            f[e + 3] = w.w;
        }
    }
}

template <typename KT, int DPL, int GQ>
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const __grid_constant__ AttnArgs p) {
    const int split = blockIdx.x, g = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hd = p.hd;
    __shared__ float s_m[kAttnWarps][GQ], s_l[kAttnWarps][GQ];
    extern __shared__ float s_acc[];  // [kAttnWarps][GQ][hd]
    __shared__ int s_last;

    allow_dependent_launch();
    grid_dependency_wait();

    const int cap = p.max_blocks * p.block_tokens;
    const int cseq = p.row_seq ? p.row_seq[seq] : seq;  // whose blocks this row reads
    int n_ctx = p.seq_lens ? p.seq_lens[seq] : p.pos[seq] + 1;
    if (n_ctx < 1 || n_ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && g == 0) flag_error(p.err, DS_ERR_POSITION);
        n_ctx = min(max(n_ctx, 1), cap);
    }
    // positions per split, never fewer than kAttnMinPerSplit; splits past the
    // context (split >= n_eff) have no work and write no partial
    const int per = max(kAttnMinPerSplit, (n_ctx + p.n_splits - 1) / p.n_splits);
    const int n_eff = (n_ctx + per - 1) / per;
    const int t0 = min(n_ctx, split * per), t1 = min(n_ctx, t0 + per);

    const bool active = lane * DPL < hd;
    const long long row_elems = (long long)p.n_kvh * hd;
    const int d0 = lane * DPL;
    const KT *kc = static_cast<const KT *>(p.k_cache);
    const KT *vc = static_cast<const KT *>(p.v_cache);

    float q[GQ][DPL];
#pragma unroll
    for (int j = 0; j < GQ; ++j)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            q[j][e] = active ? p.q[((long long)seq * p.n_qh + g * GQ + j) * hd + d0 + e] : 0.0f;

    float m[GQ], l[GQ], acc[GQ][DPL];
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.0f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[j][e] = 0.0f;
    }

    for (int tb = t0 + warp * kAttnRun; tb < t1; tb += kAttnWarps * kAttnRun) {
        const int nt = min(kAttnRun, t1 - tb);
        float kf[kAttnRun][DPL], vf[kAttnRun][DPL];
#pragma unroll
        for (int i = 0; i < kAttnRun; ++i) {
            const bool ok = active && i < nt;
            const long long off = ok ? kv_row(cseq, tb + i, p.block_table, p.max_blocks, p.block_tokens) * row_elems +
                                           (long long)g * hd + d0
                                     : 0;
            load_dims<KT, DPL>(kc, off, ok, kf[i]);
            load_dims<KT, DPL>(vc, off, ok, vf[i]);
        }
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            float sc[kAttnRun];
#pragma unroll
            for (int i = 0; i < kAttnRun; ++i) {
                float d = 0.0f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) d = fmaf(q[j][e], kf[i][e], d);
                sc[i] = warp_sum(d) * p.scale;
            }
            float mx = m[j];
#pragma unroll
            for (int i = 0; i < kAttnRun; ++i)
                if (i < nt) mx = fmaxf(mx, sc[i]);
            const float corr = expf(m[j] - mx);
            l[j] *= corr;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[j][e] *= corr;
#pragma unroll
            for (int i = 0; i < kAttnRun; ++i) {
                if (i < nt) {
                    const float w = expf(sc[i] - mx);
                    l[j] += w;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[j][e] = fmaf(w, vf[i][e], acc[j][e]);
                }
            }
            m[j] = mx;
        }
    }

    // merge the warps of this CTA
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
        if (lane == 0) {
            s_m[warp][j] = m[j];
            s_l[warp][j] = l[j];
        }
        if (active)
#pragma unroll
            for (int e = 0; e < DPL; ++e) s_acc[(warp * GQ + j) * hd + d0 + e] = acc[j][e];
    }
    __syncthreads();

    const int slot = (seq * p.n_kvh + g) * p.n_splits + split;
    const int rec = GQ * (hd + 2);  // per split: m[GQ], l[GQ], acc[GQ][hd]
    float *part = p.partials + (size_t)slot * rec;
    for (int idx = threadIdx.x; split < n_eff && idx < GQ * hd; idx += kAttnThreads) {
        const int j = idx / hd;
        float M = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][j]);
        float L = 0.0f, A = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < kAttnWarps; ++w) {
                const float c = expf(s_m[w][j] - M);
                L = fmaf(s_l[w][j], c, L);
                A = fmaf(s_acc[(w * GQ + j) * hd + idx % hd], c, A);
            }
        }
        part[2 * GQ + idx] = A;
        if (idx % hd == 0) {
            part[j] = M;
            part[GQ + j] = L;
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        int *ctr = &p.counters[seq * p.n_kvh + g];
        s_last = atomicAdd(ctr, 1) == p.n_splits - 1;
        if (s_last) *ctr = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // merge the n_eff splits in split order.  All (m, l) are staged in shared
    // memory by parallel loads, the weights exp(m_s - M) computed in
    // parallel, then every output is one fixed-order sum over the splits
    // (two outputs per thread, their loads interleaved).
    const float *base = p.partials + (size_t)(seq * p.n_kvh + g) * p.n_splits * rec;
    float *sm = s_acc;                          // [n_eff][GQ] m, then weights
    float *sl = s_acc + kAttnMaxSplits * GQ;    // [n_eff][GQ] l
    float *sM = sl + kAttnMaxSplits * GQ;       // [GQ] max, then [GQ] total
    for (int i = threadIdx.x; i < n_eff * GQ; i += kAttnThreads) {
        const int sp = i / GQ, j = i % GQ;
        sm[i] = __ldcg(base + (size_t)sp * rec + j);
        sl[i] = __ldcg(base + (size_t)sp * rec + GQ + j);
    }
    __syncthreads();
    if (threadIdx.x < GQ) {
        float M = -INFINITY;
        for (int sp = 0; sp < n_eff; ++sp) M = fmaxf(M, sm[sp * GQ + threadIdx.x]);
        sM[threadIdx.x] = M;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_eff * GQ; i += kAttnThreads) {
        const float ms = sm[i];
        sm[i] = ms == -INFINITY ? 0.0f : expf(ms - sM[i % GQ]);
    }
    __syncthreads();
    if (threadIdx.x < GQ) {
        float L = 0.0f;
        for (int sp = 0; sp < n_eff; ++sp) L = fmaf(sl[sp * GQ + threadIdx.x], sm[sp * GQ + threadIdx.x], L);
        sM[GQ + threadIdx.x] = L;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < GQ * hd; idx += 2 * kAttnThreads) {
        const int idx2 = idx + kAttnThreads;
        const bool two = idx2 < GQ * hd;
        const int j = idx / hd, j2 = two ? idx2 / hd : j;
        float A = 0.0f, A2 = 0.0f;
#pragma unroll 8
        for (int sp = 0; sp < n_eff; ++sp) {
            const float *rp = base + (size_t)sp * rec + 2 * GQ;
            const float a = __ldcg(rp + idx);
            const float a2 = two ? __ldcg(rp + idx2) : 0.0f;
            A = fmaf(a, sm[sp * GQ + j], A);
            A2 = fmaf(a2, sm[sp * GQ + j2], A2);
        }
        const long long o1 = ((long long)seq * p.n_qh + g * GQ + j) * hd + idx % hd;
        const long long o2 = ((long long)seq * p.n_qh + g * GQ + j2) * hd + idx2 % hd;
        const float r1 = A / sM[GQ + j], r2 = A2 / sM[GQ + j2];
        p.out[o1] = r1;
        if (two) p.out[o2] = r2;
        if (p.out_bf16) {  // hi + lo pair: r = hi + lo to 16 significant bits
            __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(p.out_bf16);
            const __nv_bfloat16 h1 = __float2bfloat16_rn(r1);
            ob[o1] = h1;
            if (p.out_bf16_lo) ob[o1 + p.out_bf16_lo] = __float2bfloat16_rn(r1 - __bfloat162float(h1));
            if (two) {
                const __nv_bfloat16 h2 = __float2bfloat16_rn(r2);
                ob[o2] = h2;
                if (p.out_bf16_lo) ob[o2 + p.out_bf16_lo] = __float2bfloat16_rn(r2 - __bfloat162float(h2));
            }
        }
    }
}

int attention_splits(int n_seqs, int n_kvh, long long max_ctx) {
    // about two CTAs per SM in all, at least kAttnMinPerSplit positions per
    // split at the largest context, at most kAttnMaxSplits splits
    const long long target = 2LL * sm_count();
    long long s = (target + (long long)n_seqs * n_kvh - 1) / ((long long)n_seqs * n_kvh);
    const long long by_ctx = (max_ctx + kAttnMinPerSplit - 1) / kAttnMinPerSplit;
    s = std::min(std::min(s, by_ctx), (long long)kAttnMaxSplits);
    return (int)std::max(1LL, s);
}

size_t attention_partial_floats(int n_seqs, int n_qh, int n_kvh, int hd, int n_splits) {
    const int gq = n_qh / n_kvh;
    return (size_t)n_seqs * n_kvh * n_splits * gq * (hd + 2);
}

template <typename KT, int DPL>
static cudaError_t launch_attn_g(const AttnArgs &a, int n_seqs, cudaStream_t stream, bool pdl) {
    const int gq = a.n_qh / a.n_kvh;
    const dim3 grid(a.n_splits, a.n_kvh, n_seqs);
    const size_t smem = std::max((size_t)kAttnWarps * gq * a.hd, (size_t)(2 * kAttnMaxSplits + 2) * gq) * sizeof(float);
    switch (gq) {
        case 1: return launch_ex(attention_kernel<KT, DPL, 1>, grid, dim3(kAttnThreads), smem, stream, pdl, a);
        case 2: return launch_ex(attention_kernel<KT, DPL, 2>, grid, dim3(kAttnThreads), smem, stream, pdl, a);
        case 4: return launch_ex(attention_kernel<KT, DPL, 4>, grid, dim3(kAttnThreads), smem, stream, pdl, a);
        case 8: return launch_ex(attention_kernel<KT, DPL, 8>, grid, dim3(kAttnThreads), smem, stream, pdl, a);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention(const AttnArgs &a, int n_seqs, cudaStream_t stream, bool pdl) {
    const bool wide = a.hd > 128;
    if (a.kv_dtype == DS_BF16)
        return wide ? launch_attn_g<__nv_bfloat16, 8>(a, n_seqs, stream, pdl)
                    : launch_attn_g<__nv_bfloat16, 4>(a, n_seqs, stream, pdl);
    return wide ? launch_attn_g<float, 8>(a, n_seqs, stream, pdl) : launch_attn_g<float, 4>(a, n_seqs, stream, pdl);
}

}  // namespace ds

using namespace ds;

extern "C" DS_API size_t ds_attention_workspace_bytes(int n_seqs, int n_qh, int n_kvh, int head_dim,
                                                      int64_t max_ctx) {
    if (n_seqs < 1 || n_kvh < 1 || n_qh < n_kvh || head_dim < 1 || max_ctx < 1) return 0;
    const int splits = attention_splits(n_seqs, n_kvh, max_ctx);
    const size_t partial = std::max(attention_partial_floats(n_seqs, n_qh, n_kvh, head_dim, splits),
                                    paged_attention_partial_floats(n_seqs, n_qh));
    return kWsHeader + align_up((size_t)n_seqs * n_kvh * 4, 256) + partial * 4;
}

extern "C" DS_API int ds_gqa_decode_attn(const float *q, const void *k_cache, const void *v_cache,
                                         int kv_dtype, int64_t cache_rows, const int32_t *block_table,
                                         int max_blocks_per_seq, int block_tokens, const int32_t *seq_lens,
                                         int n_seqs, int n_qh, int n_kvh, int head_dim, float scale,
                                         float *out, void *workspace, size_t workspace_bytes,
                                         ds_stream_t stream) {
    if (n_seqs < 1 || n_qh < 1 || n_kvh < 1 || head_dim < 1 || block_tokens < 1 || max_blocks_per_seq < 1 ||
        cache_rows < 1)
        return DS_EMPTY_DIMENSION;
    if (n_seqs > DS_MAX_DIM || cache_rows > DS_MAX_DIM || (int64_t)max_blocks_per_seq * block_tokens > DS_MAX_DIM)
        return DS_DIMENSION_TOO_LARGE;
    if (kv_dtype != DS_F32 && kv_dtype != DS_BF16) return DS_BAD_DTYPE;
    const int gq = n_qh / n_kvh;
    if (n_qh % n_kvh || (gq != 1 && gq != 2 && gq != 4 && gq != 8) || head_dim % 4 || head_dim > 256 ||
        (head_dim > 128 && head_dim % 8))
        return DS_BAD_ARGUMENT;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return DS_BAD_ARGUMENT;
    const int es = kv_dtype == DS_BF16 ? 2 : 4;
    if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15 || ((uintptr_t)q & 15)) return DS_BAD_ARGUMENT;
    if (((int64_t)head_dim * es) % 8) return DS_BAD_ARGUMENT;
    // every addressable row must exist: contiguous slots need n_seqs*max_blocks blocks
    if (!block_table && (int64_t)n_seqs * max_blocks_per_seq * block_tokens > cache_rows)
        return DS_CACHE_CAPACITY_EXCEEDED;
    const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_tokens;
    const size_t need = ds_attention_workspace_bytes(n_seqs, n_qh, n_kvh, head_dim, max_ctx);
    if (!workspace || workspace_bytes < need) return DS_WORKSPACE_TOO_SMALL;
    if ((uintptr_t)workspace & 255) return DS_BAD_ARGUMENT;
    char *ws = static_cast<char *>(workspace);
    if (paged_attention_supported(n_qh, n_kvh, head_dim, block_tokens, n_seqs, kv_dtype)) {
        // whole 16-position blocks streamed through shared memory, work split evenly over the SMs
        PagedAttnArgs pa = {};
        pa.q = q;
        pa.k_cache = k_cache;
        pa.v_cache = v_cache;
        pa.kv_dtype = kv_dtype;
        pa.cache_rows = cache_rows;
        pa.block_table = block_table;
        pa.max_blocks = max_blocks_per_seq;
        pa.seq_lens = seq_lens;
        pa.n_seqs = n_seqs;
        pa.n_qh = n_qh;
        pa.n_kvh = n_kvh;
        pa.scale = scale;
        pa.out = out;
        pa.err = reinterpret_cast<int *>(ws);
        pa.counters = reinterpret_cast<int *>(ws + kWsHeader);
        pa.partials = reinterpret_cast<float *>(ws + kWsHeader + align_up((size_t)n_seqs * n_kvh * 4, 256));
        if (kv_dtype == DS_BF16 && !paged_attention_maps(pa)) return DS_CUDA_ERROR;
        cudaError_t e = launch_paged_attention(pa, reinterpret_cast<cudaStream_t>(stream), false);
        return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
    }
    AttnArgs a = {};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.kv_dtype = kv_dtype;
    a.cache_rows = cache_rows;
    a.block_table = block_table;
    a.max_blocks = max_blocks_per_seq;
    a.block_tokens = block_tokens;
    a.seq_lens = seq_lens;
    a.n_qh = n_qh;
    a.n_kvh = n_kvh;
    a.hd = head_dim;
    a.scale = scale;
    a.out = out;
    a.err = reinterpret_cast<int *>(ws);
    a.counters = reinterpret_cast<int *>(ws + kWsHeader);
    a.partials = reinterpret_cast<float *>(ws + kWsHeader + align_up((size_t)n_seqs * n_kvh * 4, 256));
    a.n_splits = attention_splits(n_seqs, n_kvh, max_ctx);
    cudaError_t e = launch_attention(a, n_seqs, reinterpret_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}
