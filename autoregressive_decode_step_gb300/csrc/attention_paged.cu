// Grouped-query decode attention over a paged K/V pool, streamed a block at
// a time ("Inside the engine", section 1: flash attention over each
// sequence's K/V, split across the context and reduced; section 3: the K/V
// pool of blocks, one K and one V buffer per layer; "The forward pass end to
// end", "The code": forward_token's attention).
//
// The work is the list of every sequence's cache blocks (block_tokens = 16
// positions), cut into equal contiguous ranges, one per CTA (about 16 blocks
// a CTA, 8 to 64 CTAs per sequence), so every CTA streams the same number of
// K/V bytes whatever the mix of context lengths.
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
#include "tc.h"

namespace ds {

constexpr int kPaBt = 16;            // positions per block
constexpr int kPaHd = 128;           // head dimension this kernel serves
constexpr int kPaMaxKvh = 8;
constexpr int kPaMaxSeqs = 256;
constexpr size_t kPaSmemLimit = 227 * 1024 - 4096;  // dynamic part: the kernel has 3 KB of static shared memory
constexpr int kPaRingBytes = 192 * 1024;
// Bounds on the CTAs a launch spreads its blocks over (pa_ctas)
constexpr int kPaMinCtasPerSeq = 8;
constexpr int kPaMaxCtasPerSeq = 64;
constexpr int kPaBlocksPerCta = 16;

// CTAs a launch over n_seqs sequences of T blocks in all takes part with:
// about kPaBlocksPerCta blocks per CTA, at least kPaMinCtasPerSeq and at most
// kPaMaxCtasPerSeq per sequence, at most the grid (few sequences then keep
// the merge of their per-CTA records short; many fill the grid).
__device__ __forceinline__ int pa_ctas(int G, long long T, int n_seqs) {
    long long g = T / kPaBlocksPerCta;
    g = max(g, (long long)n_seqs * kPaMinCtasPerSeq);
    g = min(g, (long long)n_seqs * kPaMaxCtasPerSeq);
    g = min(g, T);
    return (int)max(1ll, min(g, (long long)G));
}

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

// After a CTA has written its record for (sequence s, KV head g) into slot
// CTA + s: count the arrival; the last of the CTAs that covered the sequence
// (those holding its units f0 .. f1) merges the records in CTA order,
// out = sum_c w_c acc_c / sum_c w_c l_c with w_c = exp(m_c - max m), and
// writes the output rows (fp32, and the bf16 pair hi + lo when asked).
template <int GQ>
__device__ void pa_finish_sequence(const PagedAttnArgs &p, int s, int g, long long f0, long long f1, int Ge,
                                   long long T) {
    const int lane = threadIdx.x & 31;
    const int rec = kPaHd + 2;
    const int c_first = (int)(((f0 + 1) * Ge - 1) / T), c_last = (int)(((f1 + 1) * Ge - 1) / T);
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        int *ctr = p.counters + (size_t)s * p.n_kvh + g;
        last = atomicAdd(ctr, 1) == c_last - c_first;
        if (last) *ctr = 0;  // ready for the next launch
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    for (int j = 0; j < GQ; ++j) {
        const int h = g * GQ + j;
        auto rec_of = [&](int c) { return p.partials + ((size_t)c + s) * p.n_qh * rec + (size_t)h * rec; };
        // the largest record max: lanes read contributors 32 apart, then a
        // warp max (exact whatever the order)
        float M = -INFINITY;
        for (int c = c_first + lane; c <= c_last; c += 32) M = fmaxf(M, __ldcg(rec_of(c)));
        M = warp_max(M);
        // sum and accumulator in CTA order, eight contributors' loads in flight
        float L = 0.0f, A[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int c0 = c_first; c0 <= c_last; c0 += 8) {
            float mc[8], lc[8];
            float4 ac[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                mc[k] = -INFINITY;
                lc[k] = 0.0f;
                ac[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (c0 + k <= c_last) {
                    const float *rr = rec_of(c0 + k);
                    mc[k] = __ldcg(rr);
                    lc[k] = __ldcg(rr + 1);
                    ac[k] = make_float4(__ldcg(rr + 2 + lane * 4), __ldcg(rr + 3 + lane * 4), __ldcg(rr + 4 + lane * 4),
                                        __ldcg(rr + 5 + lane * 4));
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (c0 + k > c_last) break;
                const float w = mc[k] == -INFINITY ? 0.0f : expf(mc[k] - M);
                L = fmaf(lc[k], w, L);
                A[0] = fmaf(ac[k].x, w, A[0]);
                A[1] = fmaf(ac[k].y, w, A[1]);
                A[2] = fmaf(ac[k].z, w, A[2]);
                A[3] = fmaf(ac[k].w, w, A[3]);
            }
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

// The flattened block list of a launch: every CTA reads the sequence lengths
// (seq_lens, else pos + 1, clamped to the cache and flagged when outside it)
// and forms the prefix sums of their block counts.  Warp 0 does the scan.
__device__ void pa_block_list(const PagedAttnArgs &p, PaSeqs &sq) {
    const int lane = threadIdx.x & 31;
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
    if (lane == 0) sq.first[p.n_seqs] = carry;
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
        pa_block_list(p, sq);
        if (lane == 0) s_abort = 0;
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
    const int Ge = pa_ctas(G, T, p.n_seqs);
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
                const long long cs = p.row_seq ? __ldg(p.row_seq + s) : s;
                const long long blk = p.block_table ? (long long)__ldg(p.block_table + cs * p.max_blocks + b)
                                                    : cs * p.max_blocks + b;
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
        pa_finish_sequence<GQ>(p, s, g, sq.first[s], sq.first[s + 1] - 1, Ge, T);
    }
}


// ------------------------------------------------------------------ tensor-core variant (bf16 caches)
// The same work split and merge, with the two products of a block on the
// tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulators):
//   scores   S^T[16 positions][8] = K[16 x 128] . Q^T[128 x 8]
//   output   O^T[128][8]         += V^T[128 x 16] . P^T[16 x 8]
// The 8 columns hold the GQ query heads twice: their bf16 "hi" parts and,
// GQ columns further, the "lo" remainders (hi + lo = the fp32 value to 16
// significant bits), so q and the softmax weights P keep fp32-like precision
// and a column pair is summed after each product.  K and V arrive per head as
// two 64-dim x 16-position boxes with 128-byte swizzling, which ldmatrix
// reads without bank conflicts (.trans for V^T).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo_elem, __nv_bfloat16 hi_elem) {
    return (uint32_t)__bfloat16_as_ushort(lo_elem) | ((uint32_t)__bfloat16_as_ushort(hi_elem) << 16);
}
// Byte offset, within a stage, of dims d..d+7 of position pos of head g: two
// 2 KB boxes per head (dims 0-63, 64-127), rows of 128 bytes whose 16-byte
// chunks are swizzled by the row index.
__device__ __forceinline__ uint32_t pa_swz(int g, int pos, int d) {
    const int half = d >> 6, c = (d & 63) >> 3;
    return (uint32_t)(g * 4096 + half * 2048 + pos * 128 + ((c ^ (pos & 7)) << 4));
}

template <int GQ>
__global__ void __launch_bounds__(kPaMaxKvh * 32 + 32, 1) paged_attention_tc_kernel(const __grid_constant__ PagedAttnArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int n_kvh = p.n_kvh;
    const int stage_bytes = n_kvh * 4096;  // 16 positions x n_kvh heads x 128 dims of bf16
    const int stages = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + 16;
    __nv_bfloat16 *ptab_all = reinterpret_cast<__nv_bfloat16 *>(empty + 16);  // per warp [8 columns][16 positions]
    __shared__ PaSeqs sq;
    __shared__ int s_abort_raw;
    volatile int &s_abort = s_abort_raw;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;

    allow_dependent_launch();
    grid_dependency_wait();
    if (warp == 0) {
        pa_block_list(p, sq);
        if (lane == 0) s_abort = 0;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], n_kvh);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    const long long T = sq.first[p.n_seqs];
    const int Ge = pa_ctas(G, T, p.n_seqs);
    const bool in = (int)blockIdx.x < Ge;
    const long long u0 = in ? T * blockIdx.x / Ge : 0, u1 = in ? T * (blockIdx.x + 1) / Ge : 0;
    auto seq_of = [&](long long u) {
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sq.first[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };

    if (warp == n_kvh) {
        // ------------------------------------------------ producer
        if (lane == 0 && u0 < u1) {
            const uint64_t pol = policy_evict_first();
            uint32_t fill = 0;
            int s = seq_of(u0);
            for (long long u = u0; u < u1; ++u) {
                while (u >= sq.first[s + 1]) ++s;
                const int b = (int)(u - sq.first[s]);
                const long long cs = p.row_seq ? __ldg(p.row_seq + s) : s;
                const long long blk = p.block_table ? (long long)__ldg(p.block_table + cs * p.max_blocks + b)
                                                    : cs * p.max_blocks + b;
                const bool ok = blk >= 0 && (blk + 1) * kPaBt <= p.cache_rows;
                if (!ok) flag_error(p.err, DS_ERR_POSITION);
                const int row0 = ok ? (int)(blk * kPaBt) : 0;
                for (int kv = 0; kv < 2; ++kv, ++fill) {
                    const int st = fill % stages;
                    const uint32_t use = fill / stages;
                    if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1, p.err)) {
                        s_abort = 1;
                        goto drain;
                    }
                    mbar_arrive_expect_tx(&full[st], (uint32_t)stage_bytes);
                    const CUtensorMap *map = kv ? &p.tv : &p.tk;
                    unsigned char *dst = smem + (size_t)st * stage_bytes;
                    if (p.box3d) {  // the whole block in one box: [head half][16 positions][64 dims]
                        asm volatile(
                            "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                            " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
                            "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(0), "r"(smem_u32(&full[st])),
                            "l"(pol)
                            : "memory");
                    } else {
                        for (int g = 0; g < n_kvh; ++g)
                            for (int h = 0; h < 2; ++h)
                                tma_box_g2s(dst + g * 4096 + h * 2048, map, g * kPaHd + h * 64, row0, &full[st], pol);
                    }
                }
            }
        drain:
            const uint32_t first = fill > (uint32_t)stages ? fill - stages : 0;
            for (uint32_t f = first; f < fill; ++f)
                if (!mbar_wait(&full[f % stages], (f / stages) & 1, p.err)) break;
        }
        return;
    }

    // ---------------------------------------------------- consumers: warp g = KV head g
    constexpr int NC = 2 * GQ;          // columns in use: GQ hi, then GQ lo
    constexpr int PD = GQ / 2;          // lane distance between a hi column and its lo column
    const int g = warp;
    const int q4 = lane & 3, r8 = lane >> 2;
    // columns of this lane in the C fragments: 2 q4, 2 q4 + 1
    const bool use_lane = 2 * q4 < NC;           // lanes past the used columns hold padding
    const int hA = (2 * q4) % GQ, hB = hA + 1;   // heads of the lane's two columns
    const bool lo_part = 2 * q4 >= GQ && use_lane;
    __nv_bfloat16 *ptab = ptab_all + warp * 8 * kPaBt;
    const uint32_t st_base = smem_u32(smem);
    const float scale = p.scale;
    const int rec = kPaHd + 2;
    uint32_t fill = 0;
    int s = u0 < u1 ? seq_of(u0) : 0;
    long long u = u0;
    while (u < u1) {
        while (u >= sq.first[s + 1]) ++s;
        const long long seg_end = min(u1, (long long)sq.first[s + 1]);
        const int n_ctx = sq.n_ctx[s];
        // Q^T fragments: column n = r8 (head n hi, head n - GQ lo, else 0), dims 16 t + 2 q4 + {0, 1} (+ 8)
        uint32_t qb[8][2];
        {
            const int n = r8;
            const int head = n < GQ ? n : n - GQ;
            const bool have = n < NC;
            const float *qr = p.q + ((long long)s * p.n_qh + g * GQ + (have ? head : 0)) * kPaHd;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int d = 16 * t + 2 * q4 + 8 * k;
                    const float2 v = have ? __ldg(reinterpret_cast<const float2 *>(qr + d)) : make_float2(0.f, 0.f);
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(v.x), h1 = __float2bfloat16_rn(v.y);
                    if (n < GQ) {
                        qb[t][k] = pack_bf16(h0, h1);
                    } else {
                        qb[t][k] = pack_bf16(__float2bfloat16_rn(v.x - __bfloat162float(h0)),
                                             __float2bfloat16_rn(v.y - __bfloat162float(h1)));
                    }
                }
            }
        }
        float acc[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[t][e] = 0.0f;
        float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
        for (; u < seg_end; ++u) {
            const int b = (int)(u - sq.first[s]);
            const int valid = min(kPaBt, n_ctx - b * kPaBt);
            // ---- scores: S^T[pos][col] over the 8 dim slices
            int st = fill % stages;
            bool ok = !s_abort && mbar_wait(&full[st], (fill / stages) & 1, p.err);
            if (!ok) s_abort = 1;
            float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            {
                const uint32_t base = st_base + (uint32_t)(st * stage_bytes);
                const int pos = (lane & 7) + 8 * ((lane >> 3) & 1), dsub = 8 * (lane >> 4);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    uint32_t a[4];
                    ldsm_x4(a, base + pa_swz(g, pos, 16 * t + dsub));
                    mma_bf16_16816(c, a, qb[t][0], qb[t][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            ++fill;
            // hi + lo columns; rows r8 and r8 + 8 are positions
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] += __shfl_xor_sync(0xffffffffu, c[e], PD);
            const bool in0 = r8 < valid, in1 = r8 + 8 < valid;
            float sA0 = in0 ? c[0] * scale : -INFINITY, sB0 = in0 ? c[1] * scale : -INFINITY;
            float sA1 = in1 ? c[2] * scale : -INFINITY, sB1 = in1 ? c[3] * scale : -INFINITY;
            float bA = fmaxf(sA0, sA1), bB = fmaxf(sB0, sB1);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, o));
                bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, o));
            }
            const float nA = fmaxf(mA, bA), nB = fmaxf(mB, bB);
            const float cA = mA == -INFINITY ? 0.0f : expf(mA - nA), cB = mB == -INFINITY ? 0.0f : expf(mB - nB);
            mA = nA;
            mB = nB;
            const float pA0 = in0 ? expf(sA0 - nA) : 0.0f, pB0 = in0 ? expf(sB0 - nB) : 0.0f;
            const float pA1 = in1 ? expf(sA1 - nA) : 0.0f, pB1 = in1 ? expf(sB1 - nB) : 0.0f;
            float sumA = pA0 + pA1, sumB = pB0 + pB1;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                sumA += __shfl_xor_sync(0xffffffffu, sumA, o);
                sumB += __shfl_xor_sync(0xffffffffu, sumB, o);
            }
            lA = lA * cA + sumA;
            lB = lB * cB + sumB;
            // P^T table [column][position]: hi parts in columns hA, hB; lo parts GQ further
            if (use_lane) {
                const float pv[4] = {pA0, pB0, pA1, pB1};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = (e & 1) ? hB : hA, pos = r8 + 8 * (e >> 1);
                    const __nv_bfloat16 hi = __float2bfloat16_rn(pv[e]);
                    const __nv_bfloat16 w = lo_part ? __float2bfloat16_rn(pv[e] - __bfloat162float(hi)) : hi;
                    ptab[(col + (lo_part ? GQ : 0)) * kPaBt + pos] = w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) ptab[(2 * q4 + (e & 1)) * kPaBt + r8 + 8 * (e >> 1)] = __float2bfloat16_rn(0.0f);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                acc[t][0] *= cA;
                acc[t][1] *= cB;
                acc[t][2] *= cA;
                acc[t][3] *= cB;
            }
            __syncwarp();
            // ---- output: O^T[dims][col] += V^T . P^T
            const uint32_t pb0 = *reinterpret_cast<const uint32_t *>(ptab + r8 * kPaBt + 2 * q4);
            const uint32_t pb1 = *reinterpret_cast<const uint32_t *>(ptab + r8 * kPaBt + 2 * q4 + 8);
            st = fill % stages;
            ok = !s_abort && mbar_wait(&full[st], (fill / stages) & 1, p.err);
            if (!ok) s_abort = 1;
            {
                const uint32_t base = st_base + (uint32_t)(st * stage_bytes);
                const int pos = (lane & 7) + 8 * (lane >> 4), dsub = 8 * ((lane >> 3) & 1);
                // rows past the context may hold anything: their weights are 0, but 0 x NaN is not
                const bool row_ok = pos < valid;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    uint32_t a[4];
                    ldsm_x4_trans(a, base + pa_swz(g, pos, 16 * t + dsub));
                    if (valid < kPaBt) {
                        // zero the elements that came from rows past the context: a[e] holds
                        // positions 2 q4 + {0,1} (a0, a1) and 2 q4 + 8 + {0,1} (a2, a3)
                        const int p0 = 2 * q4, p1 = 2 * q4 + 8;
                        const uint32_t m0 = (p0 < valid ? 0xffffu : 0u) | (p0 + 1 < valid ? 0xffff0000u : 0u);
                        const uint32_t m1 = (p1 < valid ? 0xffffu : 0u) | (p1 + 1 < valid ? 0xffff0000u : 0u);
                        a[0] &= m0;
                        a[1] &= m0;
                        a[2] &= m1;
                        a[3] &= m1;
                    }
                    mma_bf16_16816(acc[t], a, pb0, pb1);
                }
                (void)row_ok;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            ++fill;
        }
        // hi + lo columns of the output; the hi lanes write the record
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[t][e] += __shfl_xor_sync(0xffffffffu, acc[t][e], PD);
        float *slot = p.partials + ((size_t)blockIdx.x + s) * p.n_qh * rec;
        if (use_lane && !lo_part) {
            float *rA = slot + (size_t)(g * GQ + hA) * rec, *rB = slot + (size_t)(g * GQ + hB) * rec;
            if (r8 == 0) {
                rA[0] = mA;
                rA[1] = lA;
                rB[0] = mB;
                rB[1] = lB;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                rA[2 + 16 * t + r8] = acc[t][0];
                rB[2 + 16 * t + r8] = acc[t][1];
                rA[2 + 16 * t + r8 + 8] = acc[t][2];
                rB[2 + 16 * t + r8 + 8] = acc[t][3];
            }
        }
        pa_finish_sequence<GQ>(p, s, g, sq.first[s], sq.first[s + 1] - 1, Ge, T);
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

bool paged_attention_maps(PagedAttnArgs &a) {
    // one box per block: dims {64 dims, positions, head halves}, the halves 128 bytes apart
    const long long row_bytes = (long long)a.n_kvh * kPaHd * 2;
    const long long dims[3] = {64, a.cache_rows, 2LL * a.n_kvh};
    const long long strides[2] = {row_bytes, 128};
    const int box[3] = {64, kPaBt, 2 * a.n_kvh};
    if (encode_tiled_3d(&a.tk, a.k_cache, DS_BF16, dims, strides, box, true) &&
        encode_tiled_3d(&a.tv, a.v_cache, DS_BF16, dims, strides, box, true)) {
        a.box3d = 1;
        return true;
    }
    // else sixteen 2-D boxes per block
    a.box3d = 0;
    return encode_tiled_2d(&a.tk, a.k_cache, DS_BF16, (long long)a.n_kvh * kPaHd, a.cache_rows, row_bytes, 64, kPaBt,
                           true) &&
           encode_tiled_2d(&a.tv, a.v_cache, DS_BF16, (long long)a.n_kvh * kPaHd, a.cache_rows, row_bytes, 64, kPaBt,
                           true);
}

template <int GQ>
static cudaError_t launch_pa_tc(PagedAttnArgs a, cudaStream_t stream, bool pdl) {
    const int stage_bytes = a.n_kvh * 4096;
    a.stages = std::min(16, kPaRingBytes / stage_bytes);
    const size_t smem = 1024 + (size_t)a.stages * stage_bytes + 256 + (size_t)a.n_kvh * 8 * kPaBt * 2;
    if (smem > kPaSmemLimit) return cudaErrorInvalidValue;
    return launch_ex(paged_attention_tc_kernel<GQ>, dim3(sm_count()), dim3(a.n_kvh * 32 + 32), smem, stream, pdl, a);
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
    const void *fns[] = {(const void *)paged_attention_tc_kernel<2>, (const void *)paged_attention_tc_kernel<4>,
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
    if (a.kv_dtype == DS_BF16) {  // a.tk / a.tv encoded by paged_attention_maps
        switch (gq) {
            case 2: return launch_pa_tc<2>(a, stream, pdl);
            case 4: return launch_pa_tc<4>(a, stream, pdl);
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
