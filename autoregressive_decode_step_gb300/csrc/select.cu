// Picking the next token: full-vocabulary greedy argmax and the
// temperature / top-k / top-p sampler.
//
// Argmax ("LLM inference kernels", "KV-cache growth and greedy argmax";
// "decode-ops", "Correctness"): blocks scan contiguous slices of a row, the
// last block of the row (an atomic counter) reduces their candidates.  The
// ranking — NaN above every number, equal values to the lower index — is a
// total order, so the result does not depend on reduction order.
//
// Sampler ("decode-ops", "API — Method"): no heap and no sort.  Each row is
// one thread-block cluster; the top-k threshold, the top-p cut and the draw
// are each found by a radix descent over order-preserving keys of the scaled
// logits, with exact fixed-point masses (see the sampler section below), so
// any top_k, including none, runs over a whole vocabulary.
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
//
// One thread-block cluster per row; CTA r of the cluster owns the contiguous
// slice [n r / C, n (r + 1) / C) of the row and keeps its scaled logits there
// as order-preserving 32-bit keys (shared memory).  Nothing is sorted: each
// threshold the sampler needs is found by a most-significant-byte-first radix
// descent over the keys, four levels of 256-way histograms, every level
// summed over the cluster through distributed shared memory:
//   - top-k: the k-th largest key by counts, and how many of the keys equal
//     to it survive (the lowest indices);
//   - top-p: the survivor at which the running mass in (key desc, index asc)
//     order first reaches top_p of the survivors' mass;
//   - the draw: the first kept survivor whose running mass exceeds u times
//     the kept mass.
// Masses are exp(l' - l'_max) in fp32 (as the page's softmax) turned into
// 64-bit fixed point with 2^-F resolution, F = min(46, 63 - ceil(log2 n)), so
// every sum is an exact integer sum: no result depends on the order in which
// threads or CTAs add, and the row's whole mass fits in 63 bits.  Keys equal
// to a selected key all have the same mass, so the position inside such a
// tie is arithmetic; the index of that element is then found by counting
// equal keys CTA by CTA and thread by thread in index order.
// Every CTA of a cluster computes every decision from the same summed
// histograms, so all of them take the same path through a fixed sequence of
// cluster barriers.
constexpr int kSmThreads = 512;
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kSmKeyCap = 20480;   // keys of a CTA's slice held in shared memory
constexpr int kSmListCap = 8192;   // candidates carried from a search's second level on
constexpr int kSmMaxCluster = 8;
constexpr size_t kSmSmem = (size_t)kSmWarps * 256 * 8 + 4 * 256 * 8 + (size_t)kSmWarps * 256 * 4 + 2 * 256 * 4 +
                           (size_t)kSmKeyCap * 4 + 2 * (size_t)kSmListCap * 4;

// Order-preserving map of an fp32 value to an unsigned key and back (-0 and
// +0 share the key of +0, since they compare equal).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire): a hardware barrier, executed by all threads at the same points.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of `p` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cl_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t cl_ld32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint64_t cl_ld64(uint32_t a) {
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a));
    return v;
}

// Fixed-point mass of a key: exp(l' - l'_max) in fp32 times 2^F, rounded.
__device__ __forceinline__ uint64_t key_mass(uint32_t key, float lmax, float scale) {
    const float e = expf(key_value(key) - lmax);
    return e > 0.0f ? __float2ull_rn(e * scale) : 0ull;
}

// Add one element to this warp's private histogram: a count, or (`mass`) its
// mass.  Only lanes of one warp ever touch a warp's histogram, so the
// shared-memory atomics conflict only between lanes with the same digit.
__device__ __forceinline__ void hist_add(uint32_t *cw, uint64_t *mw, bool valid, uint32_t digit, uint64_t m,
                                         bool mass) {
    if (!valid) return;
    if (mass) atomicAdd(reinterpret_cast<unsigned long long *>(mw + digit), (unsigned long long)m);
    else atomicAdd(cw + digit, 1u);
}

// Warp 0: the first digit, from 255 down, at which base + the running sum of
// vals[] reaches thr; returns it and the running sum before it (plus base).
__device__ __forceinline__ void warp_select(const uint64_t *vals, uint64_t base, uint64_t thr, uint32_t &digit,
                                            uint64_t &before) {
    const int lane = threadIdx.x & 31;
    uint64_t v[8], s = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        v[q] = vals[255 - 8 * lane - q];
        s += v[q];
    }
    uint64_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, base + incl >= thr);
    const int L = hit ? __ffs(hit) - 1 : 31;  // no crossing (never for consistent sums): the lowest digit
    uint32_t d = 0;
    uint64_t c = 0;
    if (lane == L) {
        uint64_t cc = base + incl - s;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (cc + v[q] >= thr || q == 7) {
                d = 255 - 8 * L - q;
                c = cc;
                break;
            }
            cc += v[q];
        }
    }
    digit = __shfl_sync(0xffffffffu, d, L);
    before = __shfl_sync(0xffffffffu, c, L);
}

// Decisions of one row, identical in every CTA of its cluster.
struct SmDec {
    uint32_t gmax;      // largest key of the row
    int degenerate;     // the largest scaled logit is not finite
    uint32_t prefix;    // bits of the current search fixed so far
    uint64_t base;      // mass (or count) ranked before the prefix's keys
    uint64_t thr;       // the running sum a search looks for
    uint64_t sel;       // mass (or count) of the key a search's last level selected
    uint32_t tau_k;     // the top_k-th largest key
    uint32_t need_eq;   // survivors among the keys equal to tau_k
    uint32_t cnt_k;     // keys equal to tau_k
    uint32_t tau_p;     // the key at which the top-p cut falls
    uint32_t jp1;       // survivors kept among the keys equal to tau_p
    uint64_t S2;        // mass of the kept survivors
    uint32_t tau_s;     // the key of the drawn token
    uint32_t j_s;       // its rank among the keys equal to tau_s (index order)
};

// Keys that the short path gathers into one CTA and ranks there at most.
constexpr int kSmFastCap = 256;

__global__ void __launch_bounds__(kSmThreads, 1) sample_kernel(const __grid_constant__ SampleArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint64_t *mass_w = reinterpret_cast<uint64_t *>(smem);  // [warps][256] per-warp masses
    uint64_t *hm = mass_w + kSmWarps * 256;                  // [2][256] this CTA's sums (cluster-visible)
    uint64_t *tot_m = hm + 512;                              // [256] cluster sums
    uint64_t *tot0_m = tot_m + 256;                          // [256] the first mass level's sums
    uint32_t *cnt_w = reinterpret_cast<uint32_t *>(tot0_m + 256);  // [warps][256] per-warp counts
    uint32_t *hc = cnt_w + kSmWarps * 256;                         // [2][256] (cluster-visible)
    uint32_t *keys = hc + 512;                                     // [kSmKeyCap]
    uint32_t *list = keys + kSmKeyCap;                             // [kSmListCap] candidates' local indices
    uint32_t *lkey = list + kSmListCap;                            // [kSmListCap] their keys (the short path)
    __shared__ SmDec dec;
    __shared__ uint32_t s_cta_max, s_tie, s_list_n, s_list_over;
    __shared__ float s_bv[kSmWarps];
    __shared__ int s_bi[kSmWarps];
    __shared__ uint32_t s_scan[kSmWarps];
    __shared__ uint64_t s_scan64[kSmWarps];
    __shared__ uint32_t s_off[kSmMaxCluster + 1];
    __shared__ uint32_t s_rk[kSmMaxCluster];

    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t C = cl_size(), rank = cl_rank();
    const int row = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long n = p.n;
    const float *l = p.logits + (long long)row * n;
    const long long i0 = n * rank / C, i1 = n * (rank + 1) / C;
    const int len = (int)(i1 - i0);
    const bool cached = len <= kSmKeyCap;
    const float T = p.temperature;

    if (!(T > 0.0f)) {  // greedy: first index of the maximum, NaN above every number
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (long long i = i0 + tid; i < i1; i += kSmThreads) {
            const float v = l[i];
            if (ranks_above(v, (int)i, bv, bi)) {
                bv = v;
                bi = (int)i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_above(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            s_bv[warp] = bv;
            s_bi[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < kSmWarps; ++w)
                if (ranks_above(s_bv[w], s_bi[w], bv, bi)) {
                    bv = s_bv[w];
                    bi = s_bi[w];
                }
            s_bv[0] = bv;
            s_bi[0] = bi;
        }
        cl_sync();
        if (rank == 0 && tid == 0) {
            for (uint32_t r = 1; r < C; ++r) {
                const float v = __uint_as_float(cl_ld32(cl_map(&s_bv[0], r)));
                const int ix = (int)cl_ld32(cl_map(&s_bi[0], r));
                if (ranks_above(v, ix, bv, bi)) {
                    bv = v;
                    bi = ix;
                }
            }
            p.ids[row] = bi;
            if (p.tokens_adv) p.tokens_adv[row] = bi;
            if (p.pos_adv) p.pos_adv[row] += 1;
        }
        cl_sync();
        return;
    }

    const long long K = (p.top_k <= 0 || p.top_k >= n) ? n : p.top_k;
    const bool topk_on = K < n;
    const bool topp_on = p.top_p < 1.0f;
    int lg = 0;
    while ((1LL << lg) < n) ++lg;
    const int F = min(46, 63 - lg);
    const float scale = __uint_as_float((uint32_t)(127 + F) << 23);  // 2^F
    auto key_at = [&](int j) -> uint32_t { return cached ? keys[j] : order_key(l[i0 + j] / T); };
    auto zero_hist = [&](bool counts, bool masses, bool new_list) {
        for (int i = tid; i < kSmWarps * 256; i += kSmThreads) {
            if (counts) cnt_w[i] = 0;
            if (masses) mass_w[i] = 0;
        }
        if (new_list && tid == 0) {
            s_list_n = 0;
            s_list_over = 0;
        }
        __syncthreads();
    };
    // this CTA's histogram (sum of its warps') into buffer b: counts (hc) or
    // masses (hm); after the cluster barrier, gather() sums every CTA's, in
    // rank order, into tot_m
    auto publish = [&](int b, bool masses) {
        __syncthreads();
        if (tid < 256) {
            if (masses) {
                uint64_t m = 0;
                for (int w = 0; w < kSmWarps; ++w) m += mass_w[w * 256 + tid];
                hm[b * 256 + tid] = m;
            } else {
                uint32_t c = 0;
                for (int w = 0; w < kSmWarps; ++w) c += cnt_w[w * 256 + tid];
                hc[b * 256 + tid] = c;
            }
        }
    };
    auto gather = [&](int b, bool masses) {
        if (tid < 256) {  // every rank's bucket requested before any is added
            uint64_t v[kSmMaxCluster];
#pragma unroll
            for (int r = 0; r < kSmMaxCluster; ++r) {
                v[r] = 0;
                if (r < (int)C)
                    v[r] = masses ? cl_ld64(cl_map(hm + b * 256 + tid, r)) : cl_ld32(cl_map(hc + b * 256 + tid, r));
            }
            uint64_t t = 0;
#pragma unroll
            for (int r = 0; r < kSmMaxCluster; ++r) t += v[r];
            tot_m[tid] = t;
        }
        __syncthreads();
    };
    // f(j, key, valid) over this CTA's whole slice, four consecutive keys per
    // thread per round; every lane of a warp calls f in every round
    auto full_pass = [&](auto &&f) {
        for (int b0 = 0; b0 < len; b0 += kSmThreads * 4) {
            const int jb = b0 + 4 * tid;
            uint32_t k4[4];
            if (cached && jb + 3 < len) {
                const uint4 v = *reinterpret_cast<const uint4 *>(keys + jb);
                k4[0] = v.x;
                k4[1] = v.y;
                k4[2] = v.z;
                k4[3] = v.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) k4[q] = jb + q < len ? key_at(jb + q) : 0u;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) f(jb + q, k4[q], jb + q < len);
        }
    };
    // append the matching lanes' local indices (and keys) to the candidate
    // list, one shared-memory atomic per warp; past its capacity the list is
    // marked overflowed and later levels scan the whole slice instead
    auto list_append = [&](bool match, uint32_t j, uint32_t key) {
        const unsigned m = __ballot_sync(0xffffffffu, match);
        if (!m) return;
        uint32_t base = 0;
        if (lane == __ffs(m) - 1) base = atomicAdd(&s_list_n, (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
        if (match) {
            const uint32_t slot = base + __popc(m & ((1u << lane) - 1u));
            if (slot < (uint32_t)kSmListCap) {
                list[slot] = j;
                lkey[slot] = key;
            } else {
                s_list_over = 1;
            }
        }
    };

    // ---------------- keys, the row's largest key, top-k's first-level counts
    zero_hist(true, false, false);
    uint32_t kmax = 0;
    constexpr int kLoadUnroll = 8;  // loads in flight per thread
    for (int b0 = 0; b0 < len; b0 += kSmThreads * kLoadUnroll) {
        float v[kLoadUnroll];
#pragma unroll
        for (int q = 0; q < kLoadUnroll; ++q) {
            const int j = b0 + q * kSmThreads + tid;
            v[q] = j < len ? l[i0 + j] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kLoadUnroll; ++q) {
            const int j = b0 + q * kSmThreads + tid;
            const bool valid = j < len;
            const uint32_t key = valid ? order_key(v[q] / T) : 0u;
            if (valid && cached) keys[j] = key;
            kmax = max(kmax, key);
            if (topk_on) hist_add(cnt_w + warp * 256, mass_w, valid, key >> 24, 0, false);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (lane == 0) s_scan[warp] = kmax;
    publish(0, false);
    if (tid == 0) {
        uint32_t m = 0;
        for (int w = 0; w < kSmWarps; ++w) m = max(m, s_scan[w]);
        s_cta_max = m;
    }
    cl_sync();  // 1
    gather(0, false);
    if (tid < (int)C) s_rk[tid] = cl_ld32(cl_map(&s_cta_max, tid));
    __syncthreads();
    if (tid == 0) {
        uint32_t m = 0;
        for (uint32_t r = 0; r < C; ++r) m = max(m, s_rk[r]);
        dec.gmax = m;
        const float lm = key_value(m);
        dec.degenerate = !(lm - lm == 0.0f);  // NaN or infinite
        dec.tau_k = 0;
        dec.need_eq = 0;
        dec.cnt_k = 0;
        dec.jp1 = 0;
        dec.tau_p = 0;
    }
    __syncthreads();
    const bool degenerate = dec.degenerate != 0;
    const float lmax = key_value(dec.gmax);
    const bool k_search = topk_on && !degenerate;
    if (k_search && warp == 0) {
        uint32_t d;
        uint64_t before;
        warp_select(tot_m, 0, (uint64_t)K, d, before);
        if (lane == 0) {
            dec.prefix = d << 24;
            dec.base = before;  // survivors ranked above the prefix's keys
            dec.thr = (uint64_t)K;
            dec.sel = tot_m[d];
        }
    }
    __syncthreads();

    // ---------------- the short path: when few keys can survive, rank 0
    // gathers every key at or above `kmin` (the survivors among them: the
    // first Kt in (key desc, index asc) order), ranks them by counting, and
    // takes the top-p cut and the draw over exact running sums of their masses
    auto short_path = [&](uint32_t kmin, int Kt) {
        if (tid == 0) s_list_n = 0;
        __syncthreads();
        full_pass([&](int j, uint32_t key, bool valid) { list_append(valid && key >= kmin, (uint32_t)j, key); });
        __syncthreads();
        cl_sync();  // short path 1
        if (rank == 0) {
            uint32_t *ck = cnt_w;                    // [kSmFastCap] gathered keys
            uint32_t *ci = cnt_w + kSmFastCap;       // [kSmFastCap] their row indices
            uint32_t *sk = cnt_w + 2 * kSmFastCap;   // [kSmFastCap] survivors in order: keys
            uint32_t *si = cnt_w + 3 * kSmFastCap;   // [kSmFastCap] and indices
            uint64_t *sm = mass_w;                   // [kSmFastCap] running sums of their masses
            if (tid < (int)C) s_rk[tid] = cl_ld32(cl_map(&s_list_n, tid));
            __syncthreads();
            if (tid == 0) {
                uint32_t o = 0;
                for (uint32_t r = 0; r < C; ++r) {
                    s_off[r] = o;
                    o += s_rk[r];
                }
                s_off[C] = o;
            }
            __syncthreads();
            const int M = (int)min(s_off[C], (uint32_t)kSmFastCap);
            for (int e = tid; e < M; e += kSmThreads) {
                uint32_t r = 0;
                while (e >= (int)s_off[r + 1]) ++r;
                const uint32_t q = e - s_off[r];
                const uint32_t kk = cl_ld32(cl_map(lkey + q, r));
                const uint32_t jj = cl_ld32(cl_map(list + q, r));
                ck[e] = kk;
                ci[e] = (uint32_t)(n * r / C) + jj;
            }
            __syncthreads();
            for (int e = warp; e < M; e += kSmWarps) {  // position in (key desc, index asc) order, a warp per key
                const uint32_t ke = ck[e], ie = ci[e];
                int at = 0;
                for (int f0 = 0; f0 < M; f0 += 32) {
                    const int f = f0 + lane;
                    at += __popc(__ballot_sync(0xffffffffu, f < M && (ck[f] > ke || (ck[f] == ke && ci[f] < ie))));
                }
                if (lane == 0 && at < Kt) {
                    sk[at] = ke;
                    si[at] = ie;
                }
            }
            __syncthreads();
            // survivors' masses and their running sums (exact integers)
            if (warp == 0) {
                constexpr int kPer = kSmFastCap / 32;
                uint64_t own[kPer], acc = 0;
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    const int i = lane * kPer + q;
                    own[q] = i < Kt ? key_mass(sk[i], lmax, scale) : 0ull;
                    acc += own[q];
                }
                uint64_t incl = acc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                uint64_t run = incl - acc;
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    run += own[q];
                    sm[lane * kPer + q] = run;
                }
                __syncwarp();
                if (lane == 0) {
                    // first position in [0, hi] whose running sum reaches x
                    auto first_at_least = [&](int hi, uint64_t x) {
                        int lo = 0;
                        while (lo < hi) {
                            const int mid = (lo + hi) >> 1;
                            if (sm[mid] >= x) hi = mid;
                            else lo = mid + 1;
                        }
                        return lo;
                    };
                    const uint64_t S = sm[Kt - 1];
                    int kept = Kt;
                    if (topp_on) {
                        const double x = ceil((double)p.top_p * (double)S);
                        uint64_t thr = x < 1.0 ? 1ull : (uint64_t)x;
                        if (thr > S) thr = S;
                        kept = min(Kt, first_at_least(Kt - 1, thr) + 1);
                    }
                    const uint64_t S2 = sm[kept - 1];
                    const double y = floor((double)p.u[row] * (double)S2);
                    uint64_t thr = (y < 0.0 ? 0ull : (uint64_t)y) + 1;
                    if (thr > S2) thr = S2;
                    const int chosen = first_at_least(kept - 1, thr);
                    const int id = (int)si[chosen];
                    p.ids[row] = id;
                    if (p.tokens_adv) p.tokens_adv[row] = id;
                    if (p.pos_adv) p.pos_adv[row] += 1;
                }
            }
        }
        cl_sync();  // short path 2: no CTA leaves while rank 0 may still read its list
    };
    {   // every key in the top-k's first-level bucket or above it, or the whole row when it is short
        const long long m0 = k_search ? (long long)(dec.base + dec.sel) : n;
        if (!degenerate && (k_search || !topk_on) && m0 <= kSmFastCap) {  // the same in every CTA
            short_path(k_search ? (dec.prefix & 0xff000000u) : 0u, k_search ? (int)K : (int)m0);
            return;
        }
    }

    // ---------------- top-k: levels 1..3 by counts
    for (int lv = 1; lv <= 3; ++lv) {
        const int shift = 24 - 8 * lv;
        const uint32_t mask = 0xffffffffu << (shift + 8);
        const int b = lv & 1;
        if (k_search) {
            zero_hist(true, false, lv == 1);
            const uint32_t prefix = dec.prefix;
            auto visit = [&](int j, uint32_t key, bool valid) {
                const bool match = valid && (key & mask) == prefix;
                if (lv == 1) list_append(match, (uint32_t)j, key);
                hist_add(cnt_w + warp * 256, mass_w, match, (key >> shift) & 255u, 0, false);
            };
            if (lv > 1 && !s_list_over) {
                const int cnt = (int)min(s_list_n, (uint32_t)kSmListCap);
                for (int idx = tid; idx < cnt; idx += kSmThreads) visit((int)list[idx], lkey[idx], true);
            } else {
                full_pass(visit);
            }
            publish(b, false);
        }
        cl_sync();  // 2, 3, 4
        if (k_search) {
            gather(b, false);
            if (warp == 0) {
                uint32_t d;
                uint64_t before;
                warp_select(tot_m, dec.base, dec.thr, d, before);
                if (lane == 0) {
                    dec.prefix |= d << shift;
                    dec.base = before;
                    if (lv == 3) {
                        dec.tau_k = dec.prefix;
                        dec.need_eq = (uint32_t)(dec.thr - before);
                        dec.cnt_k = (uint32_t)tot_m[d];
                    }
                }
            }
            __syncthreads();
        }
    }
    const uint32_t tau_k = dec.tau_k, need_eq = dec.need_eq;
    const uint64_t m_k = k_search ? key_mass(tau_k, lmax, scale) : 0ull;
    {   // the survivors themselves are few: the short path over the keys >= tau_k
        const long long m1 = k_search ? (K - need_eq) + dec.cnt_k : n;
        if (k_search && m1 <= kSmFastCap) {  // the same in every CTA
            short_path(tau_k, (int)K);
            return;
        }
    }

    // survivors: every key above tau_k (the keys equal to it are added as a
    // group of need_eq by the decisions)
    auto survives = [&](uint32_t key) { return !k_search || key > tau_k; };
    auto add_group = [&](uint32_t prefix, uint32_t mask, int shift) {
        if (k_search && (tau_k & mask) == prefix) tot_m[(tau_k >> shift) & 255u] += (uint64_t)need_eq * m_k;
    };

    // ---------------- survivors' masses by first digit: the mass S
    zero_hist(false, true, false);
    if (!degenerate)
        full_pass([&](int, uint32_t key, bool valid) {
            const bool sv = valid && survives(key);
            hist_add(cnt_w, mass_w + warp * 256, sv, key >> 24, sv ? key_mass(key, lmax, scale) : 0ull, true);
        });
    publish(0, true);
    cl_sync();  // 5
    gather(0, true);
    if (!degenerate) {
        if (tid == 0) add_group(0u, 0u, 24);
        __syncthreads();
        if (tid < 256) tot0_m[tid] = tot_m[tid];
        __syncthreads();
        if (warp == 0) {
            uint64_t s = 0;
            for (int d = lane; d < 256; d += 32) s += tot_m[d];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            uint64_t thr = s;
            if (topp_on) {
                const double x = ceil((double)p.top_p * (double)s);
                thr = x < 1.0 ? 1ull : (uint64_t)x;
                if (thr > s) thr = s;
                uint32_t d;
                uint64_t before;
                warp_select(tot_m, 0, thr, d, before);
                if (lane == 0) {
                    dec.prefix = d << 24;
                    dec.base = before;
                }
            }
            if (lane == 0) {
                dec.S2 = s;
                dec.thr = thr;
            }
        }
        __syncthreads();
    }

    // ---------------- a mass search's levels 1..3 (top-p, then the draw)
    auto mass_levels = [&](bool active, int b_first) {
        for (int lv = 1; lv <= 3; ++lv) {
            const int shift = 24 - 8 * lv;
            const uint32_t mask = 0xffffffffu << (shift + 8);
            const int b = (b_first + lv - 1) & 1;
            if (active) {
                zero_hist(false, true, lv == 1);
                const uint32_t prefix = dec.prefix;
                auto visit = [&](int j, uint32_t key, bool valid) {
                    const bool match = valid && (key & mask) == prefix && survives(key);
                    if (lv == 1) list_append(match, (uint32_t)j, key);
                    hist_add(cnt_w, mass_w + warp * 256, match, (key >> shift) & 255u,
                             match ? key_mass(key, lmax, scale) : 0ull, true);
                };
                if (lv > 1 && !s_list_over) {
                    const int cnt = (int)min(s_list_n, (uint32_t)kSmListCap);
                    for (int idx = tid; idx < cnt; idx += kSmThreads) visit((int)list[idx], lkey[idx], true);
                } else {
                    full_pass(visit);
                }
                publish(b, true);
            }
            cl_sync();  // 6, 7, 8 (top-p); 9, 10, 11 (the draw)
            if (active) {
                gather(b, true);
                if (tid == 0) add_group(dec.prefix, mask, shift);
                __syncthreads();
                if (warp == 0) {
                    uint32_t d;
                    uint64_t before;
                    warp_select(tot_m, dec.base, dec.thr, d, before);
                    if (lane == 0) {
                        dec.prefix |= d << shift;
                        dec.base = before;
                        if (lv == 3) dec.sel = tot_m[d];  // mass of the survivors with the selected key
                    }
                }
                __syncthreads();
            }
        }
    };
    // keys equal to a selected key `tau` all have its mass: their count is
    // the bucket's mass over one key's (one, for a key of zero mass)
    auto equal_count = [&](uint32_t tau, uint64_t bucket_mass) -> uint64_t {
        const uint64_t m = key_mass(tau, lmax, scale);
        return m ? bucket_mass / m : 1;
    };
    const bool p_search = topp_on && !degenerate;
    mass_levels(p_search, 1);
    if (p_search && tid == 0) {  // the cut falls inside the keys equal to tau_p
        const uint32_t tau = dec.prefix;
        const uint64_t m = key_mass(tau, lmax, scale);
        const uint64_t cnt = equal_count(tau, dec.sel);
        uint64_t j = m ? (dec.thr - dec.base + m - 1) / m : 1;  // kept among the equal keys
        if (j < 1) j = 1;
        if (j > cnt) j = cnt;
        dec.tau_p = tau;
        dec.jp1 = (uint32_t)j;
        dec.S2 = dec.base + j * m;
    }
    __syncthreads();
    // the draw: the first kept survivor whose running mass exceeds u * S2
    if (!degenerate) {
        if (tid < 256) tot_m[tid] = tot0_m[tid];
        __syncthreads();
        if (warp == 0) {
            const uint64_t S2 = dec.S2;
            const double y = floor((double)p.u[row] * (double)S2);
            uint64_t thr = (y < 0.0 ? 0ull : (uint64_t)y) + 1;
            if (thr > S2) thr = S2;
            uint32_t d;
            uint64_t before;
            warp_select(tot_m, 0, thr, d, before);
            if (lane == 0) {
                dec.prefix = d << 24;
                dec.base = before;
                dec.thr = thr;
            }
        }
        __syncthreads();
    }
    mass_levels(!degenerate, 0);
    if (tid == 0) {
        if (degenerate) {  // the first index of the largest key
            dec.tau_s = dec.gmax;
            dec.j_s = 0;
        } else {
            const uint32_t tau = dec.prefix;
            const uint64_t m = key_mass(tau, lmax, scale);
            uint64_t cnt = equal_count(tau, dec.sel);
            if (p_search && tau == dec.tau_p && cnt > dec.jp1) cnt = dec.jp1;
            uint64_t j = m ? (dec.thr - dec.base + m - 1) / m : 1;
            if (j < 1) j = 1;
            if (j > cnt) j = cnt;
            dec.tau_s = tau;
            dec.j_s = (uint32_t)(j - 1);
        }
    }
    __syncthreads();

    // ---------------- the j_s-th key equal to tau_s, in index order: each warp
    // counts the equal keys of its contiguous part of the slice
    const uint32_t tau_s = dec.tau_s, j_s = dec.j_s;
    const int seg = (len + kSmWarps - 1) / kSmWarps;
    const int w0 = min(len, warp * seg), w1 = min(len, w0 + seg);
    uint32_t wc = 0;
    for (int b0 = w0; b0 < w1; b0 += 32) {
        const int j = b0 + lane;
        wc += __popc(__ballot_sync(0xffffffffu, j < w1 && key_at(j) == tau_s));
    }
    if (lane == 0) s_scan[warp] = wc;
    __syncthreads();
    if (tid == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kSmWarps; ++w) t += s_scan[w];
        s_tie = t;
    }
    cl_sync();  // 12
    if (tid < (int)C) s_rk[tid] = cl_ld32(cl_map(&s_tie, tid));
    __syncthreads();
    uint32_t before = 0;
    for (uint32_t r = 0; r < rank; ++r) before += s_rk[r];
    for (int w = 0; w < warp; ++w) before += s_scan[w];
    if (j_s >= before && j_s < before + s_scan[warp]) {  // the same for every lane of the warp
        uint32_t k = before;
        for (int b0 = w0; b0 < w1; b0 += 32) {
            const int j = b0 + lane;
            unsigned bal = __ballot_sync(0xffffffffu, j < w1 && key_at(j) == tau_s);
            const uint32_t c = __popc(bal);
            if (j_s < k + c) {
                for (uint32_t q = k; q < j_s; ++q) bal &= bal - 1;  // drop the equal keys ahead of it
                if (lane == __ffs(bal) - 1) {
                    const int id = (int)(i0 + j);
                    p.ids[row] = id;
                    if (p.tokens_adv) p.tokens_adv[row] = id;
                    if (p.pos_adv) p.pos_adv[row] += 1;
                    if (degenerate) flag_error(p.err, DS_ERR_SAMPLING);
                }
                break;
            }
            k += c;
        }
    }
    cl_sync();  // 13: no CTA leaves while another may still read its shared memory
}

static bool g_sample_ready = false;

cudaError_t prepare_sample_kernel() {
    cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmSmem);
    if (e == cudaSuccess) g_sample_ready = true;
    return e;
}

int sample_cluster_size(long long n) {
    const long long c = (n + kSmKeyCap - 1) / kSmKeyCap;
    return (int)std::max(1LL, std::min((long long)kSmMaxCluster, c));
}

cudaError_t launch_sample(const SampleArgs &a, cudaStream_t stream, bool pdl) {
    if (!g_sample_ready) {
        cudaError_t e = prepare_sample_kernel();
        if (e != cudaSuccess) return e;
    }
    const int C = sample_cluster_size(a.n);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, a.n_rows);
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = kSmSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int na = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, sample_kernel, a);
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
