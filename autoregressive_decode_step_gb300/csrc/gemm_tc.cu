// Batched projections on the fifth-generation tensor cores (tcgen05).
//
// When a decode step serves n sequences at once ("Inside the engine",
// section 4: batched decode, one token per sequence per step), every
// projection y_s = A^T x_s of the step ("LLM inference kernels", "A parallel
// path for one frozen kernel's known-slow shape") is applied to n vectors and
// becomes a skinny GEMM: Y[s][j] = sum_i A[i][j] X[s][i].  The weight matrix
// goes on the MMA's M side (128 output features per tile) and the n <= 256
// activation rows on its N side, so one weight byte is fetched once for all n
// sequences and the accumulator (128 lanes x n columns of fp32) lives in
// tensor memory.  Operands are bf16, accumulation fp32.  Inside the decode
// step an fp32 activation v reaches this kernel as a bf16 pair (hi, lo) with
// hi + lo = v to 16 significant bits; both rows are multiplied into the same
// accumulator (two MMAs per k-step), so the product is that of the fp32
// activation, not of a bf16 rounding of it.  The path is bound by the weight
// stream, so the second MMA costs nothing measurable.
//
// Roles (192 threads, one CTA per SM):
//   warp 0, one thread: TMA producer.  Per 64-row k-block it loads the weight
//     tile (two 64 x 64 boxes of an [in][out] matrix, or one 128 x 64 box of
//     a [vocab][d] head) and the activation tile (n_pad x 64) into one stage
//     of a shared-memory ring, 128-byte swizzled, completing on the stage's
//     mbarrier.  With programmatic dependent launch the weight boxes of the
//     first stages are requested before the previous kernel has finished.
//   warp 1: allocates the tensor memory (two accumulator buffers) and, from
//     one thread, issues tcgen05.mma (kind::f16, M = 128, N = n_pad, K = 16)
//     four times per stage; tcgen05.commit frees the stage and, after a
//     tile's last stage, signals its accumulator buffer full.
//   warps 2-5: read the accumulator (tcgen05.ld, warp w owns lanes
//     32 (w % 4) ..) and run the fused epilogue: store, residual add,
//     SiLU-gate to bf16, or RoPE + K/V write for the q|k|v projection.
//
// Work split: the (tile, k-block) units are cut into equal contiguous ranges,
// one per CTA (every CTA streams the same weight bytes whatever the shape).
// A tile whose k-blocks fall to several CTAs is finished by all of them
// together: each writes its partial accumulator to the workspace and arrives
// on the tile's counter; at the end of its range each contributor waits
// (bounded) for its split tiles to be complete and finishes its share of
// their 32-vector chunks, adding the partials in CTA order, so results are
// bit-stable run to run whoever finishes a chunk.  Every wait (mbarrier or
// counter) is bounded; a wait that times out flags DS_ERR_WAIT_TIMEOUT and
// the kernel winds down, draining its copies and MMAs in flight and freeing
// its tensor memory before it exits.
#include <algorithm>

#include "common.cuh"
#include "tc.h"

namespace ds {

constexpr int kTcBM = 128;        // output features per tile (MMA M)
constexpr int kTcBK = 64;         // reduced rows per stage: 128 bytes of bf16, one swizzle span
constexpr int kTcThreads = 192;
constexpr int kTcEpiThreads = 128;
constexpr int kTcABytes = kTcBM * kTcBK * 2;  // 16 KB
constexpr int kTcMaxStages = 8;
constexpr int kTcXchStride = 33;  // floats per feature row of the epilogue exchange buffer
constexpr int kTcMaxN = 256;      // vectors per launch (the MMA's largest N)
constexpr int kTcSmemInts = 16 + 3 * kTcMaxN;  // tmem address, flags, agreement words, per-vector rows, scales
constexpr int kTcMaxContrib = 4;  // split partials one chunk's reduction requests at once
constexpr size_t kTcSmemLimit = 227 * 1024;

// ---------------------------------------------------------------- tcgen05 PTX
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] x B[smem]: one MMA of kind::f16 on this CTA's SM.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 32 consecutive accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, the fixed tcgen05 version field and 128-byte swizzling.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A
// MN-major (a_mn) or K-major, B K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc(int a_mn, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kTcBM >> 4) << 24);
}

// Bounded wait until the counter at ctr reaches target (acquire), giving up
// once another role has aborted.
__device__ bool tc_wait_count(const int *ctr, int target, volatile int *abort_flag, int *err) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((it & 63u) == 63u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                flag_error(err, DS_ERR_WAIT_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
        __nanosleep(32);
    }
}

// Bounded mbarrier wait that also gives up once another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                flag_error(err, DS_ERR_WAIT_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_box_g2s_nohint(void *dst, const void *map, int c0, int r0, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(smem_u32(bar))
        : "memory");
}

// Segment of a CTA's unit range that lies in one tile.
struct TcSeg {
    int tile, kb0, kb1;
};

__device__ __forceinline__ bool tc_next_seg(long long &u, long long u1, int KB, TcSeg &s) {
    if (u >= u1) return false;
    s.tile = (int)(u / KB);
    s.kb0 = (int)(u - (long long)s.tile * KB);
    s.kb1 = (int)std::min((long long)KB, s.kb0 + (u1 - u));
    u += s.kb1 - s.kb0;
    return true;
}

// silu(z) = z / (1 + e^-z); the quotient as an approximate reciprocal times
// z (two ulps at most: no per-item branch to a division slow path in the
// epilogue's unrolled loops).  1 + e^-z >= 1, and an infinite e^-z gives -0.
__device__ __forceinline__ float silu_tc(float z) { return __fdividef(z, 1.0f + expf(-z)); }

// The residual values (TC_ADD) of one chunk for the tile's feature of this
// thread, requested before the chunk's sums are waited for.
__device__ __forceinline__ void tc_load_residual(const TcArgs &p, int tile, int chunk, int r, float (&old)[32]) {
    const int j0 = chunk * 32, m = tile * kTcBM + r;
    const int nj = min(32, p.n - j0);
    const float *col = p.y + (long long)j0 * p.ldy + m;
#pragma unroll
    for (int i = 0; i < 32; ++i) old[i] = (m < p.M && i < nj) ? __ldcg(col + (long long)i * p.ldy) : 0.0f;
}

// One chunk (32 sequences) of the fused epilogue for the tile's feature of
// this thread (row r of the accumulator); `old` is the chunk's residual as
// tc_load_residual left it (TC_ADD only).
// QK-norm of one 32-vector chunk of a q|k|v tile (Qwen3's per-head RMSNorm
// before RoPE): xch[f * kTcXchStride + i] holds feature f of vector i; every q
// head and every k head (hd consecutive features, aligned to the tile) is
// scaled per vector by 1/sqrt(mean of its squares + eps) and by q_norm or
// k_norm; v features are left alone.  The four epilogue warps call it.
__device__ void tc_qk_norm(const TcArgs &p, int m, int r, float *xch) {
    const int lane = r & 31, hd = p.head_dim;
    const bool normed = m < p.nq_cols + p.nkv_cols;
    float *hs = xch + kTcBM * kTcXchStride;  // [4 warps][32 vectors] head square sums
    float sq[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float x = xch[r * kTcXchStride + i];
        sq[i] = x * x;
    }
    float tot[32];
    if (hd >= 32) {
        // halving exchanges: lane L ends with the warp's 32 features summed for vector L
#pragma unroll
        for (int c = 32, b = 16; c > 1; c >>= 1, b >>= 1) {
            const bool up = (lane & b) != 0;
#pragma unroll
            for (int k = 0; k < c / 2; ++k) {
                const float send = up ? sq[k] : sq[k + c / 2];
                const float keep = up ? sq[k + c / 2] : sq[k];
                sq[k] = keep + __shfl_xor_sync(0xffffffffu, send, b);
            }
        }
        hs[(r >> 5) * 32 + lane] = sq[0];
        named_sync(1, kTcEpiThreads);
        const int w0 = (r / hd) * (hd >> 5);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float a = 0.0f;
            for (int w = w0; w < w0 + (hd >> 5); ++w) a += hs[w * 32 + i];
            tot[i] = a;
        }
    } else {  // a head is an aligned group of hd lanes
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float a = sq[i];
            for (int o = hd >> 1; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            tot[i] = a;
        }
    }
    if (normed) {
        const bool is_q = m < p.nq_cols;
        const float w = __ldg((is_q ? p.q_norm : p.k_norm) + (is_q ? m : m - p.nq_cols) % hd);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            xch[r * kTcXchStride + i] *= (1.0f / sqrtf(tot[i] / (float)hd + p.qk_eps)) * w;
    }
    named_sync(1, kTcEpiThreads);  // the rescaled rows, before RoPE reads partner features
}

template <int EPI>
__device__ void tc_epilogue_chunk(const TcArgs &p, int tile, int chunk, const float (&v)[32], const float (&old)[32],
                                  float *xch, int *s_row, const float *s_scale, int r) {
    const int j0 = chunk * 32;
    if constexpr (EPI == TC_STORE || EPI == TC_ADD) {
        const int m = tile * kTcBM + r;
        const int nj = min(32, p.n - j0);
        if (m < p.M) {
            float *col = p.y + (long long)j0 * p.ldy + m;
            if constexpr (EPI == TC_ADD) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < nj) col[(long long)i * p.ldy] = old[i] + v[i];
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < nj) col[(long long)i * p.ldy] = v[i];
            }
        }
        if (EPI == TC_ADD && p.nw) {  // the next RMSNorm's input and this tile's square sums
            float sq[32];
            const float wm = m < p.M ? __ldg(p.nw + m) : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float x = (m < p.M && i < nj) ? old[i] + v[i] : 0.0f;
                sq[i] = x * x;
                if (m < p.M && i < nj) {
                    __nv_bfloat16 hi, lo;
                    split_bf16(x * wm, hi, lo);
                    const long long o = (long long)(j0 + i) * p.ldy + m;
                    p.hb[o] = hi;
                    p.hb[o + p.hb_lo] = lo;
                }
            }
            // halving exchanges: lane L ends with the warp's 32 features summed for vector L
            const int lane = r & 31;
#pragma unroll
            for (int c = 32, b = 16; c > 1; c >>= 1, b >>= 1) {
                const bool up = (lane & b) != 0;
#pragma unroll
                for (int k = 0; k < c / 2; ++k) {
                    const float send = up ? sq[k] : sq[k + c / 2];
                    const float keep = up ? sq[k + c / 2] : sq[k];
                    sq[k] = keep + __shfl_xor_sync(0xffffffffu, send, b);
                }
            }
            xch[(r >> 5) * 32 + lane] = sq[0];
            named_sync(1, kTcEpiThreads);
            if (r < 32 && r < nj)
                p.ssq[(long long)tile * p.ss_ld + j0 + r] = ((xch[r] + xch[32 + r]) + xch[64 + r]) + xch[96 + r];
            named_sync(1, kTcEpiThreads);
        }
        return;
    } else {
    // SILU and QKV exchange values between features through shared memory,
    // scaled by the folded RMSNorm (1 where there is none); then thread
    // (warp q, lane i) of the four takes vector j0 + i and a run of
    // consecutive features, so its items are independent of one another and
    // its outputs leave as a few 16-byte stores
#pragma unroll
    for (int i = 0; i < 32; ++i) xch[r * kTcXchStride + i] = v[i] * s_scale[j0 + i];
    named_sync(1, kTcEpiThreads);
    const int lane = r & 31, q = r >> 5;
    const int j = j0 + lane;
    if constexpr (EPI == TC_SILU) {
        // gate features 16 q .. 16 q + 15 of the tile's 64 (rows f of the
        // exchange buffer; their up features are rows f + 64)
        constexpr int kF = kTcBM / 8;
        const int f0 = q * kF, g0 = tile * (kTcBM / 2) + f0;
        if (j < p.n && g0 < p.M) {
            float f[kF];
#pragma unroll
            for (int k = 0; k < kF; ++k) {
                const float gate = xch[(f0 + k) * kTcXchStride + lane];
                const float up = xch[(f0 + k + kTcBM / 2) * kTcXchStride + lane];
                f[k] = silu_tc(gate) * up;
            }
            __nv_bfloat16 *dst = p.yb + (long long)j * p.ldy + g0;
            const bool vec = g0 + kF <= p.M && (reinterpret_cast<uintptr_t>(dst) & 15) == 0 && (p.yb_lo & 7) == 0;
            __nv_bfloat16 hi[kF], lo[kF];
#pragma unroll
            for (int k = 0; k < kF; ++k) {
                if (p.yb_lo) {
                    split_bf16(f[k], hi[k], lo[k]);
                } else {
                    hi[k] = __float2bfloat16_rn(f[k]);
                    lo[k] = hi[k];
                }
            }
            if (vec) {
#pragma unroll
                for (int k = 0; k < kF; k += 8) {
                    *reinterpret_cast<uint4 *>(dst + k) = pack8_bf16(hi + k);
                    if (p.yb_lo) *reinterpret_cast<uint4 *>(dst + p.yb_lo + k) = pack8_bf16(lo + k);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kF; ++k)
                    if (g0 + k < p.M) {
                        dst[k] = hi[k];
                        if (p.yb_lo) dst[k + p.yb_lo] = lo[k];
                    }
            }
        }
    } else {
        if (p.q_norm) tc_qk_norm(p, tile * kTcBM + r, r, xch);
        // features 32 q .. 32 q + 31 of the tile: q columns, then k, then v
        constexpr int kF = kTcBM / 4;
        const int f0 = q * kF, m0 = tile * kTcBM + f0;
        const int nq = p.nq_cols, nkv = p.nkv_cols, total = nq + 2 * nkv;
        if (j < p.n && m0 < total) {
            const int pos = s_row[kTcMaxN + j], row = s_row[j];
            const bool pos_ok = pos >= 0 && pos < p.rope_rows;
            const int hd = p.head_dim, half = hd >> 1;
            const bool split_layout = p.rope_layout == DS_ROPE_HALF_SPLIT;
            float out[kF];
            // the run's region (q, k or v columns) and place in its head: with
            // hd a multiple of 32 the run lies inside one head (and, half-split
            // with hd >= 64, inside one half of it), so the rotation pairs and
            // partner features follow from the run's first feature
            const int base = m0 < nq ? 0 : (m0 < nq + nkv ? nq : nq + nkv);
            const int rend = m0 < nq ? nq : (m0 < nq + nkv ? nq + nkv : total);
            const bool whole_run = m0 + kF <= rend && hd % kF == 0 && (!split_layout || half % kF == 0);
            if (whole_run) {
                const int ih0 = (m0 - base) % hd;
                if (!pos_ok || base == nq + nkv) {  // v columns (or no angle): as they are
#pragma unroll
                    for (int k = 0; k < kF; ++k) out[k] = xch[(f0 + k) * kTcXchStride + lane];
                } else {
                    // the run's angles: pairs pair0 .. (half-split) or pair0 .. pair0 + 15 (interleaved)
                    const bool first_half = ih0 < half;
                    const int pair0 = split_layout ? (first_half ? ih0 : ih0 - half) : ih0 >> 1;
                    constexpr int kA = kF;  // angles loaded (the interleaved layout uses the first kF / 2)
                    const int na = split_layout ? kF : kF / 2;
                    const float *cp = p.rope_cos + (long long)pos * half + pair0;
                    const float *sp = p.rope_sin + (long long)pos * half + pair0;
                    float cs[kA], sn[kA];
                    if (((reinterpret_cast<uintptr_t>(cp) | reinterpret_cast<uintptr_t>(sp)) & 15) == 0) {
#pragma unroll
                        for (int k = 0; k < kA; k += 4) {
                            if (k < na) {
                                const float4 c4 = __ldg(reinterpret_cast<const float4 *>(cp + k));
                                const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sp + k));
                                cs[k] = c4.x; cs[k + 1] = c4.y; cs[k + 2] = c4.z; cs[k + 3] = c4.w;
                                sn[k] = s4.x; sn[k + 1] = s4.y; sn[k + 2] = s4.z; sn[k + 3] = s4.w;
                            } else {
                                cs[k] = cs[k + 1] = cs[k + 2] = cs[k + 3] = 1.0f;
                                sn[k] = sn[k + 1] = sn[k + 2] = sn[k + 3] = 0.0f;
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kA; ++k) {
                            cs[k] = k < na ? __ldg(cp + k) : 1.0f;
                            sn[k] = k < na ? __ldg(sp + k) : 0.0f;
                        }
                    }
                    if (split_layout) {
                        const int pf0 = first_half ? f0 + half : f0 - half;  // the partner run
#pragma unroll
                        for (int k = 0; k < kF; ++k) {
                            const float x = xch[(f0 + k) * kTcXchStride + lane];
                            const float o = xch[(pf0 + k) * kTcXchStride + lane];
                            out[k] = first_half ? x * cs[k] - o * sn[k] : o * sn[k] + x * cs[k];
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kF; ++k) {
                            const float x = xch[(f0 + k) * kTcXchStride + lane];
                            const float o = xch[(f0 + (k ^ 1)) * kTcXchStride + lane];
                            out[k] = (k & 1) == 0 ? x * cs[k >> 1] - o * sn[k >> 1] : o * sn[k >> 1] + x * cs[k >> 1];
                        }
                    }
                }
            } else {
                // narrow heads or a run across regions: one item at a time,
                // every item's inputs loaded before any output is stored
#pragma unroll
                for (int k = 0; k < kF; ++k) {
                    const int m = m0 + k, f = f0 + k;
                    const float x = xch[f * kTcXchStride + lane];
                    const bool rot = pos_ok && m < nq + nkv;
                    const int ih = (m < nq ? m : m - nq) % hd;
                    const bool first = split_layout ? ih < half : (ih & 1) == 0;
                    const int pair = split_layout ? (first ? ih : ih - half) : ih >> 1;
                    const int partner = split_layout ? (first ? f + half : f - half) : f ^ 1;
                    float cs = 1.0f, sn = 0.0f, o = 0.0f;
                    if (rot) {
                        cs = __ldg(p.rope_cos + (long long)pos * half + pair);
                        sn = __ldg(p.rope_sin + (long long)pos * half + pair);
                        o = xch[partner * kTcXchStride + lane];
                    }
                    out[k] = rot ? (first ? x * cs - o * sn : o * sn + x * cs) : x;
                }
            }
            if (m0 + kF <= nq) {  // q columns only: fp32 to the q rows
                float *dst = p.y + (long long)j * p.ldy + m0;
                if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                    for (int k = 0; k < kF; k += 4)
                        *reinterpret_cast<float4 *>(dst + k) = make_float4(out[k], out[k + 1], out[k + 2], out[k + 3]);
                } else {
#pragma unroll
                    for (int k = 0; k < kF; ++k) dst[k] = out[k];
                }
            } else if (m0 >= nq && row >= 0 && ((m0 + kF <= nq + nkv) || (m0 >= nq + nkv && m0 + kF <= total)) &&
                       p.kv_dtype == DS_BF16) {
                // one cache's columns only, bf16: to the position's cache row
                const bool is_k = m0 < nq + nkv;
                const int c0 = is_k ? m0 - nq : m0 - nq - nkv;
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(is_k ? p.k_cache : p.v_cache) +
                                     (long long)row * nkv + c0;
                __nv_bfloat16 b[kF];
#pragma unroll
                for (int k = 0; k < kF; ++k) b[k] = __float2bfloat16_rn(out[k]);
                if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                    for (int k = 0; k < kF; k += 8) *reinterpret_cast<uint4 *>(dst + k) = pack8_bf16(b + k);
                } else {
#pragma unroll
                    for (int k = 0; k < kF; ++k) dst[k] = b[k];
                }
            } else {  // a run that straddles q / k / v, or an fp32 cache: one item at a time
#pragma unroll
                for (int k = 0; k < kF; ++k) {
                    const int m = m0 + k;
                    if (m < nq) {
                        p.y[(long long)j * p.ldy + m] = out[k];
                    } else if (m < total && row >= 0) {
                        const int kv = m - nq;
                        if (kv < nkv)
                            store_as(p.k_cache, (long long)row * nkv + kv, p.kv_dtype, out[k]);
                        else
                            store_as(p.v_cache, (long long)row * nkv + kv - nkv, p.kv_dtype, out[k]);
                    }
                }
            }
        }
    }
    named_sync(1, kTcEpiThreads);
    }
}

template <int A_MN, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled stages
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    const int MS = p.msub;
    const bool one_acc = p.acc_bufs == 1;  // a single accumulator (MS x n_pad columns)
    const int a_bytes = MS * kTcABytes;        // the tile's weight sub-tiles
    const int b_bytes = p.n_pad * kTcBK * 2;  // one activation tile (the hi part when split)
    const int stage_bytes = a_bytes + b_bytes * (p.split ? 2 : 1);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + kTcMaxStages;
    uint64_t *acc_full = empty + kTcMaxStages;   // [2]
    uint64_t *acc_empty = acc_full + 2;          // [2]
    uint64_t *mma_done = acc_empty + 2;          // [1]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(mma_done + 1);
    int *s_flags = reinterpret_cast<int *>(s_tmem + 1);  // [0] abort, [1] last-arriver broadcast
    int *s_ok = s_flags + 2;                              // [2][4]
    int *s_row = s_ok + 8;                                // [2][kTcMaxN] cache row, position (q|k|v)
    float *s_scale = reinterpret_cast<float *>(s_row + 2 * kTcMaxN);  // [kTcMaxN] folded RMSNorm scales
    float *xch = s_scale + kTcMaxN;                                   // [128][33], then [4][32]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (p.K + kTcBK - 1) / kTcBK;
    const int T = p.m_tiles;
    const long long W = (long long)T * KB;
    const int G = gridDim.x;
    const long long u0 = W * blockIdx.x / G, u1 = W * (blockIdx.x + 1) / G;
    volatile int *abort_flag = s_flags;
    const uint32_t tmem_cols = (uint32_t)p.tmem_cols;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(mma_done, 1);
        s_flags[0] = 0;
        s_flags[1] = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    allow_dependent_launch();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // prologue: the first stages' weight boxes go out before the
            // previous kernel's output is awaited
            long long u = u0;
            int pre = (int)std::min<long long>(stages, u1 - u0);
            // the unit (tile, k-block) of every stage walked incrementally: no
            // division per stage (the issuing thread's instruction count is on
            // the critical path of the weight stream)
            auto issue_a = [&](int s, int tile, int kb) {
                for (int h = 0; h < MS; ++h) {
                    const int st = tile * MS + h;  // 128-feature sub-tile
                    unsigned char *sa = smem + (size_t)s * stage_bytes + h * kTcABytes;
                    if (A_MN) {
                        if (EPI == TC_SILU) {
                            tma_box_g2s(sa, &p.ta0, st * (kTcBM / 2), kb * kTcBK, &full[s], pol);
                            tma_box_g2s(sa + kTcABytes / 2, &p.ta1, st * (kTcBM / 2), kb * kTcBK, &full[s], pol);
                        } else {
                            tma_box_g2s(sa, &p.ta0, st * kTcBM, kb * kTcBK, &full[s], pol);
                            tma_box_g2s(sa + kTcABytes / 2, &p.ta0, st * kTcBM + kTcBM / 2, kb * kTcBK, &full[s], pol);
                        }
                    } else {
                        tma_box_g2s(sa, &p.ta0, kb * kTcBK, st * kTcBM, &full[s], pol);
                    }
                }
            };
            auto issue_b = [&](int s, int kb) {
                unsigned char *sb = smem + (size_t)s * stage_bytes + a_bytes;
                tma_box_g2s_nohint(sb, &p.tb, kb * kTcBK, 0, &full[s]);
                if (p.split) tma_box_g2s_nohint(sb + b_bytes, &p.tb, kb * kTcBK, p.b_lo_row, &full[s]);
            };
            const int tile0 = (int)(u0 / KB), kb0 = (int)(u0 - (long long)tile0 * KB);
            {
                int tile = tile0, kb = kb0;
                for (int i = 0; i < pre; ++i) {
                    mbar_arrive_expect_tx(&full[i], (uint32_t)stage_bytes);
                    issue_a(i, tile, kb);
                    if (++kb == KB) {
                        kb = 0;
                        ++tile;
                    }
                }
            }
            grid_dependency_wait();
            {
                int kb = kb0;
                for (int i = 0; i < pre; ++i) {
                    issue_b(i, kb);
                    if (++kb == KB) kb = 0;
                }
            }
            uint32_t fill = (uint32_t)pre;
            int tile = tile0, kb = kb0 + pre;
            while (kb >= KB) {
                kb -= KB;
                ++tile;
            }
            int s = pre % stages;
            uint32_t use = (uint32_t)(pre / stages);
            bool ok = true;
            for (u = u0 + pre; u < u1; ++u, ++fill) {
                if (!tc_wait(&empty[s], (use - 1) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                issue_a(s, tile, kb);
                issue_b(s, kb);
                if (++kb == KB) {
                    kb = 0;
                    ++tile;
                }
                if (++s == stages) {
                    s = 0;
                    ++use;
                }
            }
            // every copy issued has landed before the CTA may exit
            const uint32_t first = fill > (uint32_t)stages ? fill - stages : 0;
            for (uint32_t f = first; f < fill; ++f) {
                int dummy = 0;
                if (!mbar_wait(&full[f % stages], (f / stages) & 1, ok ? p.err : &dummy)) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            grid_dependency_wait();
            const uint32_t idesc = tc_idesc(A_MN, p.n_pad);
            const bool split = p.split != 0;
            const uint64_t b_lo_step = (uint64_t)(b_bytes >> 4);  // the lo activation tile, b_bytes further
            uint32_t fill = 0;
            int seg_i = 0;
            long long u = u0;
            TcSeg sg;
            bool ok = true;
            while (ok && tc_next_seg(u, u1, KB, sg)) {
                const int buf = one_acc ? 0 : (seg_i & 1);
                const int use = one_acc ? seg_i : (seg_i >> 1);  // earlier uses of this accumulator
                if (use >= 1 && !tc_wait(&acc_empty[buf], (use - 1) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * MS * p.n_pad);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++fill) {
                    const int s = fill % stages;
                    if (!tc_wait(&full[s], (fill / stages) & 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors of this stage formed once; every 16-row step and
                    // sub-tile only adds a constant to the 16-byte address field
                    // (the issuing thread's instruction count bounds the MMA rate)
                    const uint32_t sa0 = smem_u32(smem + (size_t)s * stage_bytes);
                    const uint64_t a0 = A_MN ? smem_desc(sa0, kTcABytes / 2, 1024) : smem_desc(sa0, 16, 1024);
                    const uint64_t b0 = smem_desc(sa0 + a_bytes, 16, 1024);
                    const uint32_t first = kb > sg.kb0 ? 1u : 0u;
#pragma unroll
                    for (int k = 0; k < kTcBK / 16; ++k) {
                        const uint64_t bd = b0 + (uint64_t)(k * 2);  // 32 bytes further per step
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (h < MS) {
                                const uint64_t ad = a0 + (uint64_t)(h * (kTcABytes >> 4) + k * (A_MN ? 128 : 2));
                                const uint32_t d = d_tmem + (uint32_t)(h * p.n_pad);
                                tc_mma(d, ad, bd, idesc, (first | (uint32_t)k) ? 1u : 0u);
                                if (split) tc_mma(d, ad, bd + b_lo_step, idesc, 1u);
                            }
                        }
                    }
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&acc_full[buf]);
                ++seg_i;
            }
            // nothing of ours may still be running on the tensor cores at exit
            tc_commit(mma_done);
            int dummy = 0;
            mbar_wait(mma_done, 0, ok ? p.err : &dummy);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        grid_dependency_wait();
        const int q = warp & 3;
        const int r = q * 32 + lane;  // accumulator lane = feature row of the tile
        const int et = threadIdx.x - 64;
        long long u = u0;
        int seg_i = 0;
        TcSeg sg;
        const int n_chunks = p.n_pad / 32;
        const size_t sub_floats = (size_t)kTcBM * p.n_pad;
        int pend[2] = {0, 0}, n_pend = 0;  // split tiles this CTA contributed to, in range order
        if (EPI == TC_QKV) {  // every vector's cache row and position, before any accumulator is awaited
            const int cap = p.max_blocks * p.block_tokens;
            for (int j = et; j < p.n_pad; j += kTcEpiThreads) {
                int row = -1, pos = -1;
                if (j < p.n) {
                    pos = __ldcg(p.pos + j);
                    if (pos >= 0 && pos < cap && pos < p.rope_rows) {
                        const int b = pos / p.block_tokens;
                        const long long sj = p.row_seq ? __ldcg(p.row_seq + j) : j;
                        const long long blk = p.block_table ? (long long)__ldcg(p.block_table + sj * p.max_blocks + b)
                                                            : sj * p.max_blocks + b;
                        const long long rr = blk * p.block_tokens + pos % p.block_tokens;
                        if (blk >= 0 && rr < p.cache_rows) row = (int)rr;
                    }
                    if (row < 0 && blockIdx.x == 0) flag_error(p.err, DS_ERR_POSITION);
                }
                s_row[j] = row;
                s_row[kTcMaxN + j] = pos;
            }
        }
        if (EPI == TC_QKV || EPI == TC_SILU) {  // the folded RMSNorm's scale of every vector
            for (int j = et; j < p.n_pad; j += kTcEpiThreads) {
                float sc = 1.0f;
                if (p.ssq_in && j < p.n) {
                    float tot = 0.0f;
                    for (int t0 = 0; t0 < p.ss_tiles; t0 += 8) {
                        float w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            w[k] = t0 + k < p.ss_tiles ? __ldcg(p.ssq_in + (long long)(t0 + k) * p.ss_ld + j) : 0.0f;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (t0 + k < p.ss_tiles) tot += w[k];
                    }
                    sc = 1.0f / sqrtf(tot / (float)p.ss_d + p.eps);
                }
                s_scale[j] = sc;
            }
            named_sync(1, kTcEpiThreads);
        }
        while (tc_next_seg(u, u1, KB, sg)) {
            const int buf = one_acc ? 0 : (seg_i & 1);
            const int use = one_acc ? seg_i : (seg_i >> 1);
            // the four warps agree on whether the accumulator arrived, so none
            // of them can be left alone at a named barrier
            bool ok = __all_sync(0xffffffffu, tc_wait(&acc_full[buf], use & 1, abort_flag, p.err));
            if (lane == 0) s_ok[(seg_i & 1) * 4 + q] = ok ? 1 : 0;
            named_sync(1, kTcEpiThreads);
            ok = s_ok[(seg_i & 1) * 4 + 0] && s_ok[(seg_i & 1) * 4 + 1] && s_ok[(seg_i & 1) * 4 + 2] &&
                 s_ok[(seg_i & 1) * 4 + 3];
            tc_fence_after();
            const bool whole = sg.kb0 == 0 && sg.kb1 == KB;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * MS * p.n_pad);
            if (!ok) break;
            if (whole) {
                for (int h = 0; h < MS; ++h)
                    for (int c = 0; c < n_chunks; ++c) {
                        float v[32], old[32];
                        if (EPI == TC_ADD) tc_load_residual(p, sg.tile * MS + h, c, r, old);
                        tmem_ld32(tbase + h * p.n_pad + c * 32, v);
                        if (h == MS - 1 && c == n_chunks - 1) {  // the buffer may be reused once every lane has read it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&acc_empty[buf]);
                        }
                        tc_epilogue_chunk<EPI>(p, sg.tile * MS + h, c, v, old, xch, s_row, s_scale, r);
                    }
            } else {
                // partial accumulators to this (CTA, tile) slot, feature-fastest per sub-tile
                float *slot = p.partials + ((size_t)blockIdx.x + sg.tile) * MS * sub_floats;
                for (int h = 0; h < MS; ++h)
                    for (int c = 0; c < n_chunks; ++c) {
                        float v[32];
                        tmem_ld32(tbase + h * p.n_pad + c * 32, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) slot[h * sub_floats + (size_t)(c * 32 + i) * kTcBM + r] = v[i];
                    }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
                // this contribution has landed: arrive on the tile's counter
                __threadfence();
                named_sync(1, kTcEpiThreads);
                if (et == 0) atomicAdd(p.counters + sg.tile, 1);
                if (n_pend < 2) pend[n_pend++] = sg.tile;
            }
            ++seg_i;
        }
        // The split tiles (at most two: the range's first and last segments)
        // are finished together by their contributors once every partial has
        // arrived: contributor k of nc takes the tile's 32-vector chunks k,
        // k + nc, ...  A contributor waits only here, after all of its own
        // partials have been written, so every wait ends.  The counter then
        // counts departures on top of the nc arrivals; the last to leave sets
        // it back to zero for the next launch.
        for (int pi = n_pend - 1; pi >= 0; --pi) {  // (an abort ends the waits: all threads leave together)
            const int tile = pend[pi];
            // contributors of this tile: the CTAs holding its first and last unit
            const long long tu0 = (long long)tile * KB, tu1 = tu0 + KB - 1;
            const int c_first = (int)(((tu0 + 1) * G - 1) / W);
            const int c_last = (int)(((tu1 + 1) * G - 1) / W);
            const int nc = c_last - c_first + 1, kc = (int)blockIdx.x - c_first;
            if (et == 0) s_flags[1] = tc_wait_count(p.counters + tile, nc, abort_flag, p.err) ? 1 : 0;
            named_sync(1, kTcEpiThreads);
            const bool ready = s_flags[1] != 0;  // one answer for the four warps
            named_sync(1, kTcEpiThreads);
            if (!ready) break;
            __threadfence();
            for (int task = kc; task < MS * n_chunks; task += nc) {
                const int h = task / n_chunks, c = task - h * n_chunks;
                float v[32], old[32];
                if (EPI == TC_ADD) tc_load_residual(p, tile * MS + h, c, r, old);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                // up to kTcMaxContrib contributors' partials requested at once,
                // added in CTA order
                for (int c0 = c_first; c0 <= c_last; c0 += kTcMaxContrib) {
                    float t[kTcMaxContrib][32];
#pragma unroll
                    for (int k = 0; k < kTcMaxContrib; ++k)
                        if (c0 + k <= c_last) {
                            const float *src = p.partials + ((size_t)(c0 + k) + tile) * MS * sub_floats + h * sub_floats;
#pragma unroll
                            for (int i = 0; i < 32; ++i) t[k][i] = __ldcg(src + (size_t)(c * 32 + i) * kTcBM + r);
                        }
#pragma unroll
                    for (int k = 0; k < kTcMaxContrib; ++k)
                        if (c0 + k <= c_last)
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] += t[k][i];
                }
                tc_epilogue_chunk<EPI>(p, tile * MS + h, c, v, old, xch, s_row, s_scale, r);
            }
            named_sync(1, kTcEpiThreads);
            if (et == 0) {
                const int prev = atomicAdd(p.counters + tile, 1);
                if (prev == 2 * nc - 1) p.counters[tile] = 0;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

// ---------------------------------------------------------------- host
// The MMA's N: the vector count rounded up to whole 32-column chunks of the
// accumulator (the epilogue reads 32 columns at a time).
int tc_n_pad(int n) { return std::max(32, (n + 31) / 32 * 32); }

int tc_tmem_cols(int acc_bufs, int msub, int n_pad) {
    int cols = 32;
    while (cols < acc_bufs * msub * n_pad) cols *= 2;
    return cols;
}

int tc_stages(int n_pad, int split, int msub) {
    const size_t stage = (size_t)msub * kTcABytes + (size_t)n_pad * kTcBK * 2 * (split ? 2 : 1);
    const size_t fixed = 1024 + 256 + kTcSmemInts * 4 + (size_t)kTcBM * (kTcXchStride + 1) * 4 + 64;
    int s = (int)((kTcSmemLimit - fixed) / stage);
    return std::min(s, kTcMaxStages);
}

size_t tc_smem_bytes(int n_pad, int split, int msub, int stages) {
    const size_t stage = (size_t)msub * kTcABytes + (size_t)n_pad * kTcBK * 2 * (split ? 2 : 1);
    return 1024 + (size_t)stages * stage + 256 + kTcSmemInts * 4 + (size_t)kTcBM * (kTcXchStride + 1) * 4 + 64;
}

int tc_m_tiles(int M, int epi) { return epi == TC_SILU ? (M + kTcBM / 2 - 1) / (kTcBM / 2) : (M + kTcBM - 1) / kTcBM; }

int tc_grid(int m_tiles, int K) {
    const long long W = (long long)m_tiles * ((K + kTcBK - 1) / kTcBK);
    return (int)std::min<long long>(sm_count(), W);
}

size_t tc_partial_floats(int m_tiles, int n_pad, int msub) {
    return (size_t)(sm_count() + m_tiles) * msub * kTcBM * n_pad;
}

bool tc_make_maps(TcArgs &a, const void *A0, const void *A1, long long a_row_stride, const void *X) {
    if (a.a_mn) {
        // [K][M] (M contiguous): boxes of 64 features x 64 rows
        if (!encode_tiled_2d(&a.ta0, A0, DS_BF16, a.M, a.K, a_row_stride, 64, kTcBK, true)) return false;
        if (A1 && !encode_tiled_2d(&a.ta1, A1, DS_BF16, a.M, a.K, a_row_stride, 64, kTcBK, true)) return false;
    } else {
        // [M][K] (K contiguous): boxes of 64 columns x 128 rows
        if (!encode_tiled_2d(&a.ta0, A0, DS_BF16, a.K, a.M, a_row_stride, kTcBK, kTcBM, true)) return false;
    }
    // split: hi rows [0, n) then lo rows [b_lo_row, b_lo_row + n)
    const long long x_rows = a.split ? (long long)a.b_lo_row + a.n : a.n;
    return encode_tiled_2d(&a.tb, X, DS_BF16, a.K, x_rows, (long long)a.K * 2, kTcBK, a.n_pad, true);
}

template <int A_MN, int EPI>
static cudaError_t launch_tc_t(const TcArgs &a, int grid, cudaStream_t stream, bool pdl) {
    const size_t smem = tc_smem_bytes(a.n_pad, a.split, a.msub, a.stages);
    if (smem > kTcSmemLimit) return cudaErrorInvalidValue;
    return launch_ex(tc_gemm_kernel<A_MN, EPI>, dim3(grid), dim3(kTcThreads), smem, stream, pdl, a);
}

static bool g_tc_ready = false;

cudaError_t launch_tc_gemm(const TcArgs &a, int grid, cudaStream_t stream, bool pdl) {
    if (a.n_pad < 32 || a.n_pad > 256 || a.n_pad % 32 || a.stages < 2 || a.stages > kTcMaxStages) return cudaErrorInvalidValue;
    if ((a.msub != 1 && a.msub != 2) || a.tmem_cols < (a.acc_bufs == 1 ? 1 : 2) * a.msub * a.n_pad ||
        a.tmem_cols > 512)
        return cudaErrorInvalidValue;
    if (!g_tc_ready) {
        cudaError_t e = prepare_tc_kernels();
        if (e != cudaSuccess) return e;
    }
    if (a.a_mn) {
        switch (a.epi) {
            case TC_STORE: return launch_tc_t<1, TC_STORE>(a, grid, stream, pdl);
            case TC_ADD: return launch_tc_t<1, TC_ADD>(a, grid, stream, pdl);
            case TC_SILU: return launch_tc_t<1, TC_SILU>(a, grid, stream, pdl);
            case TC_QKV: return launch_tc_t<1, TC_QKV>(a, grid, stream, pdl);
            default: return cudaErrorInvalidValue;
        }
    }
    if (a.epi == TC_STORE) return launch_tc_t<0, TC_STORE>(a, grid, stream, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t prepare_tc_kernels() {
    const void *fns[] = {(const void *)tc_gemm_kernel<1, TC_STORE>, (const void *)tc_gemm_kernel<1, TC_ADD>,
                         (const void *)tc_gemm_kernel<1, TC_SILU>, (const void *)tc_gemm_kernel<1, TC_QKV>,
                         (const void *)tc_gemm_kernel<0, TC_STORE>};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemLimit);
        if (e != cudaSuccess) return e;
    }
    g_tc_ready = true;
    return cudaSuccess;
}

}  // namespace ds

// =====================================================================
// C ABI
// =====================================================================
using namespace ds;

namespace {

size_t tc_ws_bytes(int64_t n, int64_t M, int64_t K, int epi) {
    const int n_pad = tc_n_pad((int)n);
    const int T = tc_m_tiles((int)M, epi);
    (void)K;
    return kWsHeader + align_up((size_t)T * 4, 256) + tc_partial_floats(T, n_pad, 1) * 4;
}

int tc_check(const void *A, int64_t a_len, const void *X, int64_t x_len, int64_t n, int64_t rows, int64_t cols,
             const float *Y, int64_t y_len, int64_t y_need, int64_t K) {
    if (n < 1 || rows < 1 || cols < 1) return DS_EMPTY_DIMENSION;
    if (rows > DS_MAX_DIM || cols > DS_MAX_DIM) return DS_DIMENSION_TOO_LARGE;
    if (n > 256) return DS_DIMENSION_TOO_LARGE;
    if (a_len != rows * cols) return DS_GEMV_A_LENGTH_MISMATCH;
    if (x_len != n * K) return DS_GEMV_X_LENGTH_MISMATCH;
    if (y_len != y_need) return DS_A_LENGTH_MISMATCH;
    if (!A || !X || !Y) return DS_BAD_ARGUMENT;
    if (((uintptr_t)A | (uintptr_t)X) & 15) return DS_BAD_ARGUMENT;
    if ((cols * 2) % 16) return DS_BAD_ARGUMENT;  // row strides of both operands: whole 16-byte units
    if ((K * 2) % 16) return DS_BAD_ARGUMENT;
    return DS_OK;
}

int tc_run(const void *A, const void *X, int64_t n, int64_t M, int64_t K, int a_mn, long long a_row_stride, float *Y,
           void *ws, size_t ws_bytes, cudaStream_t s) {
    TcArgs a = {};
    a.a_mn = a_mn;
    a.M = (int)M;
    a.K = (int)K;
    a.n = (int)n;
    a.n_pad = tc_n_pad((int)n);
    a.epi = TC_STORE;
    a.msub = 1;
    a.acc_bufs = 2;
    a.m_tiles = tc_m_tiles(a.M, a.epi);
    a.stages = tc_stages(a.n_pad, 0, 1);
    a.tmem_cols = tc_tmem_cols(a.acc_bufs, a.msub, a.n_pad);
    a.y = Y;
    a.ldy = (int)M;
    if (!ws || ws_bytes < tc_ws_bytes(n, M, K, a.epi)) return DS_WORKSPACE_TOO_SMALL;
    char *w = static_cast<char *>(ws);
    a.err = reinterpret_cast<int *>(w);
    a.counters = reinterpret_cast<int *>(w + kWsHeader);
    a.partials = reinterpret_cast<float *>(w + kWsHeader + align_up((size_t)a.m_tiles * 4, 256));
    if (!tc_make_maps(a, A, nullptr, a_row_stride, X)) return DS_CUDA_ERROR;
    const int grid = tc_grid(a.m_tiles, a.K);
    return launch_tc_gemm(a, grid, s, false) == cudaSuccess ? DS_OK : DS_CUDA_ERROR;
}

}  // namespace

extern "C" DS_API size_t ds_gemm_workspace_bytes(int64_t n, int64_t rows, int64_t cols) {
    if (n < 1 || n > 256 || rows < 1 || cols < 1) return 0;
    // the larger of the two orientations' needs
    return std::max(tc_ws_bytes(n, cols, rows, TC_STORE), tc_ws_bytes(n, rows, cols, TC_STORE));
}

extern "C" DS_API int ds_gemm_transposed(const void *A, int64_t a_len, const void *X, int64_t x_len, int64_t n,
                                         int64_t rows, int64_t cols, float *Y, int64_t y_len, void *workspace,
                                         size_t workspace_bytes, ds_stream_t stream) {
    int st = tc_check(A, a_len, X, x_len, n, rows, cols, Y, y_len, n * cols, rows);
    if (st != DS_OK) return st;
    return tc_run(A, X, n, cols, rows, 1, cols * 2, Y, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

extern "C" DS_API int ds_gemm(const void *W, int64_t w_len, const void *X, int64_t x_len, int64_t n, int64_t rows,
                              int64_t cols, float *Y, int64_t y_len, void *workspace, size_t workspace_bytes,
                              ds_stream_t stream) {
    int st = tc_check(W, w_len, X, x_len, n, rows, cols, Y, y_len, n * rows, cols);
    if (st != DS_OK) return st;
    return tc_run(W, X, n, rows, cols, 0, cols * 2, Y, workspace, workspace_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}
