// Internal interface of the tensor-core (tcgen05) batched projections.
#pragma once

#include "internal.h"

#include <cuda_bf16.h>

namespace ds {

// Encode a 2-D tensor map over a row-major matrix of `rows` rows of `cols`
// elements (dtype DS_F32 / DS_BF16) with rows `row_stride` bytes apart, boxes
// of box_cols x box_rows elements, 128-byte swizzled or not.  False if the
// driver refuses.
bool encode_tiled_2d(CUtensorMap *map, const void *base, int dtype, long long cols, long long rows,
                     long long row_stride, int box_cols, int box_rows, bool swizzle128);

// The same for a 3-D map: dims[0] innermost, strides in bytes of dims 1 and 2.
bool encode_tiled_3d(CUtensorMap *map, const void *base, int dtype, const long long dims[3], const long long strides[2],
                     const int box[3], bool swizzle128);

// Fused epilogues of the batched projection kernel.
enum { TC_STORE = 0, TC_ADD = 1, TC_SILU = 2, TC_QKV = 3 };

struct TcArgs {
    CUtensorMap ta0;  // weights: [K][M] boxes {64 features, 64 rows} (a_mn) or [M][K] boxes {64, 128}
    CUtensorMap ta1;  // TC_SILU: the up columns' map (ta0 holds the gate columns)
    CUtensorMap tb;   // activations [n][K] bf16, boxes {64, n_pad}; split: [2][rows][K], hi rows then lo rows
    int a_mn;         // 1: weights [K][M], M contiguous; 0: [M][K], K contiguous
    int M, K, n, n_pad;
    int split;        // 1: each activation is hi + lo, two bf16 rows b_lo_row apart; both are multiplied
    int b_lo_row;
    int epi, m_tiles, stages, tmem_cols;
    int msub;         // 128-feature sub-tiles per tile (1 or 2): a tile's sub-tiles share one activation tile
    int acc_bufs;     // TMEM accumulators (1: a tile's MMAs wait for the previous tile's epilogue; else 2)
    float *y;             // TC_STORE / TC_ADD: y[s * ldy + m]; TC_QKV: q [n][ldy]
    __nv_bfloat16 *yb;    // TC_SILU: silu(gate) * up as bf16, yb[s * ldy + g] (hi part when yb_lo > 0)
    long long yb_lo;      // TC_SILU: elements from the hi part to the lo part (0: hi only)
    int ldy;
    // TC_QKV: RoPE on the q and k columns, K/V written at each sequence's pos
    const int *pos;
    const int *block_table;
    int max_blocks, block_tokens;
    long long cache_rows;
    const float *rope_cos, *rope_sin;
    int rope_rows;
    int nq_cols, nkv_cols, head_dim, rope_layout;
    void *k_cache, *v_cache;
    int kv_dtype;
    // TC_QKV: QK-norm before RoPE (null: none), every q / k head scaled by
    // 1/sqrt(mean of its squares + qk_eps) and by these [head_dim] weights
    const float *q_norm, *k_norm;
    float qk_eps;
    // the sequence whose blocks row s addresses: row_seq[s], or s when null
    // (a prompt chunk of one sequence gives every row the same sequence)
    const int *row_seq;
    // TC_ADD with nw set: the next RMSNorm folded in.  Besides y += acc it
    // writes x * nw (x the updated residual) as bf16 hi/lo to hb[s * ldy + m]
    // (lo part hb_lo elements further) and each 128-feature tile's square sums
    // of x to ssq[tile * ss_ld + s].
    const float *nw;
    __nv_bfloat16 *hb;
    long long hb_lo;
    float *ssq;
    // TC_QKV / TC_SILU with ssq_in set: the consuming side of that norm.  The
    // output of vector s is scaled by 1 / sqrt(sum_t ssq_in[t * ss_ld + s] /
    // ss_d + eps) (t < ss_tiles, added in order) before RoPE or SiLU.
    const float *ssq_in;
    int ss_tiles, ss_ld, ss_d;
    float eps;
    // split tiles: partial accumulators and arrival counters (zero between launches)
    float *partials;
    int *counters;
    int *err;
};

int tc_n_pad(int n);
// TMEM columns to allocate for acc_bufs accumulators of msub sub-tiles of
// n_pad columns (a power of two, at least 32).
int tc_tmem_cols(int acc_bufs, int msub, int n_pad);
int tc_stages(int n_pad, int split, int msub);
int tc_m_tiles(int M, int epi);
int tc_grid(int m_tiles, int K);
size_t tc_partial_floats(int m_tiles, int n_pad, int msub);
// Encode a.ta0 (and a.ta1 from A1 when set) and a.tb.
bool tc_make_maps(TcArgs &a, const void *A0, const void *A1, long long a_row_stride, const void *X);
cudaError_t launch_tc_gemm(const TcArgs &a, int grid, cudaStream_t stream, bool pdl);
// The bf16 pair (hi, lo) with hi + lo = v to 16 significant bits: the form in
// which a batched projection takes an fp32 activation.
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}
// Eight bf16 values as one 16-byte word, b[0] at the lowest address.
__device__ __forceinline__ uint4 pack8_bf16(const __nv_bfloat16 *b) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = (uint32_t)__bfloat16_as_ushort(b[2 * k]) | ((uint32_t)__bfloat16_as_ushort(b[2 * k + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}
cudaError_t prepare_tc_kernels();

}  // namespace ds
