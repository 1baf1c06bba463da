"""Batched projections on the tensor cores (ds_gemm_transposed, ds_gemm)
through the C ABI against the oracle's mat-vec applied to every row: ragged
tiles and k-blocks, 1..256 vectors, split and whole tiles, and the decode
step's full-size shapes (the output head checked on sampled rows)."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import FP32_TOL, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import abi
    return abi


def bf16_rows(n, k, seed):
    return synth.normal((n * k,), seed=seed, dtype=torch.bfloat16)


def oracle_rows_t(Ah, Xh, n, rows, cols):
    Ab = synth.to_numpy_storage(Ah)
    X = O.bf16_bits_to_f64(synth.to_numpy_storage(Xh)).reshape(n, rows)
    return np.stack([O.gemv_transposed(Ab, X[s], rows, cols, O.DT_BF16) for s in range(n)])


@pytest.mark.parametrize("rows,cols,n", [
    (64, 128, 1),        # one tile, one k-block
    (1000, 200, 3),      # ragged k-block and ragged tile
    (200, 1000, 17),     # more tiles than k-blocks
    (512, 384, 256),     # the widest batch
    (1024, 1024, 100),
    (4096, 6144, 64),    # 8B q|k|v shape, 64 sequences
    (14336, 4096, 64),   # 8B down shape: long k, few tiles (split tiles)
    (4096, 4096, 33),
])
def test_gemm_transposed_matches_oracle(A, rows, cols, n):
    Ah = bf16_rows(rows, cols, seed=rows + cols)
    Xh = bf16_rows(n, rows, seed=rows * 7 + n)
    Ad, Xd = Ah.cuda(), Xh.cuda()
    Y = torch.full((n, cols), float("nan"), device="cuda")
    ws = A.workspace(A.lib.ds_gemm_workspace_bytes(n, rows, cols))
    A.ds_gemm_transposed(Ad, Xd, n, rows, cols, Y, ws)
    ref = oracle_rows_t(Ah, Xh, n, rows, cols)
    got = host(Y)
    for s in range(n):
        assert rel_err(got[s], ref[s]) <= FP32_TOL, s
    Y2 = torch.empty_like(Y)
    A.ds_gemm_transposed(Ad, Xd, n, rows, cols, Y2, ws)
    assert torch.equal(Y, Y2)  # bit-stable
    assert A.ds_workspace_error(ws) == 0


@pytest.mark.parametrize("rows,cols,n", [(1000, 512, 5), (128, 64, 1), (300, 4096, 64)])
def test_gemm_untransposed_matches_oracle(A, rows, cols, n):
    Wh = bf16_rows(rows, cols, seed=rows * 3 + cols)
    Xh = bf16_rows(n, cols, seed=cols + n)
    Y = torch.full((n, rows), float("nan"), device="cuda")
    ws = A.workspace(A.lib.ds_gemm_workspace_bytes(n, rows, cols))
    A.ds_gemm(Wh.cuda(), Xh.cuda(), n, rows, cols, Y, ws)
    Wb = synth.to_numpy_storage(Wh)
    X = O.bf16_bits_to_f64(synth.to_numpy_storage(Xh)).reshape(n, cols)
    got = host(Y)
    for s in range(n):
        assert rel_err(got[s], O.gemv(Wb, X[s], rows, cols, O.DT_BF16)) <= FP32_TOL, s
    assert A.ds_workspace_error(ws) == 0


def test_gemm_head_full_size_on_sampled_rows(A):
    """The 8B output head (128,256 x 4096) for 64 sequences; 1,500 vocab rows
    sampled and checked against the oracle row by row."""
    V, d, n = 128256, 4096, 64
    Wh = bf16_rows(V, d, seed=11)
    Xh = bf16_rows(n, d, seed=12)
    Y = torch.full((n, V), float("nan"), device="cuda")
    ws = A.workspace(A.lib.ds_gemm_workspace_bytes(n, V, d))
    A.ds_gemm(Wh.cuda(), Xh.cuda(), n, V, d, Y, ws)
    got = host(Y)
    assert np.isfinite(got).all()
    g = np.random.default_rng(0)
    rows = np.sort(np.concatenate([g.choice(V, 1498, replace=False), [0, V - 1]]))
    Wsub = synth.to_numpy_storage(Wh.view(V, d)[torch.from_numpy(rows)])
    X = O.bf16_bits_to_f64(synth.to_numpy_storage(Xh)).reshape(n, d)
    for s in (0, 1, 31, 63):
        ref = O.gemv(Wsub, X[s], len(rows), d, O.DT_BF16)
        assert rel_err(got[s][rows], ref) <= FP32_TOL, s
