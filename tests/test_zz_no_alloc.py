"""ds_gemv_transposed_noalloc against ds_gemv_transposed and the oracle,
through the C ABI.

The no-allocation variant is for callers that cannot allocate device memory
(their device memory belongs to another allocator, or they receive only an
operation's inputs and outputs); its split-reduction scratch lives in a fixed
area inside the library.  Its tests are marked run_last (the suite's conftest
moves them to the end of the run) so that a run stopping at the first failure
has already run every other test; they must pass both on their own in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import FP32_TOL, host, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.run_last]


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import abi
    return abi


def oracle_gemv_t(Ah, xh, rows, cols, dt):
    code = O.DT_BF16 if dt == torch.bfloat16 else O.DT_F32
    return O.gemv_transposed(host(Ah), host(xh).astype(np.float64), rows, cols, code)


@pytest.mark.parametrize("rows,cols,dt", [(4096, 6144, torch.bfloat16), (777, 1000, torch.float32),
                                          (14336, 4096, torch.bfloat16), (2, 3, torch.float32)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(A, rows, cols, dt):
    assert A.ds_gemv_transposed_noalloc_error() == 0  # nothing left over from earlier calls
    for call in range(2):  # the shared scratch area must be ready again for the second call
        Ah = synth.normal((rows * cols,), seed=rows + cols + call, dtype=dt).cuda()
        xh = synth.normal((rows,), seed=rows * 7 + call).cuda()
        ref = torch.full((cols,), float("nan"), device="cuda")
        ws = A.workspace(A.ds_gemv_workspace_bytes(rows, cols, A.dtype_code(Ah)))
        A.ds_gemv_transposed(Ah, xh, rows, cols, ref, ws)
        got = torch.full((cols,), float("nan"), device="cuda")
        A.ds_gemv_transposed_noalloc(Ah, xh, rows, cols, got)
        torch.cuda.synchronize()
        assert rel_err(host(got), host(ref)) <= FP32_TOL
        assert rel_err(host(got), oracle_gemv_t(Ah, xh, rows, cols, dt)) <= FP32_TOL
        assert torch.isfinite(got).all()
        assert A.ds_gemv_transposed_noalloc_error() == 0


def test_noalloc_plain_path_needs_no_scratch(A):
    """A matrix the streamed kernel cannot take (a row of an odd number of
    fp32 values) runs the plain-load kernel, which uses no scratch, so it is
    accepted even where the streamed path's nominal scratch would not fit."""
    rows, cols = 4, (1 << 18) + 1
    assert A.ds_gemv_workspace_bytes(rows, cols, A.DS_F32) > A.lib.ds_gemv_transposed_noalloc_max_bytes()
    for call in range(2):
        Ah = synth.normal((rows * cols,), seed=50 + call).cuda()
        xh = synth.normal((rows,), seed=60 + call).cuda()
        got = torch.full((cols,), float("nan"), device="cuda")
        A.ds_gemv_transposed_noalloc(Ah, xh, rows, cols, got)
        torch.cuda.synchronize()
        assert rel_err(host(got), oracle_gemv_t(Ah, xh, rows, cols, torch.float32)) <= FP32_TOL
        assert A.ds_gemv_transposed_noalloc_error() == 0


def test_noalloc_refuses_shapes_beyond_its_area(A):
    limit = A.lib.ds_gemv_transposed_noalloc_max_bytes()
    assert limit == 1 << 20
    rows, cols = 64, 1 << 20  # scratch for this many bands exceeds the area
    assert A.ds_gemv_workspace_bytes(rows, cols, A.DS_F32) > limit
    fake = torch.empty(4, device="cuda")  # 16-byte aligned: the streamed path's shape
    code = A.lib.ds_gemv_transposed_noalloc(fake.data_ptr(), rows * cols, A.DS_F32, fake.data_ptr(), rows, rows,
                                            cols, fake.data_ptr(), cols, A.stream_handle())
    assert code == A.DS_DIMENSION_TOO_LARGE
