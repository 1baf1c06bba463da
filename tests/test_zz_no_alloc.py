"""ds_gemv_transposed_noalloc against ds_gemv_transposed, through the C ABI.

The no-allocation variant is for callers that cannot allocate device memory
(their device memory belongs to another allocator, or they receive only an
operation's inputs and outputs); its split-reduction scratch lives in a fixed
area inside the library.  This file is collected last so that a run stopping
at the first failure has already run every other test, and it must pass both
on its own in a fresh process and after the rest of the suite.
"""
import pytest
import torch

from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import FP32_TOL, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import abi
    return abi


@pytest.mark.parametrize("rows,cols,dt", [(4096, 6144, torch.bfloat16), (777, 1000, torch.float32),
                                          (14336, 4096, torch.bfloat16), (2, 3, torch.float32)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(A, rows, cols, dt):
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
        assert torch.isfinite(got).all()


def test_noalloc_refuses_shapes_beyond_its_area(A):
    limit = A.lib.ds_gemv_transposed_noalloc_max_bytes()
    assert limit == 1 << 20
    rows, cols = 64, 1 << 20  # scratch for this many bands exceeds the area
    assert A.ds_gemv_workspace_bytes(rows, cols, A.DS_F32) > limit
    fake = torch.empty(1, device="cuda")
    code = A.lib.ds_gemv_transposed_noalloc(fake.data_ptr(), rows * cols, A.DS_F32, fake.data_ptr(), rows, rows,
                                            cols, fake.data_ptr(), cols, A.stream_handle())
    assert code == A.DS_DIMENSION_TOO_LARGE
