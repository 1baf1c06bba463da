"""The C ABI on the host, without a GPU: the library loads, exports every
symbol the header declares, names its status codes, and refuses bad
arguments with the contract's codes before touching the device."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decode_step.h")


@pytest.fixture(scope="module")
def abi():
    from autoregressive_decode_step_gb300 import build
    build.build()
    from autoregressive_decode_step_gb300 import abi as A
    return A


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DS_API\s+[\w\s\*]+?\**\s*(ds_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ds_gemv_transposed", "ds_gemv", "ds_residual_add", "ds_add_rmsnorm", "ds_rope",
                     "ds_kv_cache_append", "ds_gqa_decode_attn", "ds_silu_mul", "ds_greedy_argmax", "ds_sample",
                     "ds_decode_step", "ds_model_create", "ds_status_name"):
        assert required in names


def test_library_exports_every_declared_symbol(abi):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(abi.lib, n), n


def test_status_names_follow_the_contract_vocabulary(abi):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "p1_status_contract.json")))
    for code, meaning in g["codes"].items():
        assert abi.status_name(int(code)) == "ds_" + meaning
    assert abi.status_name(1234) == "ds_code_out_of_range"
    assert abi.status_name(559) == "ds_code_out_of_range"


def test_residual_dims_check_page_examples(abi):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "p1_status_contract.json")))
    for case in g["residual_dims_check"]:
        assert abi.lib.ds_residual_dims_check(*case["args"]) == case["status"]
    assert abi.lib.ds_residual_dims_check(0, 0, 0) == abi.DS_EMPTY_DIMENSION
    assert abi.lib.ds_residual_dims_check(g["max_dim"] + 1, g["max_dim"] + 1, g["max_dim"] + 1) == \
        abi.DS_DIMENSION_TOO_LARGE


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every case below is refused on the host


def test_gemv_refusals(abi):
    L = abi.lib
    f = L.ds_gemv_transposed
    assert f(FAKE, 6, 0, FAKE, 2, 0, 3, FAKE, 3, FAKE, 1 << 20, None) == abi.DS_EMPTY_DIMENSION
    assert f(FAKE, 6, 0, FAKE, 2, 2, (1 << 24) + 1, FAKE, 3, FAKE, 1 << 20, None) == abi.DS_DIMENSION_TOO_LARGE
    assert f(FAKE, 5, 0, FAKE, 2, 2, 3, FAKE, 3, FAKE, 1 << 20, None) == abi.DS_GEMV_A_LENGTH_MISMATCH
    assert f(FAKE, 6, 0, FAKE, 3, 2, 3, FAKE, 3, FAKE, 1 << 20, None) == abi.DS_GEMV_X_LENGTH_MISMATCH
    assert f(FAKE, 6, 0, FAKE, 2, 2, 3, FAKE, 4, FAKE, 1 << 20, None) == abi.DS_A_LENGTH_MISMATCH
    assert f(FAKE, 6, 7, FAKE, 2, 2, 3, FAKE, 3, FAKE, 1 << 20, None) == abi.DS_BAD_DTYPE
    assert f(FAKE, 6, 0, FAKE, 2, 2, 3, FAKE, 3, None, 0, None) == abi.DS_WORKSPACE_TOO_SMALL
    g = L.ds_gemv
    assert g(FAKE, 6, 0, FAKE, 3, 2, 3, FAKE, 3, None) == abi.DS_A_LENGTH_MISMATCH
    assert g(FAKE, 6, 0, FAKE, 2, 2, 3, FAKE, 2, None) == abi.DS_GEMV_X_LENGTH_MISMATCH


def test_glue_refusals(abi):
    L = abi.lib
    assert L.ds_residual_add(FAKE, 2, FAKE, 6, FAKE, 6, None) == abi.DS_A_LENGTH_MISMATCH
    assert L.ds_residual_add(FAKE, 6, FAKE, 5, FAKE, 6, None) == abi.DS_B_LENGTH_MISMATCH
    assert L.ds_residual_add(FAKE, 0, FAKE, 0, FAKE, 0, None) == abi.DS_EMPTY_DIMENSION
    assert L.ds_add_rmsnorm(FAKE, 4095, FAKE, 4096, FAKE, 4096, 0, 1e-5, FAKE, 4096, 4096, None) == \
        abi.DS_A_LENGTH_MISMATCH
    assert L.ds_add_rmsnorm(FAKE, 4096, FAKE, 4000, FAKE, 4096, 0, 1e-5, FAKE, 4096, 4096, None) == \
        abi.DS_B_LENGTH_MISMATCH
    assert L.ds_silu_mul(FAKE, 3, FAKE, 4, FAKE, 4, None) == abi.DS_A_LENGTH_MISMATCH
    assert L.ds_rope(FAKE, 4096, FAKE, 1024, 5, 32, 8, 128, 1e4, 9, None) == abi.DS_BAD_DTYPE
    assert L.ds_rope(FAKE, 4095, FAKE, 1024, 5, 32, 8, 128, 1e4, 0, None) == abi.DS_A_LENGTH_MISMATCH
    assert L.ds_rope(FAKE, 4096, FAKE, 1000, 5, 32, 8, 128, 1e4, 0, None) == abi.DS_B_LENGTH_MISMATCH
    assert L.ds_rope(FAKE, 4096, FAKE, 1024, -1, 32, 8, 128, 1e4, 0, None) == abi.DS_CACHE_LENGTH_MISMATCH


def test_kv_append_refusals_mirror_the_contract(abi):
    L = abi.lib
    assert L.ds_kv_cache_append(FAKE, 0, 8, 6, FAKE, 3, 3, None) == abi.DS_CACHE_CAPACITY_EXCEEDED
    assert L.ds_kv_cache_append(FAKE, 0, 8, 0, FAKE, 0, 0, None) == abi.DS_EMPTY_DIMENSION
    assert L.ds_kv_cache_append(FAKE, 0, 8, 0, FAKE, 2, 3, None) == abi.DS_NEW_LENGTH_MISMATCH
    assert L.ds_kv_cache_append(FAKE, 0, 8, -1, FAKE, 3, 3, None) == abi.DS_CACHE_LENGTH_MISMATCH
    assert L.ds_kv_cache_append(FAKE, 5, 8, 0, FAKE, 3, 3, None) == abi.DS_BAD_DTYPE


def test_pick_refusals(abi):
    L = abi.lib
    assert L.ds_greedy_argmax(FAKE, 10, 1, 11, FAKE, None, FAKE, 1 << 20, None) == abi.DS_LOGITS_LENGTH_MISMATCH
    assert L.ds_greedy_argmax(FAKE, 0, 0, 11, FAKE, None, FAKE, 1 << 20, None) == abi.DS_EMPTY_DIMENSION
    n = 128256
    assert L.ds_sample(FAKE, n, 1, n, 0.8, 2000, float("nan"), FAKE, FAKE, FAKE, 1 << 20, None) == \
        abi.DS_BAD_SAMPLING_PARAM
    assert L.ds_sample(FAKE, n, 1, n, 0.8, 50, 0.0, FAKE, FAKE, FAKE, 1 << 20, None) == abi.DS_BAD_SAMPLING_PARAM
    assert L.ds_sample(FAKE, n, 1, n, 0.8, 50, 1.5, FAKE, FAKE, FAKE, 1 << 20, None) == abi.DS_BAD_SAMPLING_PARAM
    assert L.ds_sample(FAKE, n, 1, n, float("nan"), 50, 0.9, FAKE, FAKE, FAKE, 1 << 20, None) == \
        abi.DS_BAD_SAMPLING_PARAM
    assert L.ds_sample(FAKE, n - 1, 1, n, 0.8, 50, 0.9, FAKE, FAKE, FAKE, 1 << 20, None) == \
        abi.DS_LOGITS_LENGTH_MISMATCH


def test_attention_refusals(abi):
    L = abi.lib
    # 6 query heads cannot share 4 KV heads
    assert L.ds_gqa_decode_attn(FAKE, FAKE, FAKE, 1, 4096, None, 256, 16, FAKE, 1, 6, 4, 128, 0.1, FAKE, FAKE,
                                1 << 20, None) == abi.DS_BAD_ARGUMENT
    # contiguous slots larger than the cache
    assert L.ds_gqa_decode_attn(FAKE, FAKE, FAKE, 1, 4095, None, 256, 16, FAKE, 1, 32, 8, 128, 0.1, FAKE, FAKE,
                                1 << 20, None) == abi.DS_CACHE_CAPACITY_EXCEEDED
    assert L.ds_gqa_decode_attn(FAKE, FAKE, FAKE, 3, 4096, None, 256, 16, FAKE, 1, 32, 8, 128, 0.1, FAKE, FAKE,
                                1 << 20, None) == abi.DS_BAD_DTYPE


def test_model_config_validation(abi):
    from autoregressive_decode_step_gb300 import configs as C

    def mc(cfg, **kw):
        m = abi.ModelConfig()
        c = dict(cfg, **kw)
        for k in ("vocab", "d", "n_layer", "n_qh", "n_kvh", "head_dim", "ff", "rope_layout", "tied", "w_dtype",
                  "kv_dtype"):
            setattr(m, k, c[k])
        m.rope_base, m.eps, m.max_seqs, m.max_ctx = c["rope_base"], c["eps"], c.get("max_seqs", 1), 1280
        return m

    for cfg in (C.TOY, C.QWEN3_0_6B, C.LLAMA3_8B):
        assert abi.lib.ds_model_workspace_bytes(ctypes.byref(mc(cfg))) > 0
    assert abi.lib.ds_model_workspace_bytes(ctypes.byref(mc(C.LLAMA3_8B, n_qh=30))) == 0   # 30 % 8
    assert abi.lib.ds_model_workspace_bytes(ctypes.byref(mc(C.LLAMA3_8B, head_dim=96))) == 0  # band split
    # long-context RoPE scaling: accepted with Llama 3.1's parameters, refused
    # when the bands are empty or inverted or the factor speeds pairs up
    def scaled(factor, lo, hi, orig):
        m = mc(C.LLAMA3_8B)
        m.rope_factor, m.rope_low_freq_factor, m.rope_high_freq_factor, m.rope_orig_max_pos = factor, lo, hi, orig
        return abi.lib.ds_model_workspace_bytes(ctypes.byref(m))
    assert scaled(8.0, 1.0, 4.0, 8192.0) > 0
    assert scaled(8.0, 4.0, 1.0, 8192.0) == 0
    assert scaled(8.0, 1.0, 1.0, 8192.0) == 0
    assert scaled(0.5, 1.0, 4.0, 8192.0) == 0
    assert scaled(8.0, 1.0, 4.0, 0.0) == 0
    assert scaled(float("nan"), 1.0, 4.0, 8192.0) == 0
    out = ctypes.c_void_p()
    m = mc(C.TOY)
    assert abi.lib.ds_model_create(ctypes.byref(m), None, None, 0, ctypes.byref(out)) == abi.DS_BAD_ARGUMENT


def test_batched_projection_refusals(abi):
    L = abi.lib
    f = L.ds_gemm_transposed
    # rows 64, cols 128, n 4
    assert f(FAKE, 64 * 128, FAKE, 4 * 64, 0, 64, 128, FAKE, 0, FAKE, 1 << 24, None) == abi.DS_EMPTY_DIMENSION
    assert f(FAKE, 64 * 128, FAKE, 257 * 64, 257, 64, 128, FAKE, 257 * 128, FAKE, 1 << 24, None) == \
        abi.DS_DIMENSION_TOO_LARGE
    assert f(FAKE, 64 * 127, FAKE, 4 * 64, 4, 64, 128, FAKE, 4 * 128, FAKE, 1 << 24, None) == \
        abi.DS_GEMV_A_LENGTH_MISMATCH
    assert f(FAKE, 64 * 128, FAKE, 4 * 63, 4, 64, 128, FAKE, 4 * 128, FAKE, 1 << 24, None) == \
        abi.DS_GEMV_X_LENGTH_MISMATCH
    assert f(FAKE, 64 * 128, FAKE, 4 * 64, 4, 64, 128, FAKE, 4 * 127, FAKE, 1 << 24, None) == \
        abi.DS_A_LENGTH_MISMATCH
    # cols not a whole number of 16-byte units of bf16
    assert f(FAKE, 64 * 100, FAKE, 4 * 64, 4, 64, 100, FAKE, 4 * 100, FAKE, 1 << 24, None) == abi.DS_BAD_ARGUMENT
    g = L.ds_gemm
    assert g(FAKE, 1000 * 512, FAKE, 5 * 512, 5, 1000, 512, FAKE, 5 * 999, FAKE, 1 << 24, None) == \
        abi.DS_A_LENGTH_MISMATCH
    assert g(FAKE, 1000 * 512, FAKE, 5 * 1000, 5, 1000, 512, FAKE, 5 * 1000, FAKE, 1 << 24, None) == \
        abi.DS_GEMV_X_LENGTH_MISMATCH
    assert L.ds_gemm_workspace_bytes(0, 64, 64) == 0
    assert L.ds_gemm_workspace_bytes(257, 64, 64) == 0


def test_step_seq_refuses_before_any_launch(abi):
    """stepSeq's host checks, in order: no model, then an empty prompt and a
    token count that disagrees with the buffer's length."""
    L = abi.lib
    assert L.ds_step_seq(None, None, None, 4, 0, 0, 4, None, None, None) == abi.DS_BAD_ARGUMENT
    fake = ctypes.c_void_p(16)  # never dereferenced: the counts are refused first
    assert L.ds_step_seq(fake, None, None, 0, 0, 0, 0, None, None, None) == abi.DS_EMPTY_DIMENSION
    assert L.ds_step_seq(fake, None, fake, 3, 0, 0, 4, fake, None, None) == abi.DS_A_LENGTH_MISMATCH


def test_binding_structs_match_the_header_layout(abi, tmp_path):
    """Every struct the binding mirrors has the header's size and field
    offsets, as a C compiler lays them out (a drifted field would hand the
    library shifted values without any error)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"ds_model_config": abi.ModelConfig, "ds_model_weights": abi.ModelWeights,
               "ds_kv_cache": abi.KVCache, "ds_sampling": abi.Sampling}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "decode_step.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append('printf("%%s size %%zu\\n", "%s", sizeof(%s));' % (cname, cname))
        for f in py._fields_:
            lines.append('printf("%%s %%s %%zu\\n", "%s", "%s", offsetof(%s, %s));' % (cname, f[0], cname, f[0]))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    for line in filter(None, out):
        cname, field, value = line.split()
        py = structs[cname]
        want = ctypes.sizeof(py) if field == "size" else getattr(py, field).offset
        assert int(value) == want, (cname, field)
