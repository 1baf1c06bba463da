"""ctypes binding of ``libdecodestep.so`` (declared in ``include/decode_step.h``).

Argument marshalling only: every function here passes pointers and sizes to
the C ABI and raises :class:`DecodeStepError` on a non-OK status.  Importing
this module fails loudly when the library has not been built — there is no
fallback path.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdecodestep.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libdecodestep.so is not built (run `python -c 'import __graft_entry__ as g; g.build()'` "
                      "or `python -m autoregressive_decode_step_gb300.build`)")

lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
DS_OK = 560
DS_EMPTY_DIMENSION = 561
DS_A_LENGTH_MISMATCH = 562
DS_B_LENGTH_MISMATCH = 563
DS_DIMENSION_TOO_LARGE = 564
DS_CODE_OUT_OF_RANGE = 565
DS_CACHE_LENGTH_MISMATCH = 566
DS_NEW_LENGTH_MISMATCH = 567
DS_LOGITS_LENGTH_MISMATCH = 568
DS_GEMV_A_LENGTH_MISMATCH = 569
DS_GEMV_X_LENGTH_MISMATCH = 570
DS_CACHE_CAPACITY_EXCEEDED = 571
DS_BAD_DTYPE = 572
DS_CUDA_ERROR = 573
DS_WORKSPACE_TOO_SMALL = 574
DS_BAD_SAMPLING_PARAM = 575
DS_TOKEN_OUT_OF_RANGE = 576
DS_BAD_ARGUMENT = 577
DS_MAX_DIM = 1 << 24
DS_F32, DS_BF16 = 0, 1
DS_ROPE_HALF_SPLIT, DS_ROPE_INTERLEAVED = 0, 1
DS_ERR_TOKEN_RANGE, DS_ERR_POSITION, DS_ERR_WAIT_TIMEOUT, DS_ERR_SAMPLING = 1, 2, 4, 8
DS_STEP_ADVANCE = 1
DS_STEP_PHASE_TIMES = 2
DS_STEP_TRACE = 4
KIND_NAMES = ["embed", "qkv", "attention", "o_proj", "gate_up", "down", "head", "sample"]

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
SZ = ctypes.c_size_t
F32 = ctypes.c_float
F64 = ctypes.c_double


class ModelConfig(ctypes.Structure):
    _fields_ = [("vocab", I32), ("d", I32), ("n_layer", I32), ("n_qh", I32), ("n_kvh", I32),
                ("head_dim", I32), ("ff", I32), ("rope_layout", I32), ("rope_base", F64), ("eps", F32),
                ("tied", I32), ("w_dtype", I32), ("kv_dtype", I32), ("max_seqs", I32), ("max_ctx", I32),
                ("rope_factor", F64), ("rope_low_freq_factor", F64), ("rope_high_freq_factor", F64),
                ("rope_orig_max_pos", F64)]


class ModelWeights(ctypes.Structure):
    _fields_ = [("emb", P), ("out", P), ("final_norm", P), ("n1", P), ("wqkv", P), ("wo", P), ("n2", P),
                ("wgu", P), ("wd", P), ("q_norm", P), ("k_norm", P)]


class KVCache(ctypes.Structure):
    _fields_ = [("k", P), ("v", P), ("rows", I64), ("block_tokens", I32), ("max_blocks", I32),
                ("block_table", P)]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", F32), ("top_k", I32), ("top_p", F32)]


class SchedConfig(ctypes.Structure):
    _fields_ = [("n_blocks", I32), ("block_tokens", I32), ("max_blocks", I32), ("max_running", I32),
                ("chunk", I32), ("headroom_blocks", I32)]


class SchedRow(ctypes.Structure):
    _fields_ = [("request", I64), ("slot", I32), ("offset", I32), ("count", I32), ("decode", I32),
                ("yields", I32)]


def _sig(name, res, *args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("ds_status_name", ctypes.c_char_p, ctypes.c_int)
_sig("ds_residual_dims_check", ctypes.c_int, I64, I64, I64)
_sig("ds_workspace_error", ctypes.c_int, P, P, P)
_sig("ds_device_sm_count", ctypes.c_int)
_sig("ds_gemv_workspace_bytes", SZ, I64, I64, ctypes.c_int)
_sig("ds_gemv_transposed", ctypes.c_int, P, I64, ctypes.c_int, P, I64, I64, I64, P, I64, P, SZ, P)
_sig("ds_gemv", ctypes.c_int, P, I64, ctypes.c_int, P, I64, I64, I64, P, I64, P)
_sig("ds_gemm_workspace_bytes", SZ, I64, I64, I64)
_sig("ds_decode_steps", ctypes.c_int, P, P, P, P, ctypes.c_int, P, P, ctypes.c_uint, P)
_sig("ds_step_seq", ctypes.c_int, P, P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P)
_sig("ds_sched_create", ctypes.c_int, ctypes.POINTER(SchedConfig), P)
_sig("ds_sched_destroy", None, P)
_sig("ds_sched_submit", ctypes.c_int, P, I64, I32, I32)
_sig("ds_sched_plan", ctypes.c_int, P, P, I32, P, P, P, P)
_sig("ds_sched_commit", ctypes.c_int, P, P, I32)
_sig("ds_sched_stats", ctypes.c_int, P, P)
_sig("ds_sched_generated", I64, P, I64)
_sig("ds_gemm_transposed", ctypes.c_int, P, I64, P, I64, I64, I64, I64, P, I64, P, SZ, P)
_sig("ds_gemm", ctypes.c_int, P, I64, P, I64, I64, I64, I64, P, I64, P, SZ, P)
_sig("ds_gemv_transposed_noalloc", ctypes.c_int, P, I64, ctypes.c_int, P, I64, I64, I64, P, I64, P)
_sig("ds_gemv_transposed_noalloc_max_bytes", SZ)
_sig("ds_gemv_transposed_noalloc_error", ctypes.c_int, P, P)
_sig("ds_residual_add", ctypes.c_int, P, I64, P, I64, P, I64, P)
_sig("ds_add_rmsnorm", ctypes.c_int, P, I64, P, I64, P, I64, ctypes.c_int, F32, P, I64, I64, P)
_sig("ds_rope", ctypes.c_int, P, I64, P, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, F64, ctypes.c_int, P)
_sig("ds_kv_cache_append", ctypes.c_int, P, ctypes.c_int, I64, I64, P, I64, I64, P)
_sig("ds_silu_mul", ctypes.c_int, P, I64, P, I64, P, I64, P)
_sig("ds_attention_workspace_bytes", SZ, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, I64)
_sig("ds_gqa_decode_attn", ctypes.c_int, P, P, P, ctypes.c_int, I64, P, ctypes.c_int, ctypes.c_int, P,
     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, F32, P, P, SZ, P)
_sig("ds_argmax_workspace_bytes", SZ, ctypes.c_int, I64)
_sig("ds_greedy_argmax", ctypes.c_int, P, I64, ctypes.c_int, I64, P, P, P, SZ, P)
_sig("ds_sample_workspace_bytes", SZ, ctypes.c_int, I64)
_sig("ds_sample", ctypes.c_int, P, I64, ctypes.c_int, I64, F32, ctypes.c_int, F32, P, P, P, SZ, P)
_sig("ds_model_workspace_bytes", SZ, ctypes.POINTER(ModelConfig))
_sig("ds_model_create", ctypes.c_int, ctypes.POINTER(ModelConfig), ctypes.POINTER(ModelWeights), P, SZ,
     ctypes.POINTER(P))
_sig("ds_model_destroy", None, P)
_sig("ds_model_workspace", P, P)
_sig("ds_decode_step", ctypes.c_int, P, ctypes.POINTER(KVCache), P, P, ctypes.c_int, ctypes.POINTER(Sampling),
     P, P, P, ctypes.c_uint, P)
_sig("ds_step_graph_create", ctypes.c_int, P, ctypes.POINTER(KVCache), P, P, ctypes.c_int,
     ctypes.POINTER(Sampling), P, P, P, ctypes.c_uint, P, ctypes.POINTER(P))
_sig("ds_step_graph_launch", ctypes.c_int, P, P)
_sig("ds_step_graph_destroy", None, P)
_sig("ds_model_phase_times", ctypes.c_int, P, P, ctypes.c_int, ctypes.POINTER(ctypes.c_int), P)
_sig("ds_model_trace", ctypes.c_int, P, P, SZ, ctypes.POINTER(SZ), ctypes.POINTER(ctypes.c_int), P)
_sig("ds_decode_kernel_time", ctypes.c_int, P, ctypes.POINTER(KVCache), P, P, ctypes.c_int, ctypes.c_int,
     ctypes.POINTER(ctypes.c_float), P)
_sig("ds_decode_step_profile", ctypes.c_int, P, ctypes.POINTER(KVCache), P, P, ctypes.c_int,
     ctypes.POINTER(Sampling), P, P, P, ctypes.c_uint, ctypes.c_int, P, P, ctypes.c_int,
     ctypes.POINTER(ctypes.c_int), P)


class DecodeStepError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, status_name(code), code))


def status_name(code):
    return lib.ds_status_name(int(code)).decode()


def check(code, where="decode_step"):
    if code != DS_OK:
        raise DecodeStepError(code, where)
    return code


# ------------------------------------------------------------------ marshalling
def ptr(t):
    """Device (or host) address of a tensor, or NULL for None."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def dtype_code(t):
    if t.dtype == torch.float32:
        return DS_F32
    if t.dtype == torch.bfloat16:
        return DS_BF16
    raise TypeError("unsupported dtype %s" % t.dtype)


def stream_handle(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def workspace(nbytes_, device="cuda"):
    """A zero-filled, 256-byte-aligned workspace tensor."""
    return torch.zeros(max(int(nbytes_), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ ops
def ds_gemv_workspace_bytes(rows, cols, dtype=DS_F32):
    return lib.ds_gemv_workspace_bytes(rows, cols, dtype)


def ds_gemv_transposed(A, x, rows, cols, y, ws, stream=None):
    check(lib.ds_gemv_transposed(ptr(A), A.numel(), dtype_code(A), ptr(x), x.numel(), rows, cols, ptr(y),
                                 y.numel(), ptr(ws), nbytes(ws), stream_handle(stream)), "ds_gemv_transposed")


def ds_gemv_transposed_noalloc(A, x, rows, cols, y, stream=None):
    check(lib.ds_gemv_transposed_noalloc(ptr(A), A.numel(), dtype_code(A), ptr(x), x.numel(), rows, cols, ptr(y),
                                         y.numel(), stream_handle(stream)), "ds_gemv_transposed_noalloc")


def ds_gemv_transposed_noalloc_error(stream=None):
    """Read and clear the no-allocation area's error word (current device)."""
    word = ctypes.c_int32(0)
    check(lib.ds_gemv_transposed_noalloc_error(ctypes.byref(word), stream_handle(stream)),
          "ds_gemv_transposed_noalloc_error")
    return word.value


def ds_gemv(W, x, rows, cols, y, stream=None):
    check(lib.ds_gemv(ptr(W), W.numel(), dtype_code(W), ptr(x), x.numel(), rows, cols, ptr(y), y.numel(),
                      stream_handle(stream)), "ds_gemv")


def ds_gemm_transposed(A, X, n, rows, cols, Y, ws, stream=None):
    check(lib.ds_gemm_transposed(ptr(A), A.numel(), ptr(X), X.numel(), n, rows, cols, ptr(Y), Y.numel(), ptr(ws),
                                 nbytes(ws), stream_handle(stream)), "ds_gemm_transposed")


def ds_gemm(W, X, n, rows, cols, Y, ws, stream=None):
    check(lib.ds_gemm(ptr(W), W.numel(), ptr(X), X.numel(), n, rows, cols, ptr(Y), Y.numel(), ptr(ws), nbytes(ws),
                      stream_handle(stream)), "ds_gemm")


def ds_residual_add(a, b, out, n, stream=None):
    check(lib.ds_residual_add(ptr(a), a.numel(), ptr(b), b.numel(), ptr(out), n, stream_handle(stream)),
          "ds_residual_add")


def ds_add_rmsnorm(residual, x, w, eps, h, n, stream=None):
    check(lib.ds_add_rmsnorm(ptr(residual), residual.numel(), ptr(x), 0 if x is None else x.numel(), ptr(w),
                             w.numel(), dtype_code(w), eps, ptr(h), h.numel(), n, stream_handle(stream)),
          "ds_add_rmsnorm")


def ds_rope(q, k, pos, n_qh, n_kh, head_dim, base, layout, stream=None):
    check(lib.ds_rope(ptr(q), q.numel(), ptr(k), 0 if k is None else k.numel(), pos, n_qh, n_kh, head_dim,
                      base, layout, stream_handle(stream)), "ds_rope")


def ds_kv_cache_append(cache, capacity, cache_len, new_vals, n_new, stream=None):
    check(lib.ds_kv_cache_append(ptr(cache), dtype_code(cache), capacity, cache_len, ptr(new_vals),
                                 new_vals.numel(), n_new, stream_handle(stream)), "ds_kv_cache_append")


def ds_silu_mul(gate, up, out, n, stream=None):
    check(lib.ds_silu_mul(ptr(gate), gate.numel(), ptr(up), up.numel(), ptr(out), n, stream_handle(stream)),
          "ds_silu_mul")


def ds_attention_workspace_bytes(n_seqs, n_qh, n_kvh, head_dim, max_ctx):
    return lib.ds_attention_workspace_bytes(n_seqs, n_qh, n_kvh, head_dim, max_ctx)


def ds_gqa_decode_attn(q, k_cache, v_cache, cache_rows, block_table, max_blocks_per_seq, block_tokens, seq_lens,
                       n_seqs, n_qh, n_kvh, head_dim, scale, out, ws, stream=None):
    check(lib.ds_gqa_decode_attn(ptr(q), ptr(k_cache), ptr(v_cache), dtype_code(k_cache), cache_rows,
                                 ptr(block_table), max_blocks_per_seq, block_tokens, ptr(seq_lens), n_seqs, n_qh,
                                 n_kvh, head_dim, scale, ptr(out), ptr(ws), nbytes(ws), stream_handle(stream)),
          "ds_gqa_decode_attn")


def ds_argmax_workspace_bytes(n_rows, n):
    return lib.ds_argmax_workspace_bytes(n_rows, n)


def ds_greedy_argmax(logits, n_rows, n, ids, max_logit, ws, stream=None):
    check(lib.ds_greedy_argmax(ptr(logits), logits.numel(), n_rows, n, ptr(ids), ptr(max_logit), ptr(ws),
                               nbytes(ws), stream_handle(stream)), "ds_greedy_argmax")


def ds_sample_workspace_bytes(n_rows, n):
    return lib.ds_sample_workspace_bytes(n_rows, n)


def ds_sample(logits, n_rows, n, temperature, top_k, top_p, u, ids, ws, stream=None):
    check(lib.ds_sample(ptr(logits), logits.numel(), n_rows, n, temperature, top_k, top_p, ptr(u), ptr(ids),
                        ptr(ws), nbytes(ws), stream_handle(stream)), "ds_sample")


def ds_workspace_error(ws, stream=None):
    word = ctypes.c_int32(0)
    check(lib.ds_workspace_error(ptr(ws), ctypes.byref(word), stream_handle(stream)), "ds_workspace_error")
    return word.value
