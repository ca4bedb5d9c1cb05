"""ctypes binding of libspecverify.so: the C ABI's calls under the same
names, with argument marshalling only.

Tensor arguments may be torch tensors (their ``data_ptr()`` is passed), plain
integer addresses, or None for the ABI's optional pointers.  ``stream`` may be
a ``torch.cuda.Stream``, an integer handle, or None for torch's current
stream.  A non-OK status raises ``SVError`` with the library's message.
Every computation happens in the library's kernels; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

# sv_status
SV_OK = 0
SV_ERR_ARG = 1
SV_ERR_SHAPE = 2
SV_ERR_DTYPE = 3
SV_ERR_CUDA = 4
SV_ERR_WORKSPACE = 5
SV_ERR_DEVICE_FLAG = 6
SV_ERR_TIMEOUT = 7
SV_ERR_UNSUPPORTED = 8
# sv_dtype
SV_F32 = 0
SV_BF16 = 1
# modes
SV_SAMPLED = 0
SV_GREEDY = 1
# flag bits
SV_FLAG_BAD_K = 1
SV_FLAG_BAD_TOKEN = 2
SV_FLAG_NONFINITE = 4
SV_FLAG_BAD_TEMPERATURE = 8
SV_FLAG_BAD_UNIFORM = 16
SV_FLAG_BAD_MODE = 32
SV_FLAG_CAPACITY = 64
SV_FLAG_TIMEOUT = 128
SV_FLAG_BAD_N = 256
# diag fields
SV_DIAG_M_T = 0
SV_DIAG_S_T = 1
SV_DIAG_MASS_T = 2
SV_DIAG_P_X = 3
SV_DIAG_M_D = 4
SV_DIAG_S_D = 5
SV_DIAG_MASS_D = 6
SV_DIAG_Q_X = 7
SV_DIAG_RATIO = 8
SV_DIAG_ARGMAX = 9
SV_DIAG_S_W = 10
SV_DIAG_FIELDS = 16


class SVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"specverify status {status}: {message}")
        self.status = status


_lib = None
_c = ctypes
_vp, _i32, _i64, _f32, _sz = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_float, _c.c_size_t


def lib() -> ctypes.CDLL:
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "speculative_decoding_verification_47_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.sv_version.restype = _i32
        L.sv_version.argtypes = []
        L.sv_workspace_size.restype = _sz
        L.sv_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
        L.sv_lmhead_workspace_size.restype = _sz
        L.sv_lmhead_workspace_size.argtypes = [_i32, _i32]
        L.sv_spec_verify.restype = _i32
        L.sv_spec_verify.argtypes = [_vp, _i64, _i64, _vp, _i64, _i64, _i32, _i32, _i32, _i32,
                                     _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.sv_spec_verify_target_topp.restype = _i32
        L.sv_spec_verify_target_topp.argtypes = L.sv_spec_verify.argtypes
        L.sv_spec_verify_noalloc.restype = _i32
        L.sv_spec_verify_noalloc.argtypes = [_vp, _i64, _i64, _vp, _i64, _i64, _i32, _i32, _i32,
                                             _i32, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp,
                                             _vp]
        L.sv_kv_commit.restype = _i32
        L.sv_kv_commit.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _vp, _sz, _vp]
        L.sv_lmhead_rmsnorm.restype = _i32
        L.sv_lmhead_rmsnorm.argtypes = [_vp, _vp, _f32, _vp, _vp, _i32, _i32, _i32, _i32, _vp,
                                        _sz, _vp]
        L.sv_draft_sample_workspace_size.restype = _sz
        L.sv_draft_sample_workspace_size.argtypes = []
        L.sv_draft_sample.restype = _i32
        L.sv_draft_sample.argtypes = [_vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp, _vp, _f32, _vp,
                                      _vp, _vp, _vp, _sz, _vp]
        L.sv_kv_commit_paged.restype = _i32
        L.sv_kv_commit_paged.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp,
                                         _sz, _vp]
        L.sv_dynk_state_size.restype = _sz
        L.sv_dynk_state_size.argtypes = [_i32]
        L.sv_dynk_init.restype = _i32
        L.sv_dynk_init.argtypes = [_vp, _i32, _i32, _vp]
        L.sv_dynk_update.restype = _i32
        L.sv_dynk_update.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.sv_read_device_flags.restype = _i32
        L.sv_read_device_flags.argtypes = [_vp, _c.POINTER(_c.c_uint32), _vp]
        L.sv_last_error.restype = _c.c_char_p
        L.sv_last_error.argtypes = []
        _lib = L
    return _lib


def _ptr(x):
    """Device address of a tensor argument.  Every pointer of the ABI is a
    device pointer, so a tensor elsewhere (a CPU or pinned host tensor) is
    refused here rather than handed to a kernel as an address it cannot read."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    dev = getattr(x, "device", None)
    if dev is not None and dev.type != "cuda":
        raise ValueError(f"expected a CUDA tensor, got a tensor on {dev}")
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != SV_OK:
        msg = lib().sv_last_error().decode(errors="replace")
        raise SVError(status, msg)


def sv_version() -> int:
    return lib().sv_version()


def sv_workspace_size(B: int, K: int, V: int, dtype: int) -> int:
    return lib().sv_workspace_size(B, K, V, dtype)


def sv_lmhead_workspace_size(M: int, H: int) -> int:
    return lib().sv_lmhead_workspace_size(M, H)


def sv_spec_verify(target_logits, target_seq_stride, target_pos_stride, draft_logits,
                   draft_seq_stride, draft_pos_stride, dtype, B, K, V, draft_tokens, k_per_row,
                   temperature, top_p, uniforms, mode, out_tokens, n_accepted, diag, workspace,
                   workspace_bytes, stream=None):
    _check(lib().sv_spec_verify(
        _ptr(target_logits), target_seq_stride, target_pos_stride, _ptr(draft_logits),
        draft_seq_stride, draft_pos_stride, dtype, B, K, V, _ptr(draft_tokens), _ptr(k_per_row),
        _ptr(temperature), float(top_p), _ptr(uniforms), _ptr(mode), _ptr(out_tokens),
        _ptr(n_accepted), _ptr(diag), _ptr(workspace), workspace_bytes, _stream(stream)))


def sv_spec_verify_target_topp(target_logits, target_seq_stride, target_pos_stride, draft_logits,
                               draft_seq_stride, draft_pos_stride, dtype, B, K, V, draft_tokens,
                               k_per_row, temperature, top_p, uniforms, mode, out_tokens, n_accepted,
                               diag, workspace, workspace_bytes, stream=None):
    """sv_spec_verify with top-p on the target rows only (the draft untruncated)."""
    _check(lib().sv_spec_verify_target_topp(
        _ptr(target_logits), target_seq_stride, target_pos_stride, _ptr(draft_logits),
        draft_seq_stride, draft_pos_stride, dtype, B, K, V, _ptr(draft_tokens), _ptr(k_per_row),
        _ptr(temperature), float(top_p), _ptr(uniforms), _ptr(mode), _ptr(out_tokens),
        _ptr(n_accepted), _ptr(diag), _ptr(workspace), workspace_bytes, _stream(stream)))


def sv_spec_verify_noalloc(target_logits, target_seq_stride, target_pos_stride, draft_logits,
                           draft_seq_stride, draft_pos_stride, dtype, B, K, V, draft_tokens,
                           k_per_row, temperature, top_p, uniforms, mode, out_tokens, n_accepted,
                           diag, stream=None):
    """sv_spec_verify with the library's built-in scratch: no workspace."""
    _check(lib().sv_spec_verify_noalloc(
        _ptr(target_logits), target_seq_stride, target_pos_stride, _ptr(draft_logits),
        draft_seq_stride, draft_pos_stride, dtype, B, K, V, _ptr(draft_tokens), _ptr(k_per_row),
        _ptr(temperature), float(top_p), _ptr(uniforms), _ptr(mode), _ptr(out_tokens),
        _ptr(n_accepted), _ptr(diag), _stream(stream)))


def sv_kv_commit(seq_lens, n_accepted, capacity, k_per_row, B, K, workspace, workspace_bytes,
                 stream=None):
    _check(lib().sv_kv_commit(_ptr(seq_lens), _ptr(n_accepted), _ptr(capacity), _ptr(k_per_row), B, K,
                              _ptr(workspace), workspace_bytes, _stream(stream)))


def sv_lmhead_rmsnorm(hidden, norm_w, eps, W, logits, out_dtype, M, H, V, workspace,
                      workspace_bytes, stream=None):
    _check(lib().sv_lmhead_rmsnorm(_ptr(hidden), _ptr(norm_w), float(eps), _ptr(W), _ptr(logits),
                                   out_dtype, M, H, V, _ptr(workspace), workspace_bytes,
                                   _stream(stream)))


def sv_draft_sample_workspace_size() -> int:
    return lib().sv_draft_sample_workspace_size()


def sv_draft_sample(draft_logits, seq_stride, pos_stride, dtype, B, K, V, k_per_row, temperature,
                    top_p, uniforms, mode, out_tokens, workspace, workspace_bytes, stream=None):
    _check(lib().sv_draft_sample(
        _ptr(draft_logits), seq_stride, pos_stride, dtype, B, K, V, _ptr(k_per_row),
        _ptr(temperature), float(top_p), _ptr(uniforms), _ptr(mode), _ptr(out_tokens),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def sv_kv_commit_paged(seq_lens, n_accepted, k_per_row, block_table, max_pages, page_size,
                       free_pages, free_top, free_capacity, B, workspace, workspace_bytes,
                       stream=None):
    _check(lib().sv_kv_commit_paged(_ptr(seq_lens), _ptr(n_accepted), _ptr(k_per_row),
                                    _ptr(block_table), max_pages, page_size, _ptr(free_pages),
                                    _ptr(free_top), free_capacity, B, _ptr(workspace),
                                    workspace_bytes, _stream(stream)))


def sv_dynk_state_size(B: int) -> int:
    return lib().sv_dynk_state_size(B)


def sv_dynk_init(state, B, k0, stream=None):
    _check(lib().sv_dynk_init(_ptr(state), B, k0, _stream(stream)))


def sv_dynk_update(state, B, n_accepted, k_used, cap, k_next, workspace, workspace_bytes,
                   stream=None):
    _check(lib().sv_dynk_update(_ptr(state), B, _ptr(n_accepted), _ptr(k_used), _ptr(cap),
                                _ptr(k_next), _ptr(workspace), workspace_bytes, _stream(stream)))


def sv_read_device_flags(workspace, stream=None) -> int:
    """Synchronise the stream and return the device flag word (no raise on
    non-zero flags; the status is only raised for CUDA failures)."""
    v = _c.c_uint32(0)
    st = lib().sv_read_device_flags(_ptr(workspace), _c.byref(v), _stream(stream))
    if st not in (SV_OK, SV_ERR_DEVICE_FLAG, SV_ERR_TIMEOUT):
        _check(st)
    return int(v.value)


def sv_last_error() -> str:
    return lib().sv_last_error().decode(errors="replace")
