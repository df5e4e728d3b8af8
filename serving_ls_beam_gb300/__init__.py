"""Python binding of the ls_beam CUDA library (``libls_beam.so``).

Argument marshalling only: every function passes device pointers, sizes and the
stream handle to the C entry point of the same name (declared in
``include/ls_beam.h``) and returns its status code.  All computation happens in
the library's sm_103a kernels; there is no Python or CPU fallback, and a missing
library raises ``LsBeamError``.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "LS_OK", "LS_ERR_INVALID_ARG", "LS_ERR_UNSUPPORTED", "LS_ERR_CUDA", "LS_ERR_TIMEOUT", "LS_ERR_INTERNAL",
    "LS_DTYPE_F32", "LS_DTYPE_F16", "LS_DTYPE_BF16", "LS_MAX_K", "LsBeamError", "library_path", "load_library",
    "check", "ls_beam_step_workspace_size", "ls_workspace_init", "ls_beam_step", "ls_cache_reorder",
    "ls_read_status", "ls_status_string", "ls_read_row_stats", "ls_beam_step_noalloc", "ls_beam_step_noalloc_status",
    "ls_backtrack",
    "ls_sample_workspace_size", "ls_sample", "ls_cache_refresh_inplace", "ls_logits_beam_step",
    "ls_beam_step_refresh_inplace",
]

LS_OK, LS_ERR_INVALID_ARG, LS_ERR_UNSUPPORTED, LS_ERR_CUDA, LS_ERR_TIMEOUT, LS_ERR_INTERNAL = range(6)
LS_DTYPE_F32, LS_DTYPE_F16, LS_DTYPE_BF16 = 0, 1, 2
LS_MAX_K = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class LsBeamError(RuntimeError):
    pass


def library_path() -> str:
    return os.path.join(_HERE, "libls_beam.so")


def load_library():
    """Load libls_beam.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise LsBeamError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        vp, ip, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.ls_beam_step_workspace_size.argtypes = [ip, ip, ip]
        lib.ls_beam_step_workspace_size.restype = sz
        lib.ls_workspace_init.argtypes = [vp, sz, vp]
        lib.ls_workspace_init.restype = ip
        lib.ls_beam_step.argtypes = [vp, ip, vp, vp, vp, ip, ip, ip, ip, vp, vp, vp, vp, vp, sz, vp]
        lib.ls_beam_step.restype = ip
        lib.ls_cache_reorder.argtypes = [vp, vp, ip, vp, ip, ip, ip, ip, ip, ip, ip, vp, vp]
        lib.ls_cache_reorder.restype = ip
        lib.ls_read_status.argtypes = [vp, vp]
        lib.ls_read_status.restype = ip
        lib.ls_status_string.argtypes = [ip]
        lib.ls_status_string.restype = ctypes.c_char_p
        lib.ls_read_row_stats.argtypes = [vp, ip, ip, ip, vp, vp, vp, vp, vp]
        lib.ls_read_row_stats.restype = ip
        lib.ls_beam_step_noalloc.argtypes = [vp, ip, vp, vp, vp, ip, ip, ip, ip, vp, vp, vp, vp, vp]
        lib.ls_beam_step_noalloc.restype = ip
        lib.ls_beam_step_noalloc_status.argtypes = [vp]
        lib.ls_beam_step_noalloc_status.restype = ip
        lib.ls_backtrack.argtypes = [vp, vp, ip, ip, ip, ip, vp, vp, vp, vp]
        lib.ls_backtrack.restype = ip
        lib.ls_sample_workspace_size.argtypes = [ip, ip, ip]
        lib.ls_sample_workspace_size.restype = sz
        lib.ls_sample.argtypes = [vp, ip, vp, vp, ip, ip, ip, ctypes.c_float, vp, vp, vp, sz, vp]
        lib.ls_sample.restype = ip
        lib.ls_cache_refresh_inplace.argtypes = [vp, ip, vp, ip, ip, ip, ip, ip, ip, ip, vp, vp]
        lib.ls_cache_refresh_inplace.restype = ip
        lib.ls_logits_beam_step.argtypes = [vp, vp, ip, ip, vp, vp, vp, ip, ip, ip, ip, vp, vp, vp, vp, vp, sz, vp]
        lib.ls_logits_beam_step.restype = ip
        lib.ls_beam_step_refresh_inplace.argtypes = [vp, ip, vp, vp, vp, ip, ip, ip, ip, vp, vp, vp, vp, vp, ip, ip,
                                                     ip, ip, ip, ip, vp, sz, vp]
        lib.ls_beam_step_refresh_inplace.restype = ip
        _lib = lib
        return lib


def _dtype_code(t) -> int:
    import torch

    codes = {torch.float32: LS_DTYPE_F32, torch.float16: LS_DTYPE_F16, torch.bfloat16: LS_DTYPE_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int, what: str = "ls_beam") -> None:
    if status != LS_OK:
        raise LsBeamError(f"{what}: {ls_status_string(status)} ({status})")


def ls_status_string(status: int) -> str:
    return load_library().ls_status_string(int(status)).decode()


def ls_beam_step_workspace_size(batch: int, k: int, vocab: int) -> int:
    return int(load_library().ls_beam_step_workspace_size(batch, k, vocab))


def ls_workspace_init(workspace, stream=None) -> int:
    return load_library().ls_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream(stream))


def ls_beam_step(logits, bias, beam_scores, finished, eos_id: int, out_token, out_parent, out_score,
                 out_finished, workspace, stream=None) -> int:
    """logits [batch, k, vocab] (f32/f16/bf16), bias [vocab] f32 or None, beam_scores [batch, k] f32,
    finished [batch, k] uint8 or None, outputs [batch, k] (int32, int32, f32, uint8 or None),
    workspace a uint8 device tensor of ls_beam_step_workspace_size() bytes."""
    batch, k, vocab = logits.shape
    return load_library().ls_beam_step(
        _ptr(logits), _dtype_code(logits), _ptr(bias), _ptr(beam_scores), _ptr(finished), batch, k, vocab,
        int(eos_id), _ptr(out_token), _ptr(out_parent), _ptr(out_score), _ptr(out_finished), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))


def ls_beam_step_refresh_inplace(logits, bias, beam_scores, finished, eos_id: int, out_token, out_parent, out_score,
                                 out_finished, cache, length: int, workspace, stream=None) -> int:
    """ls_beam_step, then the in-place refresh of cache [layers, batch*k, heads, max_len, head_dim] by
    out_parent over positions [0, length); one kernel where the step runs a batch per CTA."""
    batch, k, vocab = logits.shape
    layers, rows, heads, max_len, head_dim = cache.shape
    if rows != batch * k:
        raise ValueError("cache rows do not match batch * k")
    return load_library().ls_beam_step_refresh_inplace(
        _ptr(logits), _dtype_code(logits), _ptr(bias), _ptr(beam_scores), _ptr(finished), batch, k, vocab,
        int(eos_id), _ptr(out_token), _ptr(out_parent), _ptr(out_score), _ptr(out_finished), _ptr(cache),
        _dtype_code(cache), layers, heads, max_len, int(length), head_dim, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))


def ls_logits_beam_step(hidden, weight, bias, beam_scores, finished, eos_id: int, out_token, out_parent, out_score,
                        out_finished, workspace, stream=None) -> int:
    """The beam step fused into the output projection: hidden [batch, k, dim] and weight [vocab, dim]
    (both f16 or both bf16, logits = hidden . weight^T, never stored); everything else as ls_beam_step.
    The workspace is the one of ls_beam_step_workspace_size(batch, k, vocab)."""
    batch, k, dim = hidden.shape
    vocab, dim_w = weight.shape
    if dim_w != dim or weight.dtype != hidden.dtype:
        raise ValueError("weight must be [vocab, dim] of the hidden states' dtype")
    return load_library().ls_logits_beam_step(
        _ptr(hidden), _ptr(weight), _dtype_code(hidden), dim, _ptr(bias), _ptr(beam_scores), _ptr(finished), batch, k,
        vocab, int(eos_id), _ptr(out_token), _ptr(out_parent), _ptr(out_score), _ptr(out_finished), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))


def ls_beam_step_noalloc(logits, bias, beam_scores, finished, eos_id: int, out_token, out_parent, out_score,
                         out_finished, stream=None) -> int:
    """ls_beam_step for callers that cannot allocate: no workspace argument, the library's
    fixed device scratch is used instead (shapes needing more than 64 MiB are rejected)."""
    batch, k, vocab = logits.shape
    return load_library().ls_beam_step_noalloc(
        _ptr(logits), _dtype_code(logits), _ptr(bias), _ptr(beam_scores), _ptr(finished), batch, k, vocab,
        int(eos_id), _ptr(out_token), _ptr(out_parent), _ptr(out_score), _ptr(out_finished), _stream(stream))


def ls_beam_step_noalloc_status(stream=None) -> int:
    """Device-detected status of the last ls_beam_step_noalloc on the current device (read and
    cleared; synchronises the stream)."""
    return load_library().ls_beam_step_noalloc_status(_stream(stream))


def ls_cache_reorder(src, dst, parent, length: int, workspace=None, stream=None) -> int:
    """src, dst [layers, batch*k, heads, max_len, head_dim]; parent [batch, k] int32."""
    layers, rows, heads, max_len, head_dim = src.shape
    batch, k = parent.shape
    if batch * k != rows:
        raise ValueError("parent shape does not match cache rows")
    return load_library().ls_cache_reorder(
        _ptr(src), _ptr(dst), _dtype_code(src), _ptr(parent), layers, batch, k, heads, max_len, int(length),
        head_dim, _ptr(workspace), _stream(stream))


def ls_backtrack(token_hist, parent_hist, eos_id: int, out_seq, out_len, workspace=None, stream=None) -> int:
    """token_hist, parent_hist [steps, batch, k] int32; out_seq [batch, k, steps] int32; out_len [batch, k] int32."""
    steps, batch, k = token_hist.shape
    return load_library().ls_backtrack(_ptr(token_hist), _ptr(parent_hist), steps, batch, k, int(eos_id),
                                       _ptr(out_seq), _ptr(out_len), _ptr(workspace), _stream(stream))


def ls_sample_workspace_size(rows: int, top_k: int, vocab: int) -> int:
    return int(load_library().ls_sample_workspace_size(rows, top_k, vocab))


def ls_sample(logits, bias, u, top_k: int, top_p: float, out_token, out_logprob, workspace, stream=None) -> int:
    """logits [rows, vocab] (f32/f16/bf16), bias [vocab] f32 or None, u [rows] f32, out_token [rows] int32,
    out_logprob [rows] f32 or None, workspace a uint8 device tensor of ls_sample_workspace_size() bytes."""
    rows, vocab = logits.shape
    return load_library().ls_sample(_ptr(logits), _dtype_code(logits), _ptr(bias), _ptr(u), rows, vocab, int(top_k),
                                    float(top_p), _ptr(out_token), _ptr(out_logprob), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))


def ls_cache_refresh_inplace(cache, parent, length: int, workspace=None, stream=None) -> int:
    """cache [layers, batch*k, heads, max_len, head_dim] (refreshed in place); parent [batch, k] int32."""
    layers, rows, heads, max_len, head_dim = cache.shape
    batch, k = parent.shape
    if batch * k != rows:
        raise ValueError("parent shape does not match cache rows")
    return load_library().ls_cache_refresh_inplace(
        _ptr(cache), _dtype_code(cache), _ptr(parent), layers, batch, k, heads, max_len, int(length), head_dim,
        _ptr(workspace), _stream(stream))


def ls_read_status(workspace, stream=None) -> int:
    return load_library().ls_read_status(_ptr(workspace), _stream(stream))


def ls_read_row_stats(workspace, batch: int, k: int, vocab: int, stream=None):
    """Host numpy arrays (lse, rtopk, ncand, path) of the last step run on `workspace`."""
    import numpy as np

    lse = np.empty(batch * k, np.float32)
    rt = np.empty(batch * k, np.float32)
    nc = np.empty(batch * k, np.int32)
    path = np.empty(batch, np.int32)
    st = load_library().ls_read_row_stats(_ptr(workspace), batch, k, vocab, lse.ctypes.data, rt.ctypes.data,
                                          nc.ctypes.data, path.ctypes.data, _stream(stream))
    check(st, "ls_read_row_stats")
    return lse.reshape(batch, k), rt.reshape(batch, k), nc.reshape(batch, k), path
