"""Oracle for the hierarchical beam-search step: TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product path (the CUDA library and
its binding in ``serving_ls_beam_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``ls_beam_oracle.c`` (plain single-threaded C, fp64),
which restates the naive decoding definition from the LightSeq inference
article (31duo.com, itemid-283120, section on the hierarchical rewrite of
decoding).  This module only compiles it with gcc and marshals numpy arrays.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, invariants, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ls_beam_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, so x86 and Arm agree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, ip = ctypes.c_void_p, ctypes.c_int
            lib.oracle_beam_step.argtypes = [vp, ip, vp, vp, vp, ip, ip, ip, ip, ip, vp, vp, vp, vp, vp]
            lib.oracle_beam_step.restype = ip
            lib.oracle_rtopk_stats.argtypes = [vp, ip, vp, ip, ip, ip, ip, vp, vp, vp]
            lib.oracle_rtopk_stats.restype = ip
            lib.oracle_cache_reorder.argtypes = [vp, vp, ip, vp, ip, ip, ip, ip, ip, ip, ip]
            lib.oracle_cache_reorder.restype = ip
            lib.oracle_backtrack.argtypes = [vp, vp, ip, ip, ip, ip, vp, vp]
            lib.oracle_backtrack.restype = ip
            lib.oracle_sample.argtypes = [vp, ip, vp, ip, ip, ip, ctypes.c_double, vp, vp, vp, vp]
            lib.oracle_sample.restype = ip
            lib.oracle_cache_refresh_inplace.argtypes = [vp, ip, vp, ip, ip, ip, ip, ip, ip, ip]
            lib.oracle_cache_refresh_inplace.restype = ip
            lib.oracle_logits.argtypes = [vp, vp, ip, ip, ip, ip, vp]
            lib.oracle_logits.restype = ip
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _logit_code(logits: np.ndarray, dtype: str | None) -> tuple[np.ndarray, int]:
    if logits.dtype == np.float64:
        return np.ascontiguousarray(logits), DTYPE_CODES["f64"]
    if logits.dtype == np.float32:
        return np.ascontiguousarray(logits), DTYPE_CODES["f32"]
    if logits.dtype == np.float16:
        return np.ascontiguousarray(logits).view(np.uint16), DTYPE_CODES["f16"]
    if logits.dtype == np.uint16 and dtype in ("f16", "bf16"):
        return np.ascontiguousarray(logits), DTYPE_CODES[dtype]
    raise TypeError(f"unsupported logits dtype {logits.dtype} / {dtype}")


def beam_step(logits, beam_scores, *, bias=None, finished=None, eos_id=0, m_out=None, dtype=None):
    """Naive beam step.  Returns dict of per-batch sorted lists of length m_out (default k):
    token, parent (int32), score (float64), finished (uint8), and lse [batch, k] (float64)."""
    lib = _load()
    lg, code = _logit_code(np.asarray(logits), dtype)
    batch, k, vocab = lg.shape
    m_out = k if m_out is None else int(m_out)
    bs = np.ascontiguousarray(beam_scores, dtype=np.float32).reshape(batch, k)
    bi = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(vocab)
    fin = None if finished is None else np.ascontiguousarray(finished, dtype=np.uint8).reshape(batch, k)
    tok = np.empty((batch, m_out), np.int32)
    par = np.empty((batch, m_out), np.int32)
    sc = np.empty((batch, m_out), np.float64)
    of = np.empty((batch, m_out), np.uint8)
    lse = np.empty((batch, k), np.float64)
    rc = lib.oracle_beam_step(_ptr(lg), code, _ptr(bi), _ptr(bs), _ptr(fin), batch, k, vocab, int(eos_id),
                              m_out, _ptr(tok), _ptr(par), _ptr(sc), _ptr(of), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_beam_step failed ({rc})")
    return {"token": tok, "parent": par, "score": sc, "finished": of, "lse": lse}


def rtopk_stats(logits, k, *, groups=None, bias=None, dtype=None):
    """Per-row first-traversal diagnostics: R (k-th largest of group maxima), true k-th largest, count x >= R."""
    lib = _load()
    lg, code = _logit_code(np.asarray(logits), dtype)
    vocab = lg.shape[-1]
    rows = lg.size // vocab
    groups = k if groups is None else int(groups)
    bi = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(vocab)
    R = np.empty(rows, np.float64)
    kth = np.empty(rows, np.float64)
    nc = np.empty(rows, np.int64)
    rc = lib.oracle_rtopk_stats(_ptr(lg), code, _ptr(bi), rows, int(k), vocab, groups, _ptr(R), _ptr(kth), _ptr(nc))
    if rc != 0:
        raise ValueError(f"oracle_rtopk_stats failed ({rc})")
    return {"R": R, "kth": kth, "ncand": nc}


def cache_reorder(src, parent, length, dst=None):
    """Gather of the [layers, batch*k, heads, max_len, head_dim] cache by parent beam (positions < length)."""
    lib = _load()
    src = np.ascontiguousarray(src)
    layers, rows, heads, max_len, head_dim = src.shape
    par = np.ascontiguousarray(parent, dtype=np.int32)
    batch, k = par.shape
    if batch * k != rows:
        raise ValueError("parent shape does not match cache rows")
    out = np.zeros_like(src) if dst is None else dst
    rc = lib.oracle_cache_reorder(_ptr(src), _ptr(out), src.dtype.itemsize, _ptr(par), layers, batch, k, heads,
                                  max_len, int(length), head_dim)
    if rc != 0:
        raise ValueError(f"oracle_cache_reorder failed ({rc})")
    return out


def backtrack(token_hist, parent_hist, eos_id):
    """Token sequences [batch, k, steps] and lengths [batch, k] of the final beams, read back through
    the parent pointers of the per-step history [steps, batch, k]."""
    lib = _load()
    tok = np.ascontiguousarray(token_hist, dtype=np.int32)
    par = np.ascontiguousarray(parent_hist, dtype=np.int32)
    steps, batch, k = tok.shape
    seq = np.empty((batch, k, steps), np.int32)
    ln = np.empty((batch, k), np.int32)
    rc = lib.oracle_backtrack(_ptr(tok), _ptr(par), steps, batch, k, int(eos_id), _ptr(seq), _ptr(ln))
    if rc != 0:
        raise ValueError(f"oracle_backtrack failed ({rc})")
    return seq, ln


def sample(logits, u, top_k, top_p=1.0, *, bias=None, dtype=None):
    """Sampling decoding of rows of logits [..., vocab]: top_k / top_p restriction, inverse CDF at u.
    Returns token (int32), logprob (float64, under the full softmax) and margin (distance of u from
    the nearest cumulative boundary of the kept candidates, or of top_p from one of the top_k's)."""
    lib = _load()
    lg, code = _logit_code(np.asarray(logits), dtype)
    vocab = lg.shape[-1]
    rows = lg.size // vocab
    bi = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(vocab)
    uu = np.ascontiguousarray(u, dtype=np.float64).reshape(rows)
    tok = np.empty(rows, np.int32)
    lp = np.empty(rows, np.float64)
    mg = np.empty(rows, np.float64)
    rc = lib.oracle_sample(_ptr(lg), code, _ptr(bi), rows, vocab, int(top_k), float(top_p), _ptr(uu), _ptr(tok),
                           _ptr(lp), _ptr(mg))
    if rc != 0:
        raise ValueError(f"oracle_sample failed ({rc})")
    return {"token": tok, "logprob": lp, "margin": mg}


def cache_refresh_inplace(cache, parent, length):
    """In-place refresh of the [layers, batch*k, heads, max_len, head_dim] cache by parent beam
    (positions < length; every row reads the state before the step).  Returns the new cache."""
    lib = _load()
    out = np.ascontiguousarray(cache).copy()
    layers, rows, heads, max_len, head_dim = out.shape
    par = np.ascontiguousarray(parent, dtype=np.int32)
    batch, k = par.shape
    if batch * k != rows:
        raise ValueError("parent shape does not match cache rows")
    rc = lib.oracle_cache_refresh_inplace(_ptr(out), out.dtype.itemsize, _ptr(par), layers, batch, k, heads, max_len,
                                          int(length), head_dim)
    if rc != 0:
        raise ValueError(f"oracle_cache_refresh_inplace failed ({rc})")
    return out


def logits(hidden, weight, dtype=None):
    """Output projection in double: x[r, v] = sum_d hidden[r, d] * weight[v, d].
    hidden [rows, dim], weight [vocab, dim]: float32, float16, or uint16 bits with dtype 'f16' / 'bf16'.
    Returns float64 [rows, vocab]."""
    lib = _load()
    h, code = _logit_code(np.asarray(hidden), dtype)
    w, wcode = _logit_code(np.asarray(weight), dtype)
    if code != wcode or code == DTYPE_CODES["f64"]:
        raise TypeError("hidden and weight need one element type (f32, f16 or bf16)")
    rows, dim = h.shape
    vocab, dim_w = w.shape
    if dim_w != dim:
        raise ValueError(f"hidden dim {dim} != weight dim {dim_w}")
    out = np.empty((rows, vocab), np.float64)
    rc = lib.oracle_logits(_ptr(h), _ptr(w), code, rows, vocab, dim, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_logits failed ({rc})")
    return out


def logits_beam_step(hidden, weight, beam_scores, *, dtype=None, bias=None, finished=None, eos_id=0, m_out=None):
    """Beam step on the projection's logits: hidden [batch, k, dim], weight [vocab, dim].
    The logits are those of logits() (double); the step is beam_step() on them."""
    hd = np.asarray(hidden)
    batch, k, dim = hd.shape
    x = logits(hd.reshape(batch * k, dim), weight, dtype)
    return beam_step(x.reshape(batch, k, -1), beam_scores, bias=bias, finished=finished, eos_id=eos_id,
                     m_out=m_out)
