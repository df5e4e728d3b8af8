"""Seeded synthetic inputs for the beam-search step and the cache refresh.

Shared by the tests, the benchmark and the smoke check, and by both sides of
every parity check (the oracle and the CUDA library).  It holds none of the
method's arithmetic: only random draws, shapes, and rounding to the storage
dtype.  Every array comes from its own numpy PCG64 stream keyed by
``SeedSequence([seed, tag, step, index])``, so any batch of any step can be
regenerated on its own (sampled parity checks at full size rely on that).

Workloads (variances are read as sigma^2, e.g. N(0,2) has variance 2):

=====  ==============================================================================
name   recipe
=====  ==============================================================================
c1     batch 4, beam 4, vocab 1024, fp32 logits N(0,1), beam scores U(-5,0), seed 0
c2     batch 32, beam 4, vocab 40000, fp32 logits N(0,2) + fp32 bias N(0,0.1),
       beam scores U(-20,0), round(10%) of beams finished, eos 2, seed 1
c3     batch 128, beam 4, vocab 40000, fp16 logits N(0,3), beam scores U(-30,0),
       cache [6, 512, 16, 64, 64] fp16 N(0,1), seed 2
c4     batch 8, beam 8, vocab 120000, fp32 logits 2*t(3); round(5%) of rows get 16
       distinct positions set to (row max + 1); beam scores U(-10,0), seed 3
c5     batch 256, beam 4, vocab 40000, fp16 logits N(0,2) + per-step scalar offset
       U(-5,5) (added before fp16 rounding), 64 steps, step-1 beam scores 0, eos 2,
       cache [6, 1024, 16, 64, 64] fp16 N(0,1), seed 4
p5     the c5 decode step with its logits made by the output projection: batch 256, beam 4,
       vocab 40000, hidden size 1024; decoder states N(0,1) and projection N(0, 2/1024)
       (so the logits are ~N(0,2) as in c5), both bf16; beam scores U(-5,0), eos 2, seed 6
=====  ==============================================================================
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

TAG_LOGITS, TAG_BIAS, TAG_BEAM, TAG_FINISHED, TAG_TIED, TAG_OFFSET, TAG_KV, TAG_PARENT, TAG_UNIFORM = range(1, 10)
TAG_HIDDEN, TAG_WEIGHT = 10, 11

_THREADS = max(1, min(16, os.cpu_count() or 1))


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    k: int
    vocab: int
    dtype: str  # "f32" | "f16" | "bf16"
    seed: int
    logit_dist: str = "normal"  # "normal" | "t3x2"
    logit_var: float = 1.0
    bias_var: float | None = None
    beam_range: tuple[float, float] = (-5.0, 0.0)
    finished_frac: float = 0.0
    tied_frac: float = 0.0
    tied_count: int = 16
    eos_id: int = 2
    steps: int = 1
    step_offset: tuple[float, float] | None = None
    kv_shape: tuple[int, int, int, int] | None = None  # (layers, heads, max_len, head_dim)
    first_step_zero_beams: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.batch * self.k


WORKLOADS = {
    "c1": Workload("c1", 4, 4, 1024, "f32", 0, logit_var=1.0, beam_range=(-5.0, 0.0)),
    "c2": Workload("c2", 32, 4, 40000, "f32", 1, logit_var=2.0, bias_var=0.1, beam_range=(-20.0, 0.0),
                   finished_frac=0.10),
    "c3": Workload("c3", 128, 4, 40000, "f16", 2, logit_var=3.0, beam_range=(-30.0, 0.0),
                   kv_shape=(6, 16, 64, 64)),
    "c4": Workload("c4", 8, 8, 120000, "f32", 3, logit_dist="t3x2", beam_range=(-10.0, 0.0), tied_frac=0.05),
    "c5": Workload("c5", 256, 4, 40000, "f16", 4, logit_var=2.0, steps=64, step_offset=(-5.0, 5.0),
                   kv_shape=(6, 16, 64, 64), first_step_zero_beams=True),
}

NP_DTYPE = {"f32": np.float32, "f16": np.float16}


def rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), *[int(x) for x in key]]))


def _round_to(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return a32.astype(np.float32, copy=False)
    if dtype == "f16":
        return a32.astype(np.float16)
    if dtype == "bf16":  # round-to-nearest-even to the top 16 bits, kept as uint16 bits
        u = a32.astype(np.float32).view(np.uint32)
        lsb = (u >> 16) & 1
        return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    raise ValueError(dtype)


def step_offset(w: Workload, step: int) -> float:
    if w.step_offset is None:
        return 0.0
    lo, hi = w.step_offset
    return float(np.float32(rng(w.seed, TAG_OFFSET, step).uniform(lo, hi)))


def _batch_logits(w: Workload, step: int, b: int, offset: float) -> np.ndarray:
    g = rng(w.seed, TAG_LOGITS, step, b)
    if w.logit_dist == "normal":
        a = g.standard_normal((w.k, w.vocab), dtype=np.float32)
        a *= np.float32(np.sqrt(w.logit_var))
    elif w.logit_dist == "t3x2":
        a = (2.0 * g.standard_t(3, size=(w.k, w.vocab))).astype(np.float32)
    else:
        raise ValueError(w.logit_dist)
    if offset:
        a += np.float32(offset)
    return a


def tied_rows(w: Workload) -> np.ndarray:
    n = int(round(w.tied_frac * w.rows))
    return np.sort(rng(w.seed, TAG_TIED).permutation(w.rows)[:n])


def logits(w: Workload, step: int = 0, batches=None, threads: int | None = None) -> np.ndarray:
    """[len(batches), k, vocab] logits of one step in the workload's storage dtype."""
    batches = list(range(w.batch)) if batches is None else list(batches)
    off = step_offset(w, step)
    tied = set(tied_rows(w).tolist()) if w.tied_frac > 0 else set()
    out_dtype = np.uint16 if w.dtype == "bf16" else NP_DTYPE[w.dtype]
    out = np.empty((len(batches), w.k, w.vocab), out_dtype)

    def one(i):
        b = batches[i]
        a = _batch_logits(w, step, b, off)
        for j in range(w.k):
            row = b * w.k + j
            if row in tied:
                pos = rng(w.seed, TAG_TIED, row).choice(w.vocab, size=w.tied_count, replace=False)
                a[j, pos] = a[j].max() + np.float32(1.0)
        out[i] = _round_to(a, w.dtype)

    nt = threads or _THREADS
    if nt > 1 and len(batches) > 1:
        with _cf.ThreadPoolExecutor(nt) as ex:
            list(ex.map(one, range(len(batches))))
    else:
        for i in range(len(batches)):
            one(i)
    return out


def bias(w: Workload) -> np.ndarray | None:
    if w.bias_var is None:
        return None
    g = rng(w.seed, TAG_BIAS)
    return (g.standard_normal(w.vocab, dtype=np.float32) * np.float32(np.sqrt(w.bias_var))).astype(np.float32)


def beam_scores(w: Workload, step: int = 0) -> np.ndarray:
    if w.first_step_zero_beams and step == 0:
        return np.zeros((w.batch, w.k), np.float32)
    lo, hi = w.beam_range
    return rng(w.seed, TAG_BEAM, step).uniform(lo, hi, (w.batch, w.k)).astype(np.float32)


def finished(w: Workload) -> np.ndarray | None:
    if w.finished_frac <= 0:
        return None
    n = int(round(w.finished_frac * w.rows))
    f = np.zeros(w.rows, np.uint8)
    f[rng(w.seed, TAG_FINISHED).permutation(w.rows)[:n]] = 1
    return f.reshape(w.batch, w.k)


def step_inputs(w: Workload, step: int = 0, batches=None) -> dict:
    """All inputs of one beam step (host arrays)."""
    fin = finished(w)
    bs = beam_scores(w, step)
    if batches is not None:
        idx = np.asarray(list(batches))
        bs = bs[idx]
        fin = None if fin is None else fin[idx]
    return {
        "logits": logits(w, step, batches),
        "bias": bias(w),
        "beam_scores": bs,
        "finished": fin,
        "eos_id": w.eos_id,
        "dtype": w.dtype,
    }


def kv_cache(shape, seed: int, which: int = 0, dtype=np.float16, threads: int | None = None) -> np.ndarray:
    """N(0,1) cache [layers, rows, heads, max_len, head_dim]; one stream per (which, layer, row)."""
    layers, rows = shape[0], shape[1]
    out = np.empty(shape, dtype)

    def one(i):
        l, r = divmod(i, rows)
        g = rng(seed, TAG_KV, which, l, r)
        out[l, r] = g.standard_normal(shape[2:], dtype=np.float32).astype(dtype)

    nt = threads or _THREADS
    with _cf.ThreadPoolExecutor(nt) as ex:
        list(ex.map(one, range(layers * rows)))
    return out


def kv_cache_rows(shape, seed: int, rows_idx, which: int = 0, dtype=np.float16) -> np.ndarray:
    """The same values as kv_cache() for a subset of rows: [layers, len(rows_idx), heads, max_len, head_dim]."""
    rows_idx = list(rows_idx)
    out = np.empty((shape[0], len(rows_idx)) + tuple(shape[2:]), dtype)
    for l in range(shape[0]):
        for i, r in enumerate(rows_idx):
            out[l, i] = rng(seed, TAG_KV, which, l, r).standard_normal(shape[2:], dtype=np.float32).astype(dtype)
    return out


def parents(batch: int, k: int, seed: int, step: int = 0) -> np.ndarray:
    return rng(seed, TAG_PARENT, step).integers(0, k, (batch, k)).astype(np.int32)


def normal(shape, seed: int, *key: int, dtype=np.float32, scale: float = 1.0) -> np.ndarray:
    a = rng(seed, *key).standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a.astype(dtype)


def uniform(shape, lo: float, hi: float, seed: int, *key: int) -> np.ndarray:
    return rng(seed, *key).uniform(lo, hi, shape).astype(np.float32)


# Sampling decoding: one row of logits per sequence (a Workload with k = 1), the kept
# candidates (top_k, top_p) and one uniform per row, all seeded.
#   s1  1024 rows, vocab 40000, fp16 N(0,2), top_k 8, top_p 0.9, u ~ U(0,1), seed 5
SAMPLE_WORKLOADS = {
    "s1": Workload("s1", 1024, 1, 40000, "f16", 5, logit_var=2.0, extra={"top_k": 8, "top_p": 0.9}),
}


def sample_inputs(w: Workload, step: int = 0) -> dict:
    """Logits [rows, vocab], bias, uniforms [rows] (f32 in [0, 1)), top_k and top_p of a sampling workload."""
    lg = logits(w, step).reshape(w.batch, w.vocab)
    u = rng(w.seed, TAG_UNIFORM, step).random(w.batch).astype(np.float32)
    u = np.minimum(u, np.float32(1.0) - np.float32(2.0 ** -24))
    return {"logits": lg, "bias": bias(w), "u": u, "top_k": int(w.extra["top_k"]), "top_p": float(w.extra["top_p"])}


# Projection-fused step (the logits are hidden . weight^T, computed by the step itself).
PROJ_WORKLOADS = {
    "p5": Workload("p5", 256, 4, 40000, "bf16", 6, logit_var=2.0, beam_range=(-5.0, 0.0), extra={"dim": 1024}),
}


def hidden_states(w: Workload, dim: int, step: int = 0, batches=None) -> np.ndarray:
    """Decoder states [batch, k, dim] N(0,1) in w.dtype (bf16 as uint16 bits); one stream per batch."""
    idx = range(w.batch) if batches is None else list(batches)
    out = [_round_to(rng(w.seed, TAG_HIDDEN, step, b).standard_normal((w.k, dim), dtype=np.float32), w.dtype)
           for b in idx]
    return np.stack(out)


def projection(w: Workload, dim: int) -> np.ndarray:
    """Output projection [vocab, dim] N(0, logit_var / dim) in w.dtype (bf16 as uint16 bits)."""
    a = rng(w.seed, TAG_WEIGHT).standard_normal((w.vocab, dim), dtype=np.float32)
    a *= np.float32(np.sqrt(w.logit_var / dim))
    return _round_to(a, w.dtype)


def projection_inputs(w: Workload, dim: int | None = None, step: int = 0, batches=None) -> dict:
    """All inputs of one projection-fused step (host arrays)."""
    dim = int(dim or w.extra["dim"])
    fin = finished(w)
    bs = beam_scores(w, step)
    if batches is not None:
        idx = np.asarray(list(batches))
        bs = bs[idx]
        fin = None if fin is None else fin[idx]
    return {
        "hidden": hidden_states(w, dim, step, batches),
        "weight": projection(w, dim),
        "bias": bias(w),
        "beam_scores": bs,
        "finished": fin,
        "eos_id": w.eos_id,
        "dtype": w.dtype,
        "dim": dim,
    }
