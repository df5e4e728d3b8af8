"""Comparison of the CUDA beam step with the oracle, shared by the GPU tests.

The rule (hierarchical decoding is exact, so the GPU must reproduce the naive
definition): per batch, the selected (token, parent) pairs equal the oracle's
top-k, except that a pair may differ when the oracle's score gap at the k-th
place is below GAP_TOL; scores agree within 1e-5 for fp32 logits and 2e-3 for
fp16/bf16 logits; the order agrees except between candidates whose oracle scores
are within GAP_TOL of each other.
"""
from __future__ import annotations

import numpy as np

GAP_TOL = 1e-4
SCORE_TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def compare_step(gpu: dict, ora: dict, k: int, dtype: str, finished=None, eos_id: int = 0,
                 batches=None, score_tol=None, gap_tol=None) -> dict:
    """gpu: token/parent/score/finished [B, k] numpy; ora: oracle.beam_step(..., m_out >= k + 1).
    score_tol / gap_tol (floats, or arrays indexed by batch) replace the dtype's tolerances.
    Returns counts; raises AssertionError with a message on a violation."""
    B = gpu["token"].shape[0]
    batches = range(B) if batches is None else batches
    near_ties = 0
    for b in batches:
        tol = SCORE_TOL[dtype] if score_tol is None else float(np.broadcast_to(score_tol, (B,))[b])
        gtol = GAP_TOL if gap_tol is None else float(np.broadcast_to(gap_tol, (B,))[b])
        o_pairs = list(zip(ora["parent"][b].tolist(), ora["token"][b].tolist()))
        o_score = ora["score"][b]
        s_k = o_score[k - 1]
        look = {pt: float(s) for pt, s in zip(o_pairs, o_score) if pt[0] >= 0}
        g_pairs = list(zip(gpu["parent"][b].tolist(), gpu["token"][b].tolist()))
        g_score = gpu["score"][b].astype(np.float64)
        # scores: monotone, and matching the oracle's score of the same pair
        assert np.all(np.diff(g_score) <= 0) or np.all(np.isneginf(g_score)), f"batch {b}: scores not sorted"
        o_of_g = []
        for i, pt in enumerate(g_pairs):
            assert pt in look, f"batch {b}: GPU pair {pt} (rank {i}) outside the oracle's top-{len(o_pairs)}"
            so = look[pt]
            o_of_g.append(so)
            if np.isfinite(so):
                assert abs(g_score[i] - so) <= tol, f"batch {b} rank {i}: score {g_score[i]} vs oracle {so}"
            else:
                assert g_score[i] == so, f"batch {b} rank {i}: score {g_score[i]} vs oracle {so}"
            assert so >= s_k - gtol or (np.isneginf(so) and np.isneginf(s_k)), \
                f"batch {b}: GPU pair {pt} score {so} below the k-th oracle score {s_k}"
        # set and order: identical unless the oracle has near-ties there
        if g_pairs != o_pairs[:k]:
            tied = False
            if set(g_pairs) != set(o_pairs[:k]):
                gap = o_score[k - 1] - o_score[k]
                assert gap < gtol, f"batch {b}: selected set differs with oracle gap {gap}"
                tied = True
            for i in range(k - 1):
                assert o_of_g[i] >= o_of_g[i + 1] - gtol, f"batch {b}: order differs beyond near-ties"
            near_ties += 1
            _ = tied
        # finished flag
        for i, (par, tok) in enumerate(g_pairs):
            exp = bool(finished is not None and finished[b, par]) or tok == eos_id
            assert bool(gpu["finished"][b, i]) == exp, f"batch {b} rank {i}: finished flag"
    return {"near_ties": near_ties}


def boundary_gaps(ora: dict, k: int) -> np.ndarray:
    """Per batch, the smallest gap between consecutive oracle scores among the first k+1."""
    s = ora["score"][:, : k + 1]
    d = s[:, :-1] - s[:, 1:]
    d = np.where(np.isnan(d), np.inf, d)
    return d.min(axis=1)


def projection_logit_bound(hidden_vals: np.ndarray, weight_vals: np.ndarray) -> np.ndarray:
    """Bound on |computed - exact| of every logit of the projection-fused step, [rows, vocab].

    The products of two f16 / bf16 values are exact in f32; the tensor cores add the dim
    products of a logit in f32, at most dim / 16 additions into the accumulator (one per
    16-element instruction) plus the additions inside an instruction, each rounding by at
    most 2^-23 of a partial sum whose magnitude is at most sum_d |h_d w_d|.  Taking 16
    roundings for the inside of an instruction and doubling for margin:
        B = 2 * (dim / 16 + 16) * 2^-23 * sum_d |h_d w_d|.
    hidden_vals [rows, dim], weight_vals [vocab, dim] as float64 values."""
    dim = hidden_vals.shape[1]
    return 2.0 * (dim / 16 + 16) * 2.0 ** -23 * (np.abs(hidden_vals) @ np.abs(weight_vals).T)
