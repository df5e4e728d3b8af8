"""Pins of the oracle's end-of-search backtrack (token sequences of the final beams read back
through the per-step parent pointers), CPU only.

The backward walk is checked against things it does not share code with: a hand-worked
history, the identity-parent closed form, and a forward simulation that carries every beam's
whole prefix and log-probability from step to step (scores recomputed with scipy's logsumexp
from the logits), run on a trajectory produced by the oracle's own beam step.
"""
import numpy as np
import pytest
from scipy.special import logsumexp

import oracle


def test_hand_worked_history():
    # steps x batch x k = 3 x 1 x 2.  Final beam 0: step 3 token 9 from beam 1 of step 2,
    # whose token 8 came from beam 0 of step 1 (token 5)  ->  5 8 9.
    tok = np.array([[[5, 6]], [[7, 8]], [[9, 2]]], np.int32)
    par = np.array([[[0, 1]], [[1, 0]], [[1, 1]]], np.int32)
    seq, ln = oracle.backtrack(tok, par, eos_id=2)
    assert seq.tolist() == [[[5, 8, 9], [5, 8, 2]]]
    assert ln.tolist() == [[3, 3]]
    seq, ln = oracle.backtrack(tok, par, eos_id=8)
    assert ln.tolist() == [[2, 2]]


def test_identity_parents_give_the_columns():
    g = np.random.default_rng(1)
    steps, batch, k = 7, 3, 4
    tok = g.integers(0, 100, (steps, batch, k)).astype(np.int32)
    par = np.broadcast_to(np.arange(k, dtype=np.int32), (steps, batch, k)).copy()
    seq, ln = oracle.backtrack(tok, par, eos_id=1000)
    np.testing.assert_array_equal(seq, np.transpose(tok, (1, 2, 0)))
    assert (ln == steps).all()


def test_lengths_stop_at_the_first_eos():
    steps, batch, k = 6, 1, 2
    tok = np.full((steps, batch, k), 4, np.int32)
    par = np.broadcast_to(np.arange(k, dtype=np.int32), (steps, batch, k)).copy()
    tok[2, 0, 0] = 3
    tok[4, 0, 0] = 3  # a second eos does not move the length
    tok[5, 0, 1] = 3
    _, ln = oracle.backtrack(tok, par, eos_id=3)
    assert ln.tolist() == [[3, 6]]


def test_out_of_range_parent_is_rejected():
    tok = np.zeros((2, 1, 2), np.int32)
    par = np.array([[[0, 1]], [[0, 2]]], np.int32)
    with pytest.raises(ValueError):
        oracle.backtrack(tok, par, eos_id=0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_backtrack_matches_a_forward_simulation(seed):
    g = np.random.default_rng(100 + seed)
    batch, k, vocab, steps, eos = 3, 3, 40, 6, 5
    beam = g.uniform(-3, 0, (batch, k)).astype(np.float32)
    fin = np.zeros((batch, k), np.uint8)
    prefix = [[[] for _ in range(k)] for _ in range(batch)]
    logp = beam.astype(np.float64).copy()
    toks, pars = [], []
    for _ in range(steps):
        lg = (g.standard_normal((batch, k, vocab)) * 2).astype(np.float32)
        r = oracle.beam_step(lg, beam, finished=fin, eos_id=eos)
        toks.append(r["token"])
        pars.append(r["parent"])
        # forward: every new beam = its parent's prefix + its token; its log-probability grows by
        # log-softmax(logits of the parent row)[token], or not at all when the parent had finished
        new_prefix = [[None] * k for _ in range(batch)]
        new_logp = np.empty_like(logp)
        for b in range(batch):
            for j in range(k):
                p, t = int(r["parent"][b, j]), int(r["token"][b, j])
                new_prefix[b][j] = prefix[b][p] + [t]
                x = lg[b, p].astype(np.float64)
                new_logp[b, j] = logp[b, p] + (0.0 if fin[b, p] else x[t] - logsumexp(x))
        prefix, logp = new_prefix, new_logp
        beam = r["score"].astype(np.float32)
        fin = r["finished"]
        np.testing.assert_allclose(r["score"], logp, rtol=0, atol=1e-5)
    seq, ln = oracle.backtrack(np.stack(toks), np.stack(pars), eos_id=eos)
    for b in range(batch):
        for j in range(k):
            assert seq[b, j].tolist() == prefix[b][j]
            first = [i for i, t in enumerate(prefix[b][j]) if t == eos]
            assert ln[b, j] == (first[0] + 1 if first else steps)
