"""Pins of the oracle to facts that do not come from the oracle itself.

Each test fixes part of what the LightSeq inference article (31duo.com,
itemid-283120, hierarchical decoding section) defines, by a route independent
of the oracle's C code: brute force on tiny inputs (repeated argmax instead of
a sort), closed forms, invariants, library routines (scipy's logsumexp,
numpy's fp16 decoding and fancy indexing), and the article's k=2 / vocab=8
example counts.  A plausible slip in the oracle (a dropped bias or beam score,
a wrong sign on lse, swapped token/parent, a reversed tie-break, a wrong
finished-beam rule, an fp16 decoding error, a wrong gather index) fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_force(x, beam, finished, eos, k):
    """Repeated argmax over all (beam, token) pairs of one batch; math.fsum log-sum-exp."""
    kk, vocab = x.shape
    cands = []
    for j in range(kk):
        if finished is not None and finished[j]:
            cands.append((float(beam[j]), j * vocab + eos))
            continue
        m = max(x[j])
        lse = m + math.log(math.fsum(math.exp(v - m) for v in x[j]))
        for v in range(vocab):
            cands.append((float(beam[j]) + float(x[j, v]) - lse, j * vocab + v))
    out = []
    used = set()
    for _ in range(k):
        best = None
        for i, (s, flat) in enumerate(cands):
            if i in used:
                continue
            if best is None or s > cands[best][0] or (s == cands[best][0] and flat < cands[best][1]):
                best = i
        used.add(best)
        out.append(cands[best])
    return out


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny(oracle_mod, seed):
    g = np.random.default_rng(1000 + seed)
    batch, k, vocab = int(g.integers(1, 3)), int(g.integers(1, 4)), int(g.integers(1, 7))
    vocab = max(vocab, k)
    # a coarse value grid produces exact ties, exercising the tie-break
    logits = (g.integers(-3, 4, (batch, k, vocab)) * 0.5).astype(np.float32)
    beam = (g.integers(-4, 1, (batch, k)) * 0.25).astype(np.float32)
    bias = (g.integers(-2, 3, vocab) * 0.25).astype(np.float32) if seed % 2 else None
    fin = (g.random((batch, k)) < 0.3).astype(np.uint8) if seed % 3 == 0 else None
    eos = int(g.integers(0, vocab))
    r = oracle_mod.beam_step(logits, beam, bias=bias, finished=fin, eos_id=eos)
    for b in range(batch):
        x = logits[b].astype(np.float64) + (0.0 if bias is None else bias.astype(np.float64))
        ref = _brute_force(x, beam[b], None if fin is None else fin[b], eos, k)
        for r_i, (s, flat) in enumerate(ref):
            assert r["parent"][b, r_i] == flat // vocab
            assert r["token"][b, r_i] == flat % vocab
            assert abs(r["score"][b, r_i] - s) < 1e-12
            par = flat // vocab
            exp_fin = bool(fin is not None and fin[b, par]) or (flat % vocab == eos)
            assert bool(r["finished"][b, r_i]) == exp_fin


def test_all_equal_logits_closed_form(oracle_mod):
    """Equal logits in a row give p = 1/V exactly: s = beam - log V, order = index order."""
    batch, k, vocab = 3, 4, 37
    logits = np.full((batch, k, vocab), 1.75, np.float32)
    beam = np.array([[-1.0, -0.5, -0.5, -3.0], [0.0, 0.0, 0.0, 0.0], [-2.0, -1.0, -4.0, -1.0]], np.float32)
    r = oracle_mod.beam_step(logits, beam, eos_id=0)
    for b in range(batch):
        order = sorted(range(k), key=lambda j: (-beam[b, j], j))
        # every token of the best beam ties, so the top-k is its first k token ids
        # unless another beam has the same score (then lower flat index first: same beam, lower ids)
        exp = []
        for j in order:
            for v in range(vocab):
                exp.append((j, v))
        exp = exp[:k]
        for i, (j, v) in enumerate(exp):
            assert r["parent"][b, i] == j and r["token"][b, i] == v
            assert abs(r["score"][b, i] - (float(beam[b, j]) - math.log(vocab))) < 1e-12


def test_greedy_k1_is_argmax(oracle_mod):
    g = np.random.default_rng(7)
    logits = g.standard_normal((5, 1, 333)).astype(np.float32)
    logits[2, 0, [10, 20]] = 9.0  # tie: smaller index wins
    beam = g.uniform(-3, 0, (5, 1)).astype(np.float32)
    r = oracle_mod.beam_step(logits, beam, eos_id=1)
    assert (r["token"][:, 0] == np.argmax(logits[:, 0, :], axis=1)).all()
    assert (r["parent"] == 0).all()
    exp = beam[:, 0].astype(np.float64) + logits.max(axis=2)[:, 0].astype(np.float64) - logsumexp(logits[:, 0, :].astype(np.float64), axis=1)
    np.testing.assert_allclose(r["score"][:, 0], exp, rtol=0, atol=1e-12)


def test_lse_matches_scipy_and_fsum(oracle_mod):
    g = np.random.default_rng(11)
    logits = (g.standard_normal((2, 3, 5000)) * 4).astype(np.float32)
    logits[1, 2] += 800.0  # large values: a missing max-shift overflows exp
    r = oracle_mod.beam_step(logits, np.zeros((2, 3), np.float32), eos_id=0)
    ref = logsumexp(logits.astype(np.float64), axis=2)
    np.testing.assert_allclose(r["lse"], ref, rtol=0, atol=1e-11)
    row = logits[0, 1].astype(np.float64)
    m = row.max()
    assert abs(r["lse"][0, 1] - (m + math.log(math.fsum(math.exp(v - m) for v in row)))) < 1e-11


def test_softmax_normalises(oracle_mod):
    """Full candidate list: sum over a live beam of exp(s - beam) = 1 (probabilities)."""
    g = np.random.default_rng(3)
    batch, k, vocab = 2, 3, 50
    logits = g.standard_normal((batch, k, vocab)).astype(np.float32)
    beam = g.uniform(-5, 0, (batch, k)).astype(np.float32)
    bias = g.standard_normal(vocab).astype(np.float32)
    r = oracle_mod.beam_step(logits, beam, bias=bias, eos_id=0, m_out=k * vocab)
    for b in range(batch):
        for j in range(k):
            sel = r["parent"][b] == j
            assert sel.sum() == vocab
            p = np.exp(r["score"][b][sel] - float(beam[b, j]))
            assert abs(math.fsum(p) - 1.0) < 1e-12
            # within one beam, scores follow the logits + bias order
            toks = r["token"][b][sel]
            xs = logits[b, j, toks].astype(np.float64) + bias[toks]
            assert (np.diff(xs) <= 0).all()


def test_shift_invariance(oracle_mod):
    """Adding a constant to one beam's logits changes nothing (lse absorbs it)."""
    g = np.random.default_rng(5)
    # values on a 2^-10 grid, so that adding the shifts below is exact in fp32
    logits = (np.round(g.standard_normal((3, 4, 200)) * 1024) / 1024).astype(np.float32)
    beam = g.uniform(-5, 0, (3, 4)).astype(np.float32)
    shift = np.array([0.0, 64.0, -32.0, 1024.0], np.float32)[None, :, None]
    a = oracle_mod.beam_step(logits, beam, eos_id=0)
    b = oracle_mod.beam_step(logits + shift, beam, eos_id=0)
    assert (a["token"] == b["token"]).all() and (a["parent"] == b["parent"]).all()
    np.testing.assert_allclose(a["score"], b["score"], rtol=0, atol=1e-9)


def test_bias_equals_logits(oracle_mod):
    g = np.random.default_rng(9)
    vocab = 300
    bias = g.standard_normal(vocab).astype(np.float32)
    beam = g.uniform(-2, 0, (2, 3)).astype(np.float32)
    a = oracle_mod.beam_step(np.zeros((2, 3, vocab), np.float32), beam, bias=bias, eos_id=0)
    b = oracle_mod.beam_step(np.broadcast_to(bias, (2, 3, vocab)).copy(), beam, eos_id=0)
    for key in ("token", "parent", "score"):
        assert (a[key] == b[key]).all()


def test_vocab_permutation(oracle_mod):
    g = np.random.default_rng(13)
    logits = g.standard_normal((2, 3, 400)).astype(np.float32)
    beam = g.uniform(-2, 0, (2, 3)).astype(np.float32)
    perm = g.permutation(400)
    a = oracle_mod.beam_step(logits, beam, eos_id=0)
    b = oracle_mod.beam_step(logits[:, :, perm], beam, eos_id=0)
    inv = np.argsort(perm)
    assert (perm[b["token"]] == a["token"]).all() or (b["token"] == inv[a["token"]]).all()
    np.testing.assert_allclose(a["score"], b["score"], rtol=0, atol=1e-12)


def test_finished_beam_rule(oracle_mod):
    vocab = 16
    logits = np.zeros((1, 3, vocab), np.float32)
    logits[0, 2, 5] = 10.0
    beam = np.array([[0.0, -1.0, -50.0]], np.float32)
    fin = np.array([[1, 0, 1]], np.uint8)
    r = oracle_mod.beam_step(logits, beam, finished=fin, eos_id=3, m_out=4)
    # beam 0 finished: exactly one candidate (eos, score unchanged); beam 2 finished: its big logit is ignored
    assert (r["parent"][0, 0], r["token"][0, 0], r["score"][0, 0], r["finished"][0, 0]) == (0, 3, 0.0, 1)
    assert r["parent"][0, 1] == 1 and r["token"][0, 1] == 0
    assert abs(r["score"][0, 1] - (-1.0 - math.log(vocab))) < 1e-12
    assert r["finished"][0, 1] == 0
    # the live beam's eos token is marked finished
    r2 = oracle_mod.beam_step(logits, beam, finished=fin, eos_id=3, m_out=1 + vocab + 1)
    toks = list(zip(r2["parent"][0], r2["token"][0], r2["finished"][0]))
    assert (1, 3, 1) in toks and (2, 3, 1) in toks
    assert sum(1 for p, t, f in toks if p == 2) == 1


def test_minus_inf_beam_scores(oracle_mod):
    logits = np.random.default_rng(2).standard_normal((1, 2, 10)).astype(np.float32)
    beam = np.array([[-np.inf, -np.inf]], np.float32)
    r = oracle_mod.beam_step(logits, beam, eos_id=0, m_out=3)
    assert np.isneginf(r["score"]).all()
    assert list(r["token"][0]) == [0, 1, 2] and list(r["parent"][0]) == [0, 0, 0]


def test_fp16_and_bf16_decoding(oracle_mod):
    g = np.random.default_rng(21)
    bits = g.integers(0, 1 << 16, (2, 2, 3000), dtype=np.uint64).astype(np.uint16)
    # drop NaN/inf patterns; keep subnormals and large finite values
    h = bits.view(np.float16)
    h[~np.isfinite(h)] = np.float16(0.0)
    h = h / np.float16(256)  # keep exp() sane while keeping subnormal patterns
    beam = np.zeros((2, 2), np.float32)
    a = oracle_mod.beam_step(h, beam, eos_id=0, m_out=6)
    b = oracle_mod.beam_step(h.astype(np.float32), beam, eos_id=0, m_out=6)
    for key in ("token", "parent", "score"):
        assert (a[key] == b[key]).all()
    f32 = g.standard_normal((2, 2, 3000)).astype(np.float32)
    bf = (f32.view(np.uint32) >> 16).astype(np.uint16)
    as_f32 = (bf.astype(np.uint32) << 16).view(np.float32)
    c = oracle_mod.beam_step(bf, beam, eos_id=0, m_out=6, dtype="bf16")
    d = oracle_mod.beam_step(as_f32, beam, eos_id=0, m_out=6)
    for key in ("token", "parent", "score"):
        assert (c[key] == d[key]).all()


# ---------------------------------------------------------------- R-top-k (first traversal)


@pytest.mark.parametrize("dist", ["normal", "t3", "ties", "coarse"])
def test_rtopk_lower_bound(oracle_mod, dist):
    g = np.random.default_rng(hash(dist) % 1000)
    for k in (1, 2, 3, 4, 8, 17):
        vocab = 500 + 37 * k
        if dist == "normal":
            x = g.standard_normal((6, vocab))
        elif dist == "t3":
            x = 2 * g.standard_t(3, (6, vocab))
        elif dist == "ties":
            x = g.standard_normal((6, vocab))
            x[:, g.choice(vocab, 20, replace=False)] = x.max() + 1
        else:
            x = g.integers(-2, 3, (6, vocab)).astype(float)
        x = x.astype(np.float32)
        for groups in (k, 2 * k + 1):
            st = oracle_mod.rtopk_stats(x, k, groups=groups)
            kth = -np.sort(-x.astype(np.float64), axis=1)[:, k - 1]
            np.testing.assert_array_equal(st["kth"], kth)
            assert (st["R"] <= st["kth"]).all()
            # the candidate set (x >= R) contains every row's top-k
            assert (st["ncand"] >= k).all()
            assert (st["ncand"] == (x.astype(np.float64) >= st["R"][:, None]).sum(axis=1)).all()


def test_rtopk_group_rule(oracle_mod):
    g = np.random.default_rng(4)
    k, vocab = 4, 4000
    x = g.standard_normal((5, vocab)).astype(np.float32)
    st = oracle_mod.rtopk_stats(x, k)
    gmax = x.reshape(5, vocab // k, k).max(axis=1)  # group g = {v : v mod k == g}
    np.testing.assert_array_equal(st["R"], gmax.min(axis=1).astype(np.float64))
    # with k == vocab every group has one element, R is the row minimum and every token survives
    y = x[:, :k]
    st2 = oracle_mod.rtopk_stats(y, k)
    np.testing.assert_array_equal(st2["R"], y.min(axis=1).astype(np.float64))
    assert (st2["ncand"] == k).all()


def _read_golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            d[key] = [float(t) for t in val.split()]
    return d


def test_k2_v8_example_counts(oracle_mod):
    d = _read_golden("k2_v8_example.txt")
    k, vocab = int(d["k"][0]), int(d["vocab"][0])
    x = np.array([d["beam0"], d["beam1"]], np.float32)
    assert x.size == int(d["elements_before"][0]) == 16
    st = oracle_mod.rtopk_stats(x, k)
    np.testing.assert_array_equal(st["R"], np.array(d["R"], np.float32).astype(np.float64))
    assert list(st["ncand"]) == [int(c) for c in d["ncand"]]
    assert st["ncand"].sum() == int(d["elements_after"][0]) == 5


def test_k2_v8_statistics_match_article(oracle_mod):
    """Soft check: on N(0,1) logits, k=2, vocab=8 keeps about 5 of 16 elements per sequence."""
    x = synth.normal((20000 * 2, 8), 77, 1)
    st = oracle_mod.rtopk_stats(x, 2)
    per_seq = st["ncand"].reshape(-1, 2).sum(axis=1).mean()
    assert 4.5 < per_seq < 6.0, per_seq


def test_top4_keeps_about_a_dozen(oracle_mod):
    """Soft check: k=4 over tens of thousands of N(0,sigma^2) tokens keeps on the order of ten per beam."""
    x = synth.normal((64, 40000), 78, 1, scale=math.sqrt(2.0))
    st = oracle_mod.rtopk_stats(x, 4)
    assert 5 < st["ncand"].mean() < 20


# ---------------------------------------------------------------- cache refresh


@pytest.mark.parametrize("dtype", [np.float16, np.float32, np.uint8])
def test_cache_reorder_matches_fancy_indexing(oracle_mod, dtype):
    g = np.random.default_rng(8)
    layers, batch, k, heads, max_len, head_dim = 2, 3, 4, 3, 9, 5
    src = g.integers(0, 255, (layers, batch * k, heads, max_len, head_dim)).astype(dtype)
    parent = g.integers(0, k, (batch, k)).astype(np.int32)
    for length in (0, 1, 5, max_len):
        sentinel = np.full_like(src, 7)
        out = oracle_mod.cache_reorder(src, parent, length, dst=sentinel.copy())
        rows = (np.arange(batch)[:, None] * k + parent).reshape(-1)
        exp = sentinel.copy()
        exp[:, :, :, :length] = src[:, rows][:, :, :, :length]
        assert out.tobytes() == exp.tobytes()


def test_cache_reorder_rejects_bad_parent(oracle_mod):
    src = np.zeros((1, 4, 1, 2, 2), np.float16)
    with pytest.raises(ValueError):
        oracle_mod.cache_reorder(src, np.array([[0, 1], [2, 0]], np.int32), 2)
