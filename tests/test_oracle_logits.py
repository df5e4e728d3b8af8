"""Pins of the oracle's output projection (oracle.logits) and of the beam step on its logits.

The projection is the plain definition x[r, v] = sum_d hidden[r, d] * weight[v, d]; these
tests fix it against values the mathematics decides without the oracle's own formula:
one-hot operands (the product selects one entry, so a wrong index, a transposed operand or a
dropped last term changes the value), integer matrices (exact in double and in numpy's
integer matmul), known bit patterns of f16 / bf16, and the closed form of a projection
whose weight rows are all equal (every logit of a row equal).
"""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (exact for the values used here)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_one_hot_weight_selects_hidden_entries(dtype):
    rng = np.random.default_rng(1)
    rows, vocab, dim = 5, 23, 19
    sel = np.arange(vocab) % dim  # every d, the last one included
    sel[3] = dim - 1
    hv = rng.integers(-64, 64, size=(rows, dim)).astype(np.float32) / 8.0  # exact in every dtype
    w = np.zeros((vocab, dim), np.float32)
    w[np.arange(vocab), sel] = 1.0
    if dtype == "f32":
        h_in, w_in = hv, w
    elif dtype == "f16":
        h_in, w_in = hv.astype(np.float16), w.astype(np.float16)
    else:
        h_in, w_in = bf16_bits(hv), bf16_bits(w)
    x = oracle.logits(h_in, w_in, dtype)
    assert x.shape == (rows, vocab)
    np.testing.assert_array_equal(x, hv.astype(np.float64)[:, sel])


def test_one_hot_hidden_selects_weight_columns():
    rng = np.random.default_rng(2)
    rows, vocab, dim = 4, 17, 9
    w = rng.standard_normal((vocab, dim)).astype(np.float32)
    pick = np.array([0, 8, 3, 8])
    scale = np.array([1.0, -2.0, 0.5, 4.0], np.float32)  # powers of two: exact products
    h = np.zeros((rows, dim), np.float32)
    h[np.arange(rows), pick] = scale
    x = oracle.logits(h, w, "f32")
    np.testing.assert_array_equal(x, (w[:, pick] * scale).T.astype(np.float64))


def test_integer_matrices_match_integer_matmul():
    # small integers: every product and partial sum is exact, so any summation order gives
    # numpy's exact int64 matmul
    rng = np.random.default_rng(3)
    rows, vocab, dim = 7, 31, 64
    h = rng.integers(-8, 9, size=(rows, dim))
    w = rng.integers(-8, 9, size=(vocab, dim))
    x = oracle.logits(bf16_bits(h.astype(np.float32)), bf16_bits(w.astype(np.float32)), "bf16")
    np.testing.assert_array_equal(x, (h @ w.T).astype(np.float64))


def test_known_bit_patterns():
    # bf16 0x3F80 = 1, 0xC000 = -2, 0x3E80 = 0.25; f16 0x3C00 = 1, 0x3555 = 1365/4096
    hb = np.array([[0x3F80, 0xC000, 0x3E80]], np.uint16)
    wb = np.array([[0x3E80, 0x3F80, 0xC000], [0xC000, 0xC000, 0xC000]], np.uint16)
    x = oracle.logits(hb, wb, "bf16")
    np.testing.assert_array_equal(x, [[0.25 - 2.0 - 0.5, -2.0 + 4.0 - 0.5]])
    hf = np.array([[0x3555, 0x3C00]], np.uint16)
    wf = np.array([[0x3C00, 0x3555]], np.uint16)
    x = oracle.logits(hf, wf, "f16")
    assert x[0, 0] == 2 * 1365 / 4096


def test_swapped_operands_transpose():
    rng = np.random.default_rng(4)
    a = bf16_bits(rng.standard_normal((6, 40)).astype(np.float32))
    b = bf16_bits(rng.standard_normal((11, 40)).astype(np.float32))
    x = oracle.logits(a, b, "bf16")
    y = oracle.logits(b, a, "bf16")
    np.testing.assert_array_equal(x, y.T)
    # and the value of one entry by an independent exact computation (Python floats, fsum)
    av, bv = bf16_value(a), bf16_value(b)
    assert x[2, 7] == math.fsum(float(p) * float(q) for p, q in zip(av[2], bv[7]))


def test_dimension_checks():
    with pytest.raises(ValueError):
        oracle.logits(np.zeros((2, 3), np.float32), np.zeros((4, 5), np.float32), "f32")
    with pytest.raises(TypeError):
        oracle.logits(np.zeros((2, 3), np.float32), np.zeros((4, 3), np.float16), None)


def test_beam_step_on_equal_weight_rows_closed_form():
    # every weight row equal -> every logit of a row equal -> s = beam - log V exactly and the
    # selection is the flattened index order (beam 0 tokens first, then beam 1 ...)
    batch, k, vocab, dim = 2, 3, 50, 16
    rng = np.random.default_rng(5)
    h = bf16_bits(rng.standard_normal((batch, k, dim)).astype(np.float32))
    row = bf16_bits(rng.standard_normal(dim).astype(np.float32))
    w = np.tile(row, (vocab, 1))
    beam = np.array([[0.0, -1.0, -2.0], [-0.5, -0.5, -3.0]], np.float32)
    out = oracle.logits_beam_step(h, w, beam, dtype="bf16", eos_id=7)
    for b in range(batch):
        best = int(np.argmax(beam[b]))  # the largest beam score wins, ties by beam index
        np.testing.assert_array_equal(out["parent"][b], [best] * k)
        np.testing.assert_array_equal(out["token"][b], np.arange(k))
        np.testing.assert_allclose(out["score"][b], float(beam[b, best]) - math.log(vocab), rtol=0, atol=1e-12)


def test_beam_step_on_projection_equals_step_on_its_logits():
    # the composed oracle is the beam step of the projection's double logits: with small
    # integer operands the logits are integers, exact in f32 as well, so the step on an f32
    # copy made by numpy's integer matmul must agree exactly (ties included)
    rng = np.random.default_rng(6)
    batch, k, vocab, dim = 3, 4, 97, 32
    h = rng.integers(-4, 5, size=(batch, k, dim)).astype(np.float32)
    w = rng.integers(-4, 5, size=(vocab, dim)).astype(np.float32)
    beam = rng.uniform(-3, 0, size=(batch, k)).astype(np.float32)
    a = oracle.logits_beam_step(bf16_bits(h), bf16_bits(w), beam, dtype="bf16", eos_id=1)
    x = (h.reshape(batch * k, dim).astype(np.int64) @ w.T.astype(np.int64)).astype(np.float32)
    b = oracle.beam_step(x.reshape(batch, k, vocab), beam, eos_id=1)
    np.testing.assert_array_equal(a["token"], b["token"])
    np.testing.assert_array_equal(a["parent"], b["parent"])
    np.testing.assert_allclose(a["score"], b["score"], rtol=0, atol=1e-12)
