"""End-of-search backtrack on the GPU (ls_backtrack) against the oracle, bit-exact:
random histories of many shapes (one tile of steps and several, k = 1 .. 64), eos
lengths, a parent outside [0, k) reported through the workspace status, and argument
checks."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _history(g, steps, batch, k, vocab, eos):
    tok = g.integers(0, vocab, (steps, batch, k)).astype(np.int32)
    tok[g.random(tok.shape) < 0.05] = eos
    par = g.integers(0, k, (steps, batch, k)).astype(np.int32)
    return tok, par


def _run(dev, tok, par, eos, ws=None):
    steps, batch, k = tok.shape
    t = torch.from_numpy(tok).to(dev)
    p = torch.from_numpy(par).to(dev)
    seq = torch.full((batch, k, steps), -7, dtype=torch.int32, device=dev)
    ln = torch.full((batch, k), -7, dtype=torch.int32, device=dev)
    lsb.check(lsb.ls_backtrack(t, p, eos, seq, ln, ws), "ls_backtrack")
    torch.cuda.synchronize()
    return seq.cpu().numpy(), ln.cpu().numpy()


# (steps, batch, k): single step, ragged, the c5 shape, several tiles of steps (4096 / k per tile)
SHAPES = [(1, 1, 1), (5, 3, 4), (64, 256, 4), (150, 5, 64), (1000, 2, 8), (7, 4, 33), (4097, 1, 1), (3, 2, 2)]


@pytest.mark.parametrize("shape", SHAPES)
def test_backtrack_matches_oracle(dev, oracle_mod, shape):
    steps, batch, k = shape
    g = np.random.default_rng(steps * 1000 + batch * 10 + k)
    tok, par = _history(g, steps, batch, k, vocab=500, eos=3)
    seq, ln = _run(dev, tok, par, 3)
    o_seq, o_len = oracle_mod.backtrack(tok, par, 3)
    np.testing.assert_array_equal(seq, o_seq)
    np.testing.assert_array_equal(ln, o_len)


def test_bad_parent_is_reported(dev, oracle_mod):
    g = np.random.default_rng(5)
    tok, par = _history(g, 10, 3, 4, vocab=50, eos=1)
    par[9, 1, 2] = 9  # the last step: final beam 2 of batch 1 follows it
    ws = torch.zeros(lsb.ls_beam_step_workspace_size(1, 1, 1), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    seq, _ = _run(dev, tok, par, 1, ws)
    # batch 1 is unspecified; the other batches must be exact
    o_seq, _ = oracle_mod.backtrack(tok[:, [0, 2]], par[:, [0, 2]], 1)
    np.testing.assert_array_equal(seq[[0, 2]], o_seq)
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_INTERNAL
    assert lsb.ls_read_status(ws) == lsb.LS_OK
    # the context is still usable
    tok2, par2 = _history(g, 4, 2, 2, vocab=50, eos=1)
    seq2, ln2 = _run(dev, tok2, par2, 1)
    o2, l2 = oracle_mod.backtrack(tok2, par2, 1)
    np.testing.assert_array_equal(seq2, o2)


def test_backtrack_argument_checks(dev):
    t = torch.zeros((4, 2, 3), dtype=torch.int32, device=dev)
    seq = torch.zeros((2, 3, 4), dtype=torch.int32, device=dev)
    ln = torch.zeros((2, 3), dtype=torch.int32, device=dev)
    lib = lsb.load_library()
    assert lib.ls_backtrack(None, t.data_ptr(), 4, 2, 3, 0, seq.data_ptr(), ln.data_ptr(), None, None) == \
        lsb.LS_ERR_INVALID_ARG
    assert lib.ls_backtrack(t.data_ptr(), t.data_ptr(), 4, 2, 65, 0, seq.data_ptr(), ln.data_ptr(), None, None) == \
        lsb.LS_ERR_INVALID_ARG
    assert lib.ls_backtrack(t.data_ptr(), t.data_ptr(), -1, 2, 3, 0, seq.data_ptr(), ln.data_ptr(), None, None) == \
        lsb.LS_ERR_INVALID_ARG
    assert lib.ls_backtrack(t.data_ptr(), t.data_ptr(), 0, 2, 3, 0, seq.data_ptr(), ln.data_ptr(), None, None) == \
        lsb.LS_OK
