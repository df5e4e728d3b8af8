"""In-place, copy-on-change cache refresh on the GPU (ls_cache_refresh_inplace) against the
oracle, bitwise: parent patterns that make in-place writing hazardous (swaps, cycles, one
parent for all), every element width, odd head sizes, k up to 64 (slabs staged in several
tiles), len < max_len, a bad parent reported through the workspace, and a c5 decode loop
refreshed in place against the oracle's trajectory.  The cases run under each implementation:
the plan's choice, the word kernel, bulk copies and the staged CTA kernel."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402
from serving_ls_beam_gb300.loop import BeamSearchLoop  # noqa: E402

NP = {"f16": np.float16, "f32": np.float32, "bf16": np.uint16}
TDT = {"f16": torch.float16, "f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _cache(g, shape, dtype):
    if dtype == "bf16":
        return g.integers(0, 1 << 15, shape).astype(np.uint16)
    return g.standard_normal(shape).astype(NP[dtype])


def _to_dev(a, dtype, dev):
    t = torch.from_numpy(a)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev)


def _bits(t, dtype):
    a = t.cpu()
    if dtype == "bf16":
        a = a.view(torch.int16)
    a = a.numpy()
    return a.view(np.int16) if a.dtype == np.float16 else (a.view(np.int32) if a.dtype == np.float32 else a)


def _parents(g, batch, k):
    pats = [np.zeros(k), np.arange(k), np.roll(np.arange(k), 1), np.arange(k)[::-1], g.integers(0, k, k)]
    return np.stack([pats[b % len(pats)] for b in range(batch)]).astype(np.int32)


CASES = [  # (dtype, layers, batch, k, heads, max_len, len, head_dim)
    ("f16", 2, 10, 4, 3, 16, 16, 64),
    ("f16", 3, 7, 4, 2, 16, 9, 64),
    ("f32", 1, 6, 8, 2, 12, 5, 33),
    ("bf16", 2, 5, 3, 4, 8, 8, 7),
    ("f16", 1, 4, 64, 2, 64, 64, 64),  # 64 rows of 8 KB slabs: staged in tiles
    ("f32", 2, 3, 5, 1, 10, 1, 16),
    ("f16", 1, 3, 4, 16, 64, 20, 64),  # short slabs: 3 heads per item, a last group of 1
    ("f16", 2, 5, 4, 7, 64, 3, 64),    # all 7 heads in one item
    ("f16", 2, 6, 4, 16, 64, 6, 64),   # word kernel: 48 words a slab, items of 5 heads (5, 5, 5, 1)
    ("bf16", 1, 9, 8, 3, 32, 32, 64),  # word kernel, k = 8, 1 head per item
    ("f16", 1, 5, 2, 4, 16, 1, 8),     # one 16-byte word per slab
]

# LS_BEAM_DEBUG settings of the implementations: the plan's choice (the word kernel for short
# slabs and k <= 8, bulk copies otherwise), the word kernel, bulk copies (with a workspace,
# also with a fixed share of items per CTA, and with items sized for one needed parent, so
# that an item takes several steps) and the staged CTA kernel forced
IMPLS = [None, "ipwords", "iptma", "iptma,ipstatic", "iptma,ipkeff=1", "ipplain"]


def _with_env(env, fn):
    import os

    old = os.environ.get("LS_BEAM_DEBUG")
    try:
        if env is not None:
            os.environ["LS_BEAM_DEBUG"] = env
        return fn()
    finally:
        if env is not None:
            if old is None:
                os.environ.pop("LS_BEAM_DEBUG", None)
            else:
                os.environ["LS_BEAM_DEBUG"] = old


@pytest.mark.parametrize("with_ws", [False, True])
@pytest.mark.parametrize("env", IMPLS)
@pytest.mark.parametrize("case", CASES)
def test_inplace_matches_oracle(dev, oracle_mod, case, env, with_ws):
    """Bitwise against the oracle.  With a workspace the bulk-copy kernel's CTAs take items from
    a counter in it (twice in a row here, so the second call starts from the counter the first
    left); without one each CTA takes a fixed share."""
    dtype, layers, batch, k, heads, max_len, length, head_dim = case
    g = np.random.default_rng(CASES.index(case))
    shape = (layers, batch * k, heads, max_len, head_dim)
    cache = _cache(g, shape, dtype)
    parent = _parents(g, batch, k)
    parent2 = _parents(g, batch, k)
    t = _to_dev(cache, dtype, dev)
    ws = None
    if with_ws:
        ws = torch.empty(lsb.ls_beam_step_workspace_size(1, 1, 1), dtype=torch.uint8, device=dev)
        lsb.check(lsb.ls_workspace_init(ws))
    for par in (parent, parent2):
        _with_env(env, lambda: lsb.check(lsb.ls_cache_refresh_inplace(t, torch.from_numpy(par).to(dev), length, ws),
                                         "ls_cache_refresh_inplace"))
    want = oracle_mod.cache_refresh_inplace(oracle_mod.cache_refresh_inplace(cache, parent, length), parent2, length)
    got = _bits(t, dtype)
    exp = want.view(got.dtype) if want.dtype != got.dtype else want
    assert np.array_equal(got, exp)
    if with_ws:
        assert lsb.ls_read_status(ws) == lsb.LS_OK
        assert (ws[:256].cpu().numpy() == 0).all()  # the status word and the work counter are back to zero


@pytest.mark.parametrize("env", IMPLS)
def test_bad_parent_leaves_the_row_and_is_reported(dev, oracle_mod, env):
    g = np.random.default_rng(3)
    shape = (1, 8, 2, 4, 16)
    cache = g.standard_normal(shape).astype(np.float16)
    parent = np.array([[1, 0, 3, 2], [0, 7, 1, 1]], np.int32)
    ws = torch.zeros(lsb.ls_beam_step_workspace_size(1, 1, 1), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    t = torch.from_numpy(cache).to(dev)
    _with_env(env, lambda: lsb.check(lsb.ls_cache_refresh_inplace(t, torch.from_numpy(parent).to(dev), 4, ws)))
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_INTERNAL
    fixed = parent.copy()
    fixed[1, 1] = 1  # the bad row is left as it is
    want = oracle_mod.cache_refresh_inplace(cache, fixed, 4)
    assert np.array_equal(t.cpu().numpy().view(np.int16), want.view(np.int16))


def test_c5_loop_refreshed_in_place(dev, oracle_mod):
    """16 decode steps of c5 with the cache refreshed in place; sampled batches against the
    oracle's own trajectory.  A batch leaves the comparison only when the oracle shows a
    near-tie at the k-th place (the trajectories may then part legitimately); until then
    every step's selection must equal the oracle's, and the final cache rows must match."""
    from parity import GAP_TOL, boundary_gaps, compare_step

    w = synth.WORKLOADS["c5"]
    layers, heads, max_len, head_dim = w.kv_shape
    shape = (layers, w.rows, heads, max_len, head_dim)
    steps = 16
    sample = [0, 45, 128, 255]
    cache = torch.from_numpy(synth.kv_cache(shape, w.seed, which=0)).to(dev)
    loop = BeamSearchLoop(w.batch, w.k, w.vocab, w.eos_id, kv_shape=w.kv_shape, device=dev, caches=[cache],
                          inplace=True)
    loop.reset(torch.from_numpy(synth.beam_scores(w, 0)).to(dev))
    rows = [b * w.k + j for b in sample for j in range(w.k)]
    o_cache = synth.kv_cache_rows(shape, w.seed, rows, which=0)
    o_beam = synth.beam_scores(w, 0)[sample].copy()
    o_fin = np.zeros((len(sample), w.k), np.uint8)
    alive = set(range(len(sample)))
    compared = 0
    for t in range(1, steps + 1):
        lg = synth.logits(w, t)
        idx = loop.step(torch.from_numpy(lg).to(dev), t)
        out = {key: v.cpu().numpy()[sample] for key, v in loop.outputs(idx).items()}
        ora = oracle_mod.beam_step(lg[sample], o_beam, finished=o_fin, eos_id=w.eos_id, m_out=w.k + 8)
        gaps = boundary_gaps(ora, w.k)
        for i in sorted(alive):
            compare_step(out, ora, w.k, w.dtype, finished=o_fin, eos_id=w.eos_id, batches=[i])
            if gaps[i] < GAP_TOL:
                alive.discard(i)
            else:
                assert (out["token"][i] == ora["token"][i, : w.k]).all()
                assert (out["parent"][i] == ora["parent"][i, : w.k]).all()
                compared += 1
        o_cache = oracle_mod.cache_refresh_inplace(o_cache, ora["parent"][:, : w.k].astype(np.int32), t)
        o_beam = ora["score"][:, : w.k].astype(np.float32)
        o_fin = ora["finished"][:, : w.k].astype(np.uint8)
    assert alive and compared >= len(sample) * steps // 2
    final = loop.current_cache()[:, rows].cpu().numpy()
    for i in sorted(alive):
        sl = slice(i * w.k, (i + 1) * w.k)
        assert np.array_equal(final[:, sl, :, :steps].view(np.int16), o_cache[:, sl, :, :steps].view(np.int16))


def test_bulk_copy_wait_timeout_is_reported(dev, oracle_mod):
    """A zero wait budget makes the bulk-copy kernel's bounded waits run out: it records a
    timeout in the workspace and returns after the copies it issued have landed; the context
    stays usable and, on a restored cache, the same call gives the oracle's result."""
    g = np.random.default_rng(11)
    dtype, layers, batch, k, heads, max_len, length, head_dim = ("f16", 2, 10, 4, 3, 16, 16, 64)
    shape = (layers, batch * k, heads, max_len, head_dim)
    cache = _cache(g, shape, dtype)
    parent = torch.from_numpy(_parents(g, batch, k)).to(dev)
    ws = torch.zeros(lsb.ls_beam_step_workspace_size(1, 1, 1), dtype=torch.uint8, device=dev)
    t = _to_dev(cache, dtype, dev)
    _with_env("spin=0,iptma", lambda: lsb.check(lsb.ls_cache_refresh_inplace(t, parent, length, ws)))
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_TIMEOUT
    lsb.check(lsb.ls_workspace_init(ws))
    t = _to_dev(cache, dtype, dev)
    lsb.check(lsb.ls_cache_refresh_inplace(t, parent, length, ws))
    assert lsb.ls_read_status(ws) == lsb.LS_OK
    want = oracle_mod.cache_refresh_inplace(cache, parent.cpu().numpy(), length)
    assert np.array_equal(_bits(t, dtype), want.view(np.int16))
