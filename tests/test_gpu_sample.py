"""Sampling decoding on the GPU (ls_sample) against the oracle on the same seeded inputs:
the 1024-row workload s1 in full, random shapes over dtypes, bias, top_k 1..64 and top_p,
ties (all-equal logits, the exact fallback), the forced exact path, and argument checks,
each under the plan's choice, the one-kernel sampler and the two-kernel sampler.

A token must equal the oracle's unless the oracle's uniform lies within 1e-5 of a
cumulative-probability boundary of the kept candidates (both sides then round legitimately
either way); at most MAX_EXCUSED rows of a call may be excused that way.  The
log-probability of an agreeing token is within 1e-5 (fp32 logits) or 2e-3 (fp16, bf16) of
the oracle's."""
import os

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402

MARGIN = 1e-5
MAX_EXCUSED = 2  # rows of one call whose token may differ at a boundary
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


# LS_BEAM_DEBUG settings of the implementations every test runs under: the plan's choice, the
# one-kernel sampler forced wherever top_k <= 8, and the two-kernel sampler (K1 then K5)
IMPLS = {"plan": "", "onekernel": "fused", "twokernel": "nofused"}
_impl_env = {"value": ""}


@pytest.fixture(autouse=True, params=sorted(IMPLS))
def impl(request):
    _impl_env["value"] = IMPLS[request.param]
    yield request.param
    _impl_env["value"] = ""


def _env(extra=None):
    return ",".join(e for e in (_impl_env["value"], extra) if e)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _logits_dev(lg, dtype, dev):
    if dtype == "bf16":
        return torch.from_numpy(lg.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(lg).to(dev)


def run_gpu(dev, lg, dtype, bias, u, top_k, top_p, env=None):
    rows, vocab = lg.shape
    t_lg = _logits_dev(lg, dtype, dev)
    t_b = None if bias is None else torch.from_numpy(bias).to(dev)
    t_u = torch.from_numpy(u).to(dev)
    tok = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    lp = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(lsb.ls_sample_workspace_size(rows, top_k, vocab), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    old = os.environ.get("LS_BEAM_DEBUG")
    try:
        os.environ["LS_BEAM_DEBUG"] = _env(env)
        lsb.check(lsb.ls_sample(t_lg, t_b, t_u, top_k, top_p, tok, lp, ws), "ls_sample")
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    lsb.check(lsb.ls_read_status(ws), "device status")
    return tok.cpu().numpy(), lp.cpu().numpy()


def compare(oracle_mod, lg, dtype, bias, u, top_k, top_p, tok, lp):
    ora = oracle_mod.sample(lg, u.astype(np.float64), top_k, float(np.float32(top_p)), bias=bias, dtype=dtype)
    same = tok == ora["token"]
    near = ora["margin"] < MARGIN
    bad = np.nonzero(~same & ~near)[0]
    assert bad.size == 0, f"rows {bad[:8]}: GPU {tok[bad[:8]]} vs oracle {ora['token'][bad[:8]]}"
    excused = int((~same & near).sum())
    assert excused <= MAX_EXCUSED, f"{excused} rows differ at a cumulative boundary"
    err = np.abs(lp[same].astype(np.float64) - ora["logprob"][same])
    assert err.size == 0 or err.max() <= TOL[dtype], f"logprob error {err.max()}"
    return int(same.sum())


def test_workload_s1(dev, oracle_mod):
    w = synth.SAMPLE_WORKLOADS["s1"]
    inp = synth.sample_inputs(w)
    tok, lp = run_gpu(dev, inp["logits"], w.dtype, inp["bias"], inp["u"], inp["top_k"], inp["top_p"])
    agree = compare(oracle_mod, inp["logits"], w.dtype, inp["bias"], inp["u"], inp["top_k"], inp["top_p"], tok, lp)
    assert agree >= w.batch - 2


def _case(seed):
    g = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][seed % 3]
    vocab = int(g.choice([7, 64, 1000, 4099, 20001, 50257]))
    top_k = int(min(vocab, g.choice([1, 2, 5, 8, 13, 33, 64])))
    top_p = float(g.choice([1.0, 0.9, 0.5, 0.2]))
    rows = int(g.integers(1, 40))
    lg = g.standard_normal((rows, vocab)).astype(np.float32) * np.float32(g.uniform(0.5, 3))
    if dtype == "f16":
        lg = lg.astype(np.float16)
    elif dtype == "bf16":
        uu = lg.view(np.uint32)
        lg = ((uu + 0x7FFF + ((uu >> 16) & 1)) >> 16).astype(np.uint16)
    bias = g.standard_normal(vocab).astype(np.float32) * np.float32(0.3) if seed % 4 == 1 else None
    u = g.random(rows).astype(np.float32)
    return lg, dtype, bias, u, top_k, top_p


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(dev, oracle_mod, seed):
    lg, dtype, bias, u, top_k, top_p = _case(seed)
    tok, lp = run_gpu(dev, lg, dtype, bias, u, top_k, top_p)
    compare(oracle_mod, lg, dtype, bias, u, top_k, top_p, tok, lp)


@pytest.mark.parametrize("seed", range(6))
def test_forced_exact_path_agrees(dev, oracle_mod, seed):
    lg, dtype, bias, u, top_k, top_p = _case(500 + seed)
    a = run_gpu(dev, lg, dtype, bias, u, top_k, top_p)
    b = run_gpu(dev, lg, dtype, bias, u, top_k, top_p, env="exact")
    np.testing.assert_array_equal(a[0], b[0])
    compare(oracle_mod, lg, dtype, bias, u, top_k, top_p, *b)


@pytest.mark.parametrize("top_k", [16, 32, 64])
def test_large_top_k_full_vocab(dev, oracle_mod, top_k):
    """Large top_k at a full vocabulary, where the rows' survivors outnumber a warp's list (the
    bound is raised and the survivors gathered again) or the chunks' slots overflow (each row is
    scanned by its warp): against the oracle."""
    g = np.random.default_rng(top_k)
    rows, vocab = 96, 40000
    lg = (g.standard_normal((rows, vocab)) * 2).astype(np.float16)
    u = g.random(rows).astype(np.float32)
    tok, lp = run_gpu(dev, lg, "f16", None, u, top_k, 0.9)
    compare(oracle_mod, lg, "f16", None, u, top_k, 0.9, tok, lp)


def test_all_equal_logits_take_the_first_tokens(dev, oracle_mod):
    rows, vocab, top_k = 64, 40000, 8
    lg = np.zeros((rows, vocab), np.float16)
    u = ((np.arange(rows) + 0.5) / rows).astype(np.float32)
    tok, lp = run_gpu(dev, lg, "f16", None, u, top_k, 1.0)
    np.testing.assert_array_equal(tok, (np.arange(rows) * top_k) // rows)
    compare(oracle_mod, lg, "f16", None, u, top_k, 1.0, tok, lp)


def test_tied_maxima_and_masked_tokens(dev, oracle_mod):
    g = np.random.default_rng(9)
    rows, vocab, top_k = 20, 30000, 4
    lg = g.standard_normal((rows, vocab)).astype(np.float32)
    for r in range(0, rows, 2):
        lg[r, g.choice(vocab, 16, replace=False)] = lg[r].max() + 1  # 16 tied maxima
    lg[1, :] = -np.inf
    lg[1, 123] = 0.0
    lg[1, 9] = -1.0  # only two finite tokens: top_k 4 keeps them and two -inf ones
    u = g.random(rows).astype(np.float32)
    tok, lp = run_gpu(dev, lg, "f32", None, u, top_k, 1.0)
    compare(oracle_mod, lg, "f32", None, u, top_k, 1.0, tok, lp)


def test_sample_argument_checks(dev):
    lg = torch.zeros((4, 100), dtype=torch.float16, device=dev)
    u = torch.zeros(4, dtype=torch.float32, device=dev)
    tok = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = torch.zeros(lsb.ls_sample_workspace_size(4, 8, 100), dtype=torch.uint8, device=dev)
    assert lsb.ls_sample(lg, None, u, 0, 1.0, tok, None, ws) == lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_sample(lg, None, u, 65, 1.0, tok, None, ws) == lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_sample(lg, None, u, 8, 0.0, tok, None, ws) == lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_sample(lg, None, u, 8, 1.5, tok, None, ws) == lsb.LS_ERR_INVALID_ARG
    small = torch.zeros(64, dtype=torch.uint8, device=dev)
    assert lsb.ls_sample(lg, None, u, 8, 1.0, tok, None, small) == lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_sample_workspace_size(4, 101, 100) == 0


def test_device_wait_timeout_is_reported(dev, oracle_mod):
    """A zero wait budget makes the first traversal's bounded waits run out: the timeout is
    reported by ls_read_status, and a re-initialised workspace gives the oracle's draws again."""
    lg, dtype, bias, u, top_k, top_p = _case(7)
    rows, vocab = lg.shape
    t_lg = _logits_dev(lg, dtype, dev)
    t_b = None if bias is None else torch.from_numpy(bias).to(dev)
    t_u = torch.from_numpy(u).to(dev)
    tok = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    ws = torch.empty(lsb.ls_sample_workspace_size(rows, top_k, vocab), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    old = os.environ.get("LS_BEAM_DEBUG")
    os.environ["LS_BEAM_DEBUG"] = "spin=0,nofused"  # the two-kernel sampler has the bounded waits
    try:
        st = lsb.ls_sample(t_lg, t_b, t_u, top_k, top_p, tok, None, ws)
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    assert st == lsb.LS_OK
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_TIMEOUT
    tok2, lp2 = run_gpu(dev, lg, dtype, bias, u, top_k, top_p)
    compare(oracle_mod, lg, dtype, bias, u, top_k, top_p, tok2, lp2)
