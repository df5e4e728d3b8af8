"""ls_beam_step_refresh_inplace: the beam step followed by the in-place cache refresh by its
parents, as two launches by default and, with LS_BEAM_DEBUG=steprefresh, in one kernel where
the step runs a batch per CTA.  Its outputs and its cache must equal, bitwise, those of
ls_beam_step followed by ls_cache_refresh_inplace; the outputs are checked against the
oracle's beam step and the cache against the oracle's refresh by the GPU's parents.  Cases:
c3 and one c5 step at several lengths in both forms, random shapes with the one-kernel form
forced (every logit and cache dtype, bias, finished beams, k from 1 to 8, slabs the bulk
copies cannot take), the default form, and a zero wait budget."""
import os

import numpy as np
import pytest

import synth
from parity import compare_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402

TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _env(value, fn):
    old = os.environ.get("LS_BEAM_DEBUG")
    try:
        if value is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = value
        return fn()
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old


def _logits(lg, dtype, dev):
    t = torch.from_numpy(lg)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev)


def _cache_np(g, shape, dtype):
    if dtype == "bf16":
        return g.integers(0, 1 << 15, shape).astype(np.uint16)
    return g.standard_normal(shape).astype(np.float16 if dtype == "f16" else np.float32)


def _cache_dev(a, dtype, dev):
    t = torch.from_numpy(a)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev)


def _bits(t):
    a = t.cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    a = a.numpy()
    return a.view(np.int16) if a.dtype == np.float16 else (a.view(np.int32) if a.dtype == np.float32 else a)


def _run(inp, cache, length, dev, combined, env=None):
    """Outputs (numpy) and the device cache after the step and the refresh."""
    lg = inp["logits"]
    B, K, V = lg.shape
    t_lg = _logits(lg, inp["dtype"], dev)
    bias = None if inp.get("bias") is None else torch.from_numpy(inp["bias"]).to(dev)
    beam = torch.from_numpy(np.ascontiguousarray(inp["beam_scores"], np.float32)).to(dev)
    fin = None if inp.get("finished") is None else torch.from_numpy(inp["finished"].astype(np.uint8)).to(dev)
    tok = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    par = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    sc = torch.full((B, K), float("nan"), device=dev)
    fo = torch.full((B, K), 9, dtype=torch.uint8, device=dev)
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))

    def go():
        if combined:
            return lsb.ls_beam_step_refresh_inplace(t_lg, bias, beam, fin, inp["eos_id"], tok, par, sc, fo, cache,
                                                    length, ws)
        st = lsb.ls_beam_step(t_lg, bias, beam, fin, inp["eos_id"], tok, par, sc, fo, ws)
        return st if st != lsb.LS_OK else lsb.ls_cache_refresh_inplace(cache, par, length, ws)

    lsb.check(_env(env, go), "step and refresh")
    status = lsb.ls_read_status(ws)
    torch.cuda.synchronize()
    out = {"token": tok.cpu().numpy(), "parent": par.cpu().numpy(), "score": sc.cpu().numpy(),
           "finished": fo.cpu().numpy()}
    return out, status


def _check(inp, cache_np, cache_dtype, length, dev, oracle_mod, env=None):
    c_sep = _cache_dev(cache_np, cache_dtype, dev)
    c_one = _cache_dev(cache_np, cache_dtype, dev)
    o_sep, st_sep = _run(inp, c_sep, length, dev, False, env)
    o_one, st_one = _run(inp, c_one, length, dev, True, env)
    assert st_sep == lsb.LS_OK and st_one == lsb.LS_OK
    for key in ("token", "parent", "score", "finished"):
        assert np.array_equal(o_one[key].view(np.uint8), o_sep[key].view(np.uint8)), key
    got = _bits(c_one)
    assert np.array_equal(got, _bits(c_sep))
    # the outputs against the oracle's step, the cache against the oracle's refresh
    K = inp["logits"].shape[1]
    ora = oracle_mod.beam_step(inp["logits"], inp["beam_scores"], bias=inp.get("bias"), finished=inp.get("finished"),
                               eos_id=inp["eos_id"], m_out=K + 8, dtype=inp["dtype"])
    compare_step(o_one, ora, K, inp["dtype"], finished=inp.get("finished"), eos_id=inp["eos_id"])
    want = oracle_mod.cache_refresh_inplace(cache_np, o_one["parent"], length)
    assert np.array_equal(got, want.view(got.dtype))


@pytest.mark.parametrize("env", [None, "steprefresh"])
@pytest.mark.parametrize("length", [1, 7, 33, 64])
def test_c3_step_and_refresh(dev, oracle_mod, length, env):
    w = synth.WORKLOADS["c3"]
    layers, heads, max_len, head_dim = w.kv_shape
    cache = synth.kv_cache((layers, w.rows, heads, max_len, head_dim), w.seed)
    _check(synth.step_inputs(w, 0), cache, "f16", length, dev, oracle_mod, env=env)


@pytest.mark.parametrize("env", [None, "steprefresh"])
@pytest.mark.parametrize("length", [2, 64])
def test_c5_step_and_refresh(dev, oracle_mod, length, env):
    w = synth.WORKLOADS["c5"]
    layers, heads, max_len, head_dim = w.kv_shape
    cache = synth.kv_cache((layers, w.rows, heads, max_len, head_dim), w.seed)
    _check(synth.step_inputs(w, length), cache, "f16", length, dev, oracle_mod, env=env)


def _random_case(seed):
    g = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][seed % 3]
    k = int(g.choice([1, 2, 3, 4, 5, 8]))
    vocab = int(g.choice([64, 1000, 4099, 20001]))
    batch = int(g.integers(1, 7))
    lg = g.standard_normal((batch, k, vocab)).astype(np.float32) * np.float32(g.uniform(0.5, 3))
    if dtype == "f16":
        lg = lg.astype(np.float16)
    elif dtype == "bf16":
        u = lg.view(np.uint32)
        lg = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    bias = g.standard_normal(vocab).astype(np.float32) * np.float32(0.3) if seed % 4 == 1 else None
    fin = (g.random((batch, k)) < 0.2).astype(np.uint8) if seed % 5 == 2 else None
    beam = g.uniform(-10, 0, (batch, k)).astype(np.float32)
    inp = {"logits": lg, "bias": bias, "beam_scores": beam, "finished": fin, "eos_id": int(g.integers(0, vocab)),
           "dtype": dtype}
    cache_dtype = ["f16", "f32", "bf16"][(seed // 3) % 3]
    layers, heads = int(g.integers(1, 4)), int(g.integers(1, 6))
    max_len = int(g.choice([4, 16, 64]))
    head_dim = int(g.choice([8, 64, 33, 7]))  # 33 and 7: slabs the bulk copies cannot take
    length = int(g.integers(1, max_len + 1))
    cache = _cache_np(g, (layers, batch * k, heads, max_len, head_dim), cache_dtype)
    return inp, cache, cache_dtype, length


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_one_kernel(dev, oracle_mod, seed):
    inp, cache, cache_dtype, length = _random_case(seed)
    _check(inp, cache, cache_dtype, length, dev, oracle_mod, env="fused,steprefresh")


@pytest.mark.parametrize("seed", range(4))
def test_default_two_launches(dev, oracle_mod, seed):
    inp, cache, cache_dtype, length = _random_case(50 + seed)
    _check(inp, cache, cache_dtype, length, dev, oracle_mod)


def test_refresh_wait_timeout_is_reported(dev, oracle_mod):
    """A zero wait budget makes the refresh's bounded waits in the one-kernel step run out: the
    timeout is reported, the copies issued land, and the call on a restored cache is exact."""
    w = synth.WORKLOADS["c3"]
    layers, heads, max_len, head_dim = w.kv_shape
    cache = synth.kv_cache((layers, w.rows, heads, max_len, head_dim), w.seed)
    inp = synth.step_inputs(w, 0)
    c = _cache_dev(cache, "f16", dev)
    _, st = _run(inp, c, 64, dev, True, env="spin=0,steprefresh")
    assert st == lsb.LS_ERR_TIMEOUT
    _check(inp, cache, "f16", 64, dev, oracle_mod)
