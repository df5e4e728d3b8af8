"""GPU parity of ls_beam_step against the oracle (called through the C ABI).

Workloads c1-c4 run at their full sizes, in the launch configuration the
benchmark uses, and are compared with the oracle element by element, and so
does one step of the multi-step workload c5 (all 256 batches); its whole
decode loop is covered in test_gpu_multistep.py.  The sweeps below
add ragged vocabularies (not a multiple of the 16-byte vector), misaligned
logits, k = 1 and k = 64, vocab == k, bias, finished beams and bf16.

Every test runs under each implementation of the step (the `impl` fixture):
the plan's own choice, the one-kernel step K3 forced wherever k <= 8, and the
two-kernel step (K1 + K2) forced everywhere.
"""
import os

import numpy as np
import pytest

import synth
from parity import compare_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# LS_BEAM_DEBUG settings of the implementations every test runs under: the plan's choice, K3
# (a CTA per batch), K3's cluster form (a CTA per row, a cluster per batch), K1s then K2
IMPLS = {"plan": "", "onekernel": "fused", "cluster": "cluster", "twokernel": "nofused"}
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


def _to_dev(a, dev, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype) if t.dtype in (torch.int16,) else t
    return t.to(dev)


def logits_tensor(lg: np.ndarray, dtype: str, dev, offset_elems: int = 0):
    """Device logits; with offset_elems > 0 they start that many elements into a larger buffer."""
    if dtype == "bf16":
        base = torch.from_numpy(lg.view(np.int16)).view(torch.bfloat16)
    else:
        base = torch.from_numpy(lg)
    if offset_elems:
        flat = torch.empty(base.numel() + offset_elems, dtype=base.dtype)
        flat[offset_elems:] = base.reshape(-1)
        return flat.to(dev)[offset_elems:].view(base.shape)
    return base.to(dev)


def run_gpu(inp, dev, offset_elems=0, workspace=None, env=None):
    lg = inp["logits"]
    B, K, V = lg.shape
    dtype = inp["dtype"]
    t_lg = logits_tensor(lg, dtype, dev, offset_elems)
    t_bias = None if inp.get("bias") is None else torch.from_numpy(inp["bias"]).to(dev)
    t_beam = torch.from_numpy(np.ascontiguousarray(inp["beam_scores"], np.float32)).to(dev)
    t_fin = None if inp.get("finished") is None else torch.from_numpy(inp["finished"].astype(np.uint8)).to(dev)
    out_tok = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    out_par = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    out_sc = torch.full((B, K), float("nan"), dtype=torch.float32, device=dev)
    out_fin = torch.full((B, K), 9, dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
        lsb.check(lsb.ls_workspace_init(workspace))
    old = os.environ.get("LS_BEAM_DEBUG")
    os.environ["LS_BEAM_DEBUG"] = _env(env)
    try:
        st = lsb.ls_beam_step(t_lg, t_bias, t_beam, t_fin, inp["eos_id"], out_tok, out_par, out_sc, out_fin,
                              workspace)
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    lsb.check(st, "ls_beam_step")
    lsb.check(lsb.ls_read_status(workspace), "device status")
    torch.cuda.synchronize()
    res = {"token": out_tok.cpu().numpy(), "parent": out_par.cpu().numpy(), "score": out_sc.cpu().numpy(),
           "finished": out_fin.cpu().numpy()}
    return res, workspace


def run_oracle(oracle_mod, inp, m_extra=8):
    K = inp["logits"].shape[1]
    return oracle_mod.beam_step(inp["logits"], inp["beam_scores"], bias=inp.get("bias"), finished=inp.get("finished"),
                                eos_id=inp["eos_id"], m_out=K + m_extra, dtype=inp["dtype"])


_oracle_cache = {}


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_workload_parity(dev, oracle_mod, impl, name):
    """Every batch of each workload at its full size (c5: one step of its decode loop, step 1,
    whose beams are no longer tied, all 256 batches)."""
    w = synth.WORKLOADS[name]
    inp = synth.step_inputs(w, 1 if name == "c5" else 0)
    gpu, ws = run_gpu(inp, dev)
    if name not in _oracle_cache:  # the same inputs under every implementation
        _oracle_cache[name] = run_oracle(oracle_mod, inp)
    ora = _oracle_cache[name]
    compare_step(gpu, ora, w.k, w.dtype, finished=inp["finished"], eos_id=w.eos_id)
    # diagnostics: lse per beam and the R-top-k lower bound against the true k-th largest
    lse, rtopk, ncand, path = lsb.ls_read_row_stats(ws, w.batch, w.k, w.vocab)
    live = np.ones((w.batch, w.k), bool) if inp["finished"] is None else inp["finished"] == 0
    tol = 1e-5 if w.dtype == "f32" else 2e-3
    np.testing.assert_allclose(lse[live], ora["lse"][live], rtol=0, atol=tol)
    # the kernel works on x = fp32(logit + bias); its R-top-k must not exceed the k-th largest of those
    x32 = inp["logits"].astype(np.float32)
    if inp["bias"] is not None:
        x32 = x32 + inp["bias"][None, None, :]
    st = oracle_mod.rtopk_stats(x32, w.k)
    kth = st["kth"].reshape(w.batch, w.k)
    assert (rtopk[live].astype(np.float64) <= kth[live]).all()
    assert (path == 0).all()
    assert (ncand[live] >= 1).all()


def _random_case(seed):
    g = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][seed % 3]
    k = int(g.choice([1, 2, 3, 4, 5, 8, 13, 16, 33, 64]))
    vocab = int(max(k, g.choice([k, 7, 64, 1000, 4099, 8191, 12289, 20001, 50257])))
    batch = int(g.integers(1, 6))
    lg = g.standard_normal((batch, k, vocab)).astype(np.float32) * np.float32(g.uniform(0.5, 3))
    if dtype == "f16":
        lg = lg.astype(np.float16)
    elif dtype == "bf16":
        u = lg.view(np.uint32)
        lg = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    bias = g.standard_normal(vocab).astype(np.float32) * np.float32(0.3) if seed % 4 == 1 else None
    fin = (g.random((batch, k)) < 0.2).astype(np.uint8) if seed % 5 == 2 else None
    beam = g.uniform(-10, 0, (batch, k)).astype(np.float32)
    offset = int(g.choice([0, 0, 1, 3, 5]))
    return {"logits": lg, "bias": bias, "beam_scores": beam, "finished": fin, "eos_id": int(g.integers(0, vocab)),
            "dtype": dtype}, offset


@pytest.mark.parametrize("seed", range(36))
def test_random_shapes(dev, oracle_mod, seed):
    inp, offset = _random_case(seed)
    gpu, _ = run_gpu(inp, dev, offset_elems=offset)
    ora = run_oracle(oracle_mod, inp)
    k = inp["logits"].shape[1]
    compare_step(gpu, ora, k, inp["dtype"], finished=inp["finished"], eos_id=inp["eos_id"])


@pytest.mark.parametrize("seed", range(6))
def test_forced_exact_path(dev, oracle_mod, seed):
    """The exact fallback (radix select per beam) gives the same answer as the queue path."""
    inp, offset = _random_case(100 + seed)
    gpu_q, _ = run_gpu(inp, dev, offset_elems=offset)
    gpu_x, ws = run_gpu(inp, dev, offset_elems=offset, env="exact")
    B, K, V = inp["logits"].shape
    _, _, _, path = lsb.ls_read_row_stats(ws, B, K, V)
    assert (path == 2).all()
    ora = run_oracle(oracle_mod, inp)
    compare_step(gpu_x, ora, K, inp["dtype"], finished=inp["finished"], eos_id=inp["eos_id"])
    for key in ("token", "parent", "score", "finished"):
        assert (gpu_q[key] == gpu_x[key]).all()


@pytest.mark.parametrize("k", [16, 32, 64])
def test_large_k_exact_path(dev, oracle_mod, k):
    """Large beams at a full vocabulary: the k-group bound lets hundreds of candidates per beam
    through, the queue overflows and the exact path selects from the slots (or, where a chunk's
    slots overflowed, from the rows), one warp per beam.  Outputs against the oracle, and the
    path taken is the exact one for at least one batch."""
    g = np.random.default_rng(k)
    B, V = 4, 40000
    lg = (g.standard_normal((B, k, V)) * 2).astype(np.float16)
    inp = {"logits": lg, "bias": None, "beam_scores": g.uniform(-10, 0, (B, k)).astype(np.float32),
           "finished": None, "eos_id": 2, "dtype": "f16"}
    gpu, ws = run_gpu(inp, dev)
    _, _, _, path = lsb.ls_read_row_stats(ws, B, k, V)
    if _impl_env["value"] in ("", "nofused"):
        assert (np.asarray(path) != 0).any()
    ora = run_oracle(oracle_mod, inp)
    compare_step(gpu, ora, k, "f16", eos_id=2)


def test_all_equal_logits_overflow(dev, oracle_mod):
    """Every logit ties with R-top-k: the chunk slots overflow and the exact fallback answers."""
    B, K, V = 3, 4, 40000
    lg = np.full((B, K, V), 0.5, np.float32)
    beam = np.array([[-1, -0.5, -0.5, -3], [0, 0, 0, 0], [-2, -1, -4, -1]], np.float32)
    inp = {"logits": lg, "bias": None, "beam_scores": beam, "finished": None, "eos_id": 2, "dtype": "f32"}
    gpu, ws = run_gpu(inp, dev)
    _, _, _, path = lsb.ls_read_row_stats(ws, B, K, V)
    assert (path == 1).all()
    ora = run_oracle(oracle_mod, inp)
    for key in ("token", "parent"):
        assert (gpu[key] == ora[key][:, :K]).all()
    np.testing.assert_allclose(gpu["score"], ora["score"][:, :K], rtol=0, atol=1e-5)


def test_tied_maxima_and_masked_tokens(dev, oracle_mod):
    g = np.random.default_rng(5)
    B, K, V = 2, 8, 30011
    lg = (g.standard_normal((B, K, V)) * 2).astype(np.float32)
    lg[0, 3, g.choice(V, 16, replace=False)] = lg[0, 3].max() + 1.0
    lg[1, :, g.choice(V, 500, replace=False)] = -np.inf  # masked vocabulary entries
    lg[1, 5, :] = -np.inf
    lg[1, 5, 17] = 3.0  # a beam with a single finite logit
    inp = {"logits": lg, "bias": None, "beam_scores": g.uniform(-3, 0, (B, K)).astype(np.float32),
           "finished": None, "eos_id": 1, "dtype": "f32"}
    gpu, _ = run_gpu(inp, dev)
    ora = run_oracle(oracle_mod, inp)
    compare_step(gpu, ora, K, "f32", eos_id=1)


def test_minus_inf_beams_and_all_finished(dev, oracle_mod):
    g = np.random.default_rng(6)
    B, K, V = 3, 4, 5000
    lg = g.standard_normal((B, K, V)).astype(np.float32)
    beam = g.uniform(-3, 0, (B, K)).astype(np.float32)
    beam[0, :] = -np.inf          # every beam dead: tokens 0..k-1 of beam 0
    beam[1, 1] = -np.inf
    fin = np.zeros((B, K), np.uint8)
    fin[2, :] = 1                 # every beam finished
    fin[1, 3] = 1
    inp = {"logits": lg, "bias": None, "beam_scores": beam, "finished": fin, "eos_id": 7, "dtype": "f32"}
    gpu, _ = run_gpu(inp, dev)
    ora = run_oracle(oracle_mod, inp)
    compare_step(gpu, ora, K, "f32", finished=fin, eos_id=7)
    assert list(gpu["token"][0]) == [0, 1, 2, 3] and list(gpu["parent"][0]) == [0, 0, 0, 0]
    assert (gpu["token"][2] == 7).all() and (gpu["finished"][2] == 1).all()


def test_workspace_reuse_across_shapes(dev, oracle_mod):
    """One workspace sized for the largest shape serves smaller steps in turn."""
    big = synth.WORKLOADS["c2"]
    ws = torch.empty(lsb.ls_beam_step_workspace_size(big.batch, 8, 120000), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    for name in ("c1", "c2", "c1", "c4"):
        w = synth.WORKLOADS[name]
        inp = synth.step_inputs(w, 0)
        gpu, _ = run_gpu(inp, dev, workspace=ws)
        ora = run_oracle(oracle_mod, inp)
        compare_step(gpu, ora, w.k, w.dtype, finished=inp["finished"], eos_id=w.eos_id)


def test_repeat_is_deterministic(dev):
    w = synth.WORKLOADS["c3"]
    inp = synth.step_inputs(w, 0)
    a, ws = run_gpu(inp, dev)
    b, _ = run_gpu(inp, dev, workspace=ws)
    for key in a:
        assert (a[key] == b[key]).all()


def test_invalid_arguments(dev):
    B, K, V = 2, 4, 100
    lg = torch.zeros((B, K, V), device=dev)
    beam = torch.zeros((B, K), device=dev)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    par = torch.empty_like(tok)
    sc = torch.empty((B, K), device=dev)
    ws = torch.zeros(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    E = lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_beam_step(lg, None, beam, None, V, tok, par, sc, None, ws) == E  # eos out of range
    assert lsb.ls_beam_step(lg, None, beam, None, 0, tok, par, sc, None, ws[:100]) == E  # workspace too small
    host = torch.zeros((B, K, V))
    assert lsb.ls_beam_step(host, None, beam, None, 0, tok, par, sc, None, ws) == E  # pageable host memory
    lib = lsb.load_library()
    assert lib.ls_beam_step(lg.data_ptr(), 0, None, beam.data_ptr(), None, B, 0, V, 0, tok.data_ptr(),
                            par.data_ptr(), sc.data_ptr(), None, ws.data_ptr(), ws.numel(), None) == E  # k = 0
    assert lib.ls_beam_step(lg.data_ptr(), 0, None, beam.data_ptr(), None, B, 65, 200, 0, tok.data_ptr(),
                            par.data_ptr(), sc.data_ptr(), None, ws.data_ptr(), ws.numel(), None) == E  # k > 64
    assert lib.ls_beam_step(lg.data_ptr() + 1, 0, None, beam.data_ptr(), None, B, K, V, 0, tok.data_ptr(),
                            par.data_ptr(), sc.data_ptr(), None, ws.data_ptr(), ws.numel(), None) == E  # misaligned
    # an empty batch is a no-op
    assert lib.ls_beam_step(None, 0, None, None, None, 0, K, V, 0, None, None, None, None, None, 0, None) == lsb.LS_OK


def test_device_wait_timeout_is_reported(dev):
    """A zero wait budget makes the bounded waits run out: the kernel records a timeout and
    returns after the copies it issued have landed; the context stays usable."""
    w = synth.WORKLOADS["c2"]
    inp = synth.step_inputs(w, 0)
    B, K, V = inp["logits"].shape
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    t_lg = torch.from_numpy(inp["logits"]).to(dev)
    t_beam = torch.from_numpy(inp["beam_scores"]).to(dev)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    par, sc = torch.empty_like(tok), torch.empty((B, K), device=dev)
    os.environ["LS_BEAM_DEBUG"] = _env("spin=0,nofused")  # the two-kernel step has the bounded waits
    try:
        st = lsb.ls_beam_step(t_lg, None, t_beam, None, 2, tok, par, sc, None, ws)
    finally:
        os.environ.pop("LS_BEAM_DEBUG", None)
    assert st == lsb.LS_OK
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_TIMEOUT
    # the context is still usable, and a re-initialised workspace gives correct results again
    lsb.check(lsb.ls_workspace_init(ws))
    gpu, _ = run_gpu(inp, dev, workspace=ws)
    assert (gpu["token"] >= 0).all()
