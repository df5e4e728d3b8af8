"""GPU parity of ls_logits_beam_step (the beam step fused into the output projection) against
the oracle's projection + naive beam step, called through the C ABI.

The logits are computed on the tensor cores (exact products, f32 sums in an unspecified
order), so the comparison allows, per batch, the logit error bound of
parity.projection_logit_bound: scores agree within twice that bound (the logit and the
log-sum-exp each move by at most the bound) plus 1e-5, and a selected pair may differ
from the oracle's only where the oracle's score gap is below twice the score tolerance.

The cases span several 128-row blocks and chunks (of 1 to 4 sub-tiles of 256 tokens) with ragged tails in rows,
vocab and hidden size (not a multiple of the 64-element stage), k = 1 ... 32 (group counts
1 ... 32, k below and equal to its group count), f16 and bf16, bias, finished beams, vocab
equal to k, ties heavy enough to overflow a chunk's slots (the chunk then keeps its own top
k) and to overflow the batch queue (the fine rank then selects from the slots), the fine
rank's exact path forced on every batch, and the full-size p5 workload on sampled batches.
"""
import os

import numpy as np
import pytest

import synth
from parity import compare_step, projection_logit_bound

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def values(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.float64)  # float16 array


def dev_tensor(a: np.ndarray, dtype: str, dev):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev)


def run_gpu(inp, dev, env=None, repeat=1):
    H, W = inp["hidden"], inp["weight"]
    B, K, D = H.shape
    V = W.shape[0]
    dtype = inp["dtype"]
    th, tw = dev_tensor(H, dtype, dev), dev_tensor(W, dtype, dev)
    tb = None if inp.get("bias") is None else torch.from_numpy(inp["bias"]).to(dev)
    beam = torch.from_numpy(np.ascontiguousarray(inp["beam_scores"], dtype=np.float32)).to(dev)
    fin = None if inp.get("finished") is None else torch.from_numpy(inp["finished"]).to(dev)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    par = torch.empty_like(tok)
    sc = torch.empty((B, K), dtype=torch.float32, device=dev)
    of = torch.empty((B, K), dtype=torch.uint8, device=dev)
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws), "init")
    old = os.environ.get("LS_BEAM_DEBUG")
    if env is not None:
        os.environ["LS_BEAM_DEBUG"] = env
    try:
        outs = []
        for _ in range(repeat):
            lsb.check(lsb.ls_logits_beam_step(th, tw, tb, beam, fin, inp["eos_id"], tok, par, sc, of, ws),
                      "ls_logits_beam_step")
            torch.cuda.synchronize()
            lsb.check(lsb.ls_read_status(ws), "device status")
            outs.append({"token": tok.cpu().numpy().copy(), "parent": par.cpu().numpy().copy(),
                         "score": sc.cpu().numpy().copy(), "finished": of.cpu().numpy().copy()})
    finally:
        if env is not None:
            if old is None:
                os.environ.pop("LS_BEAM_DEBUG", None)
            else:
                os.environ["LS_BEAM_DEBUG"] = old
    lse, _, _, path = lsb.ls_read_row_stats(ws, B, K, V)
    out = outs[0]
    out["lse"] = lse
    out["path"] = path
    out["all"] = outs
    return out


def tolerances(inp, batches=None):
    H, W = inp["hidden"], inp["weight"]
    B, K, D = H.shape
    hv = values(H, inp["dtype"]).reshape(-1, D)
    wv = values(W, inp["dtype"])
    bound = projection_logit_bound(hv, wv).reshape(B, K, -1).max(axis=(1, 2))
    score_tol = 2.0 * bound + 1e-5
    return score_tol, 2.0 * score_tol, bound


def oracle_step(oracle, inp, m_out):
    return oracle.logits_beam_step(inp["hidden"], inp["weight"], inp["beam_scores"], dtype=inp["dtype"],
                                   bias=inp.get("bias"), finished=inp.get("finished"), eos_id=inp["eos_id"],
                                   m_out=m_out)


def check(oracle, inp, gpu):
    K = inp["hidden"].shape[1]
    ora = oracle_step(oracle, inp, K + 8)
    score_tol, gap_tol, bound = tolerances(inp)
    compare_step(gpu, ora, K, inp["dtype"], finished=inp.get("finished"), eos_id=inp["eos_id"],
                 score_tol=score_tol, gap_tol=gap_tol)
    # per-beam log-sum-exp of the live beams
    live = np.ones(ora["lse"].shape, bool) if inp.get("finished") is None else inp["finished"] == 0
    fin_ok = np.isfinite(ora["lse"]) & live
    err = np.abs(gpu["lse"].astype(np.float64) - ora["lse"])[fin_ok]
    tol = (bound[:, None] + 1e-5 * (1 + np.abs(ora["lse"])))[fin_ok]
    assert np.all(err <= tol), f"lse error {err.max()} above {tol.min()}"
    return ora


def make(batch, k, vocab, dim, dtype="bf16", seed=11, bias_var=None, finished_frac=0.0, beam_range=(-5.0, 0.0)):
    w = synth.Workload(f"t{seed}", batch, k, vocab, dtype, seed, logit_var=2.0, bias_var=bias_var,
                       beam_range=beam_range, finished_frac=finished_frac)
    return synth.projection_inputs(w, dim=dim)


CASES = [
    # batch, k, vocab, dim, dtype, bias_var, finished_frac
    (2, 4, 1000, 64, "bf16", None, 0.0),      # one row block, a ragged second chunk
    (40, 4, 5000, 200, "bf16", 0.1, 0.1),     # 2 row blocks, hidden size not a multiple of 64, bias
    (3, 1, 777, 128, "bf16", None, 0.0),      # k = 1 (one group)
    (5, 3, 3000, 96, "f16", None, 0.0),       # k below its group count (4), f16
    (16, 8, 2600, 136, "bf16", 0.1, 0.0),     # k = 8
    (9, 16, 1500, 64, "bf16", None, 0.0),     # 16 groups
    (4, 32, 1100, 64, "f16", None, 0.0),      # 32 groups
    (7, 5, 2049, 512, "bf16", None, 0.2),     # k = 5 of 8 groups, one-token last chunk
    (3, 4, 4, 64, "bf16", None, 0.0),         # vocab == k
    (70, 4, 1300, 72, "bf16", None, 0.0),     # 3 row blocks, the last partial
    (1, 2, 40000, 1024, "bf16", 0.1, 0.0),    # the full vocab and hidden size, one batch
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}k{c[1]}v{c[2]}d{c[3]}{c[4]}" for c in CASES])
def test_parity(dev, oracle_mod, case):
    batch, k, vocab, dim, dtype, bias_var, ff = case
    inp = make(batch, k, vocab, dim, dtype, seed=100 + k + vocab % 97, bias_var=bias_var, finished_frac=ff)
    gpu = run_gpu(inp, dev)
    check(oracle_mod, inp, gpu)


def test_forced_exact_path_selects_from_slots(dev, oracle_mod):
    inp = make(40, 4, 5000, 200, "bf16", seed=21, bias_var=0.1, finished_frac=0.1)
    gpu = run_gpu(inp, dev, env="exact")
    assert np.all(gpu["path"] == 2)
    check(oracle_mod, inp, gpu)


def test_repeat_is_deterministic(dev):
    inp = make(20, 4, 3000, 128, "bf16", seed=22)
    gpu = run_gpu(inp, dev, repeat=3)
    for o in gpu["all"][1:]:
        for key in ("token", "parent", "score", "finished"):
            np.testing.assert_array_equal(o[key], gpu["all"][0][key])


@pytest.mark.parametrize("k,period", [(4, 7), (16, 3)])
def test_ties_overflow_chunk_slots(dev, oracle_mod, k, period):
    # weight rows repeat every `period` tokens: each row of logits holds `period` distinct
    # values, the largest 256 / period times per 256-token sub-tile -- a later sub-tile of
    # every chunk overflows the slots left to it, so it keeps its own top k (one register
    # pass for k <= 8, k passes above); ties go to the smaller token id.  For k = 4, 2 chunks
    # x 41 slots x 4 beams stay within the fine rank's queue.
    inp = make(6, k, 1000, 64, "bf16", seed=23)
    inp["weight"] = np.ascontiguousarray(inp["weight"][np.arange(1000) % period])
    gpu = run_gpu(inp, dev)
    ora = check(oracle_mod, inp, gpu)
    if k == 4:
        assert np.all(gpu["path"] == 0)
    # identical weight rows give identical logits, so the tie order is exact
    np.testing.assert_array_equal(gpu["token"], ora["token"][:, :k])
    np.testing.assert_array_equal(gpu["parent"], ora["parent"][:, :k])


def test_ties_overflow_batch_queue(dev, oracle_mod):
    # the same ties over 20000 tokens: 40 chunks x 41 slots per beam exceed the fine rank's
    # queue, which then selects exactly from the slots
    inp = make(2, 4, 20000, 64, "bf16", seed=24)
    inp["weight"] = np.ascontiguousarray(inp["weight"][np.arange(20000) % 7])
    gpu = run_gpu(inp, dev)
    assert np.all(gpu["path"] == 3)
    ora = check(oracle_mod, inp, gpu)
    np.testing.assert_array_equal(gpu["token"], ora["token"][:, :4])
    np.testing.assert_array_equal(gpu["parent"], ora["parent"][:, :4])


def test_all_equal_logits(dev, oracle_mod):
    # every weight row equal: every logit of a row equal; scores beam - log V, tokens 0, 1, ...
    inp = make(3, 4, 2500, 64, "bf16", seed=25)
    inp["weight"] = np.ascontiguousarray(np.tile(inp["weight"][:1], (2500, 1)))
    gpu = run_gpu(inp, dev)
    check(oracle_mod, inp, gpu)
    best = np.argmax(inp["beam_scores"], axis=1)
    np.testing.assert_array_equal(gpu["parent"], np.repeat(best[:, None], 4, axis=1))
    np.testing.assert_array_equal(gpu["token"], np.tile(np.arange(4), (3, 1)))


def test_neg_inf_beams_and_masked_tokens(dev, oracle_mod):
    inp = make(6, 4, 1800, 64, "bf16", seed=26, bias_var=0.1)
    inp["beam_scores"] = inp["beam_scores"].copy()
    inp["beam_scores"][1, :] = -np.inf         # a batch whose beams are all dead
    inp["beam_scores"][2, 1] = -np.inf
    inp["bias"] = inp["bias"].copy()
    inp["bias"][::3] = -np.inf                 # a third of the vocab masked by the bias
    gpu = run_gpu(inp, dev)
    check(oracle_mod, inp, gpu)


def test_full_size_p5_sampled(dev, oracle_mod):
    w = synth.PROJ_WORKLOADS["p5"]
    inp = synth.projection_inputs(w)
    gpu = run_gpu(inp, dev)
    # both batches on each side of every 128-row block edge (32 batches of 4 beams a block),
    # so every row block and every pair of adjacent blocks is compared
    batches = [0, 1] + [e + d for e in range(32, 256, 32) for d in (-1, 0)] + [254, 255]
    sub = {"hidden": inp["hidden"][batches], "weight": inp["weight"], "bias": inp["bias"],
           "beam_scores": inp["beam_scores"][batches], "finished": None, "eos_id": inp["eos_id"],
           "dtype": inp["dtype"]}
    g = {key: gpu[key][batches] for key in ("token", "parent", "score", "finished", "lse")}
    check(oracle_mod, sub, g)
    assert np.all(gpu["path"] == 0)
    # every batch: scores sorted, parents in range, tokens in the vocab
    assert np.all(np.diff(gpu["score"], axis=1) <= 0)
    assert np.all((gpu["parent"] >= 0) & (gpu["parent"] < w.k))
    assert np.all((gpu["token"] >= 0) & (gpu["token"] < w.vocab))


def test_device_wait_timeout_is_reported(dev, oracle_mod):
    """A zero wait budget makes the projection kernel's bounded waits run out: every CTA sets
    the timeout bit, lets the copies and products it issued finish, frees its tensor memory and
    returns; the status is reported and the next call on a fresh workspace matches the oracle."""
    inp = make(40, 4, 5000, 200, "bf16", seed=23)
    H, W = inp["hidden"], inp["weight"]
    B, K, D = H.shape
    V = W.shape[0]
    th, tw = dev_tensor(H, "bf16", dev), dev_tensor(W, "bf16", dev)
    beam = torch.from_numpy(np.ascontiguousarray(inp["beam_scores"], dtype=np.float32)).to(dev)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    par, sc = torch.empty_like(tok), torch.empty((B, K), dtype=torch.float32, device=dev)
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    old = os.environ.get("LS_BEAM_DEBUG")
    os.environ["LS_BEAM_DEBUG"] = "spin=0"
    try:
        st = lsb.ls_logits_beam_step(th, tw, None, beam, None, inp["eos_id"], tok, par, sc, None, ws)
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    assert st == lsb.LS_OK
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_TIMEOUT
    gpu = run_gpu(inp, dev)
    check(oracle_mod, inp, gpu)
