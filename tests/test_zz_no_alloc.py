"""ls_beam_step_noalloc, the beam step for callers that cannot allocate device memory
(e.g. plugins of a host framework that owns every byte of device memory, or serving
loops with a fixed memory budget).  It must give the same outputs as ls_beam_step with a
caller-provided workspace, call after call, since every call reuses the library's one
fixed scratch array.  This file is collected last on purpose."""
import os

import numpy as np
import pytest

import synth
from parity import SCORE_TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _outputs(B, K, dev):
    return (torch.full((B, K), -7, dtype=torch.int32, device=dev), torch.full((B, K), -7, dtype=torch.int32, device=dev),
            torch.full((B, K), float("nan"), device=dev), torch.full((B, K), 9, dtype=torch.uint8, device=dev))


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_noalloc_matches_workspace_entry_point(dev, name):
    w = synth.WORKLOADS[name]
    B, K, V = w.batch, w.k, w.vocab
    tol = SCORE_TOL[w.dtype]
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    for step in (0, 1):  # two calls in a row, different inputs
        inp = synth.step_inputs(w, step)
        lg = torch.from_numpy(inp["logits"]).to(dev)
        bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev)
        beam = torch.from_numpy(inp["beam_scores"]).to(dev)
        fin = None if inp["finished"] is None else torch.from_numpy(inp["finished"]).to(dev)
        ref = _outputs(B, K, dev)
        got = _outputs(B, K, dev)
        lsb.check(lsb.ls_beam_step(lg, bias, beam, fin, w.eos_id, *ref, ws), "ls_beam_step")
        lsb.check(lsb.ls_beam_step_noalloc(lg, bias, beam, fin, w.eos_id, *got), "ls_beam_step_noalloc")
        torch.cuda.synchronize()
        assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1]) and torch.equal(ref[3], got[3])
        np.testing.assert_allclose(got[2].cpu().numpy(), ref[2].cpu().numpy(), rtol=0, atol=tol)


def test_noalloc_rejects_shapes_beyond_its_scratch(dev):
    lg = torch.zeros((1, 1, 8), device=dev)
    tok, par, sc, fin = _outputs(1, 1, dev)
    lib = lsb.load_library()
    # 4096 x 64 beams x 100000 tokens needs far more than the fixed scratch
    assert lib.ls_beam_step_noalloc(lg.data_ptr(), 0, None, sc.data_ptr(), None, 4096, 64, 100000, 0,
                                    tok.data_ptr(), par.data_ptr(), sc.data_ptr(), None, None) == lsb.LS_ERR_UNSUPPORTED


def test_noalloc_reports_device_status(dev):
    """The fixed array's status word is readable: a zero wait budget on the two-kernel step
    (the one with bounded device waits) is reported as a timeout, and the next call, which
    clears the word, reports nothing."""
    w = synth.WORKLOADS["c2"]
    inp = synth.step_inputs(w, 0)
    B, K, V = w.batch, w.k, w.vocab
    lg = torch.from_numpy(inp["logits"]).to(dev)
    bias = torch.from_numpy(inp["bias"]).to(dev)
    beam = torch.from_numpy(inp["beam_scores"]).to(dev)
    fin = torch.from_numpy(inp["finished"]).to(dev)
    got = _outputs(B, K, dev)
    old = os.environ.get("LS_BEAM_DEBUG")
    os.environ["LS_BEAM_DEBUG"] = "spin=0,nofused"
    try:
        lsb.check(lsb.ls_beam_step_noalloc(lg, bias, beam, fin, w.eos_id, *got), "ls_beam_step_noalloc")
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    assert lsb.ls_beam_step_noalloc_status() == lsb.LS_ERR_TIMEOUT
    lsb.check(lsb.ls_beam_step_noalloc(lg, bias, beam, fin, w.eos_id, *got), "ls_beam_step_noalloc")
    assert lsb.ls_beam_step_noalloc_status() == lsb.LS_OK


def test_noalloc_allocates_nothing(dev):
    """After one warm-up call, further calls leave the device's free memory unchanged."""
    w = synth.WORKLOADS["c3"]
    inp = synth.step_inputs(w, 0)
    B, K = w.batch, w.k
    lg = torch.from_numpy(inp["logits"]).to(dev)
    beam = torch.from_numpy(inp["beam_scores"]).to(dev)
    got = _outputs(B, K, dev)
    lsb.check(lsb.ls_beam_step_noalloc(lg, None, beam, None, w.eos_id, *got), "ls_beam_step_noalloc")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(5):
        lsb.check(lsb.ls_beam_step_noalloc(lg, None, beam, None, w.eos_id, *got), "ls_beam_step_noalloc")
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert lsb.ls_beam_step_noalloc_status() == lsb.LS_OK


def test_noalloc_rejects_bad_arguments_before_touching_the_gpu(dev):
    """A call that fails the argument checks returns LS_ERR_INVALID_ARG and enqueues nothing:
    the status of the previous call is still there to be read."""
    w = synth.WORKLOADS["c2"]
    inp = synth.step_inputs(w, 0)
    B, K, V = w.batch, w.k, w.vocab
    lg = torch.from_numpy(inp["logits"]).to(dev)
    beam = torch.from_numpy(inp["beam_scores"]).to(dev)
    got = _outputs(B, K, dev)
    old = os.environ.get("LS_BEAM_DEBUG")
    os.environ["LS_BEAM_DEBUG"] = "spin=0,nofused"
    try:
        lsb.check(lsb.ls_beam_step_noalloc(lg, None, beam, None, w.eos_id, *got), "ls_beam_step_noalloc")
    finally:
        if old is None:
            os.environ.pop("LS_BEAM_DEBUG", None)
        else:
            os.environ["LS_BEAM_DEBUG"] = old
    torch.cuda.synchronize()
    # eos_id out of range: rejected on the host, the status word (a timeout) untouched
    assert lsb.ls_beam_step_noalloc(lg, None, beam, None, V, *got) == lsb.LS_ERR_INVALID_ARG
    assert lsb.ls_beam_step_noalloc_status() == lsb.LS_ERR_TIMEOUT
