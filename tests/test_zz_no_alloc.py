"""ls_beam_step_noalloc, the beam step for callers that cannot allocate device memory
(e.g. plugins of a host framework that owns every byte of device memory, or serving
loops with a fixed memory budget).  It must give the same outputs as ls_beam_step with a
caller-provided workspace, call after call, since every call reuses the library's one
fixed scratch array.  This file is collected last on purpose."""
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
