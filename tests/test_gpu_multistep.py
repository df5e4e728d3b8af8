"""64-step autoregressive workload c5 (batch 256, beam 4, vocab 40000, fp16, cache
[6, 1024, 16, 64, 64]) on the GPU against the oracle's own trajectory, then the end-of-search token sequences read
back through the parent history on the device against the oracle's backtrack.

The GPU runs every batch; the oracle runs a sample of batches, each step feeding
its own outputs (beam scores, finished flags, parents) into the next one, so no
oracle input ever comes from the GPU.  Batches are independent, so a sampled
batch is compared at every step until the oracle shows a near-tie (two scores
within 1e-4 among its first k+1 candidates), after which the two trajectories may
legitimately part; that batch is then dropped from the comparison.  At the end
the cache rows and the final token sequences of every batch still in the comparison must
match bitwise.
"""
import numpy as np
import pytest

import synth
from parity import GAP_TOL, boundary_gaps, compare_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402
from serving_ls_beam_gb300.loop import BeamSearchLoop  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def test_c5_trajectory_sampled(dev, oracle_mod):
    w = synth.WORKLOADS["c5"]
    layers, heads, max_len, head_dim = w.kv_shape
    shape = (layers, w.rows, heads, max_len, head_dim)
    steps = w.steps
    sample = [0, 37, 101, 128, 200, 255]
    caches = [torch.from_numpy(synth.kv_cache(shape, w.seed, which=i)).to(dev) for i in range(2)]
    loop = BeamSearchLoop(w.batch, w.k, w.vocab, w.eos_id, kv_shape=w.kv_shape, device=dev, caches=caches,
                          max_steps=steps)
    loop.reset(torch.from_numpy(synth.beam_scores(w, 0)).to(dev))
    # oracle state for the sampled batches
    rows = [b * w.k + j for b in sample for j in range(w.k)]
    o_cache = [synth.kv_cache_rows(shape, w.seed, rows, which=i) for i in range(2)]
    o_beam = synth.beam_scores(w, 0)[sample].copy()
    o_fin = np.zeros((len(sample), w.k), np.uint8)
    alive = set(range(len(sample)))
    cur = 0
    compared = 0
    o_tok, o_par = [], []
    for t in range(1, steps + 1):
        lg = synth.logits(w, t)
        idx = loop.step(torch.from_numpy(lg).to(dev), t)
        out = {key: v.cpu().numpy() for key, v in loop.outputs(idx).items()}
        ora = oracle_mod.beam_step(lg[sample], o_beam, finished=o_fin, eos_id=w.eos_id, m_out=w.k + 8)
        gaps = boundary_gaps(ora, w.k)
        gpu_s = {key: v[sample] for key, v in out.items()}
        for i in sorted(alive):
            compare_step(gpu_s, ora, w.k, w.dtype, finished=o_fin, eos_id=w.eos_id, batches=[i])
            if gaps[i] < GAP_TOL:
                alive.discard(i)
            else:
                assert (gpu_s["token"][i] == ora["token"][i, : w.k]).all()
                assert (gpu_s["parent"][i] == ora["parent"][i, : w.k]).all()
                compared += 1
        o_tok.append(ora["token"][:, : w.k].astype(np.int32))
        o_par.append(ora["parent"][:, : w.k].astype(np.int32))
        # the oracle's next state comes from its own outputs
        n = 1 - cur
        o_cache[n] = oracle_mod.cache_reorder(o_cache[cur], ora["parent"][:, : w.k], t, dst=o_cache[n])
        cur = n
        o_beam = ora["score"][:, : w.k].astype(np.float32)
        o_fin = ora["finished"][:, : w.k].astype(np.uint8)
    assert compared >= len(sample) * steps // 2
    final = loop.cache[loop.cur][:, rows].cpu().numpy()
    for i in sorted(alive):
        sl = slice(i * w.k, (i + 1) * w.k)
        assert np.array_equal(final[:, sl].view(np.int16), o_cache[cur][:, sl].view(np.int16))
    seq, ln = loop.finalize(steps)
    seq, ln = seq.cpu().numpy()[sample], ln.cpu().numpy()[sample]
    o_seq, o_len = oracle_mod.backtrack(np.stack(o_tok), np.stack(o_par), w.eos_id)
    for i in sorted(alive):
        np.testing.assert_array_equal(seq[i], o_seq[i])
        np.testing.assert_array_equal(ln[i], o_len[i])


def test_projection_loop_trajectory(dev, oracle_mod):
    """8 decode steps of the loop driven by decoder states (step_projection: the beam step fused into
    the output projection, bf16, hidden size 128), the cache refreshed in place, against the oracle's
    own trajectory (projection in fp64, then the naive step).  The logits carry the projection's
    rounding (parity.projection_logit_bound, B per step); a beam score carries it from every step
    before, so at step t scores agree within t (2B + 1e-5), and a batch leaves the comparison once the
    oracle's gap at the k-th place falls below twice that."""
    from parity import projection_logit_bound

    w = synth.Workload("proj_loop", 16, 4, 3000, "bf16", 31, logit_var=2.0, beam_range=(-5.0, 0.0))
    dim, steps = 128, 8
    kv = (2, 4, 8, 16)
    shape = (kv[0], w.rows, kv[1], kv[2], kv[3])
    weight = synth.projection(w, dim)
    wv = (weight.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d_weight = torch.from_numpy(weight).view(torch.int16).view(torch.bfloat16).to(dev)
    cache0 = synth.kv_cache(shape, w.seed)
    loop = BeamSearchLoop(w.batch, w.k, w.vocab, w.eos_id, kv_shape=kv, device=dev,
                          caches=[torch.from_numpy(cache0).to(dev)], max_steps=steps, inplace=True)
    beam0 = synth.beam_scores(w, 0)
    loop.reset(torch.from_numpy(beam0).to(dev))
    o_cache, o_beam = cache0.copy(), beam0.copy()
    o_fin = np.zeros((w.batch, w.k), np.uint8)
    alive = set(range(w.batch))
    compared = 0
    o_tok, o_par = [], []
    for t in range(1, steps + 1):
        hid = synth.hidden_states(w, dim, step=t)
        idx = loop.step_projection(torch.from_numpy(hid).view(torch.int16).view(torch.bfloat16).to(dev), d_weight, t)
        out = {key: v.cpu().numpy() for key, v in loop.outputs(idx).items()}
        ora = oracle_mod.logits_beam_step(hid, weight, o_beam, dtype="bf16", finished=o_fin, eos_id=w.eos_id,
                                          m_out=w.k + 8)
        hv = (hid.astype(np.uint32) << 16).view(np.float32).reshape(-1, dim).astype(np.float64)
        bound = projection_logit_bound(hv, wv).reshape(w.batch, w.k, -1).max(axis=(1, 2))
        stol = t * (2.0 * bound + 1e-5)
        gaps = boundary_gaps(ora, w.k)
        for i in sorted(alive):
            compare_step(out, ora, w.k, "bf16", finished=o_fin, eos_id=w.eos_id, batches=[i], score_tol=stol,
                         gap_tol=2.0 * stol)
            if gaps[i] < 2.0 * stol[i]:
                alive.discard(i)
            else:
                assert (out["token"][i] == ora["token"][i, : w.k]).all()
                assert (out["parent"][i] == ora["parent"][i, : w.k]).all()
                compared += 1
        o_tok.append(ora["token"][:, : w.k].astype(np.int32))
        o_par.append(ora["parent"][:, : w.k].astype(np.int32))
        o_cache = oracle_mod.cache_refresh_inplace(o_cache, ora["parent"][:, : w.k], t)
        o_beam = ora["score"][:, : w.k].astype(np.float32)
        o_fin = ora["finished"][:, : w.k].astype(np.uint8)
    assert compared >= w.batch * steps // 2
    final = loop.current_cache().cpu().numpy()
    for i in sorted(alive):
        sl = slice(i * w.k, (i + 1) * w.k)
        assert np.array_equal(final[:, sl].view(np.int16), o_cache[:, sl].view(np.int16))
    seq, ln = loop.finalize(steps)
    o_seq, o_len = oracle_mod.backtrack(np.stack(o_tok), np.stack(o_par), w.eos_id)
    seq, ln = seq.cpu().numpy(), ln.cpu().numpy()
    for i in sorted(alive):
        np.testing.assert_array_equal(seq[i], o_seq[i])
        np.testing.assert_array_equal(ln[i], o_len[i])
