"""Host-side helpers (no GPU): the seeded generators that sampled full-size parity checks rely
on, and the benchmark's record of per-kernel DRAM traffic."""
import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_hidden_states_of_a_batch_subset_equal_the_full_draw():
    # sampled parity checks regenerate only some batches' decoder states for the oracle
    w = synth.Workload("h", 9, 3, 100, "bf16", 5)
    full = synth.hidden_states(w, 40, step=2)
    part = synth.hidden_states(w, 40, step=2, batches=[0, 4, 8])
    np.testing.assert_array_equal(part, full[[0, 4, 8]])
    assert full.dtype == np.uint16 and full.shape == (9, 3, 40)
    # another step draws other states
    assert not np.array_equal(synth.hidden_states(w, 40, step=3), full)


def test_projection_scale_and_determinism():
    w = synth.Workload("p", 1, 1, 2000, "f16", 6, logit_var=2.0)
    a = synth.projection(w, 256)
    np.testing.assert_array_equal(a, synth.projection(w, 256))
    # entries ~ N(0, logit_var / dim): the variance of the draw within 5% on 512k samples
    var = float(np.var(a.astype(np.float64)))
    assert abs(var - 2.0 / 256) < 0.05 * 2.0 / 256


def test_projection_inputs_keys_and_shapes():
    w = synth.PROJ_WORKLOADS["p5"]
    small = synth.Workload("q", 3, w.k, 500, w.dtype, w.seed, logit_var=w.logit_var, extra={"dim": 64})
    inp = synth.projection_inputs(small)
    assert inp["hidden"].shape == (3, w.k, 64) and inp["weight"].shape == (500, 64)
    assert inp["beam_scores"].shape == (3, w.k) and inp["dim"] == 64 and inp["dtype"] == "bf16"


def test_recorded_traffic_lines_parse():
    import bench

    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    kernels = set()
    for ln in open(path):
        if ln.startswith("#") or not ln.strip():
            continue
        parts = ln.split()
        assert len(parts) == 4, ln
        kernel, workload, nbytes, h = parts
        assert kernel in bench.KERNEL_SOURCES and float(nbytes) > 0 and len(h) == 16
        kernels.add(kernel)
        # a line is used only while its hash matches the kernel's current sources
        got = bench.recorded_traffic(kernel, workload)
        assert got == (float(nbytes) if h == bench.source_hash(kernel) else None)
    assert kernels == set(bench.KERNEL_SOURCES)
