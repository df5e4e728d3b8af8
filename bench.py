#!/usr/bin/env python3
"""Benchmark of the hierarchical beam-search step + cache refresh on GB300.

Default workload (c5): 64 autoregressive decode steps, batch 256, beam 4, vocab 40000,
fp16 logits N(0,2) + a per-step offset, KV cache [6, 1024, 16, 64(max_len), 64] fp16
refreshed by parent beam each step (len = step).  One benchmark "step" is the whole
64-step decode of one batch of synthetic input; `value` is decode steps per second
(every decode step covers all 256 x 4 beams), measured with all inputs resident in
HBM (5.24 GB of logits, larger than L2, so no flush is needed), the 64 steps replayed
as one CUDA graph.  `e2e` repeats it through the same C ABI with the logits copied
from pinned host memory every decode step and the step's outputs read back.

--impl reference times the oracle (single-threaded fp64 C, the naive definition) on
a bounded sample of the same workload on the host cores.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run (one process per GPU, independent batches per rank: weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "beam-search decode steps/s and logit GB/s vs GB300 HBM roofline (1 GPU)"
UNIT = "decode steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0  # one earlier cuBLAS bf16 measurement on a GB300 (burst)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sampling", action="store_true", help="skip the sampling-decoding measurement")
    ap.add_argument("--no-projection", action="store_true",
                    help="skip the measurement of the beam step fused into the output projection")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="run only the first N decode steps of the workload (for small profiling runs)")
    ap.add_argument("--kernel", choices=["beam_step", "cache_refresh_inplace", "cache_reorder", "sample"], default=None,
                    help="profiling driver: time one kernel of the loop alone on the last decode steps of the "
                         "workload (inputs of a few hundred MB to 1.6 GB) and print its per-launch figures")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank gets its own independent batches (weak scaling, no data-path collective)."""
    return base_seed + 1000003 * rank


def shard_workload(w: synth.Workload, rank: int) -> synth.Workload:
    if rank == 0:
        return w
    from dataclasses import replace

    return replace(w, seed=shard_seed(w.seed, rank))


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ peaks, clocks, profiles
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor throughput (burst: kernels timed in short graphs), TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# the sources each recorded kernel's traffic depends on: its own kernels plus the shared
# launch code and headers (a change to any of them makes the recorded counters stale)
KERNEL_SOURCES = {
    "beam_step": ("beam_fused.cu", "ls_strip.cuh"),
    "cache_refresh_inplace": ("cache_inplace.cu",),
    "cache_reorder": ("cache_reorder.cu",),
}
SHARED_SOURCES = ("api.cu", "ls_internal.h", "ls_device.cuh", "ls_dtype.cuh")


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "serving_ls_beam_gb300", "csrc")
    for fn in SHARED_SOURCES + KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None if absent or stale."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for ln in f:
                if ln.startswith("#") or not ln.strip():
                    continue
                parts = ln.split()
                if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload:
                    return float(parts[2]) if parts[3] == source_hash(kernel) else None
    except OSError:
        return None
    return None


# ------------------------------------------------------------------ oracle (CPU) timing
def time_oracle_sample(w: synth.Workload, batches, steps_list, with_cache: bool):
    """Run the oracle on `batches` for the given decode steps (own trajectory); returns (seconds, batch_steps)."""
    import oracle

    oracle.build()
    k = w.k
    o_beam = synth.beam_scores(w, 0)[batches].copy()
    o_fin = np.zeros((len(batches), k), np.uint8)
    cache = None
    if with_cache and w.kv_shape is not None:
        layers, heads, max_len, head_dim = w.kv_shape
        shape = (layers, w.rows, heads, max_len, head_dim)
        rows = [b * k + j for b in batches for j in range(k)]
        cache = [synth.kv_cache_rows(shape, w.seed, rows, which=i) for i in range(2)]
    inputs = [synth.logits(w, t, batches) for t in steps_list]
    cur = 0
    t0 = time.perf_counter()
    for lg, t in zip(inputs, steps_list):
        r = oracle.beam_step(lg, o_beam, bias=synth.bias(w), finished=o_fin, eos_id=w.eos_id)
        if cache is not None:
            cache[1 - cur] = oracle.cache_reorder(cache[cur], r["parent"], t, dst=cache[1 - cur])
            cur = 1 - cur
        o_beam = r["score"].astype(np.float32)
        o_fin = r["finished"]
    dt = time.perf_counter() - t0
    return dt, len(batches) * len(steps_list)


def _oracle_worker(name: str, batches, steps):
    """One process of the all-core baseline: the unmodified oracle on its own batches."""
    return time_oracle_sample(synth.WORKLOADS[name], batches, steps, True)


def cpu_baseline(w: synth.Workload, target_s: float = 12.0, all_cores_s: float = 8.0):
    """The oracle (single-threaded fp64 C) on the host: on one core, and batch-parallel over
    every host core (one process per core, each running the same oracle on its own batches)."""
    import concurrent.futures as cf
    import multiprocessing as mp

    # calibrate on one batch-step, then size the sample to roughly target_s seconds
    dt1, n1 = time_oracle_sample(w, [0], [1], True)
    per = dt1 / n1
    n = max(2, int(target_s / max(per, 1e-4)))
    steps = min(w.steps, max(1, n // 8))
    nb = max(1, min(w.batch, n // steps))
    batches = list(range(nb))
    dt, bs = time_oracle_sample(w, batches, list(range(1, steps + 1)), True)
    per = dt / bs
    value = 1.0 / (per * w.batch)
    host_cores = os.cpu_count() or 1
    line = {"value": value, "unit": UNIT, "cores": 1, "host_cores": host_cores, "kind": "oracle",
            "sample": f"{nb} batches x {steps} decode steps of {w.name} (beam step + cache refresh), single thread; "
                      f"{per * 1e3:.1f} ms per batch-step, scaled to all {w.batch} batches (extrapolated)"}
    # batch-parallel on every host core: processes started with spawn (this process holds a
    # CUDA context), each sample sized to about all_cores_s seconds
    try:
        psteps = max(1, min(w.steps, int(all_cores_s / max(per, 1e-4))))
        nbp = min(w.batch, host_cores)
        ctx = mp.get_context("spawn")
        with cf.ProcessPoolExecutor(max_workers=nbp, mp_context=ctx) as ex:
            list(ex.map(_oracle_worker, [w.name] * nbp, [[b] for b in range(nbp)], [[1]] * nbp))  # warm-up
            t0 = time.perf_counter()
            res = list(ex.map(_oracle_worker, [w.name] * nbp, [[b] for b in range(nbp)],
                              [list(range(1, psteps + 1))] * nbp))
            wall = time.perf_counter() - t0
        done = sum(r[1] for r in res)
        line["all_cores"] = {"value": done / wall / w.batch, "unit": UNIT, "cores": nbp,
                             "sample": f"{nbp} processes x 1 batch x {psteps} decode steps, wall clock "
                                       f"{wall:.1f} s, scaled to all {w.batch} batches (extrapolated)"}
    except Exception as e:  # a baseline, not the measurement: report why it is missing
        line["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return line


# ------------------------------------------------------------------ GPU arm
def workload_config(w: synth.Workload, T: int, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": f"{w.name}: batch {w.batch}, beam {w.k}, vocab {w.vocab}, {w.dtype} logits, "
                        f"{T} decode step(s)" + (f", KV cache {[w.kv_shape[0], w.rows, *w.kv_shape[1:]]} fp16 "
                                                 f"refreshed by parent (len = step), in place" if w.kv_shape else ""),
            "batch": w.batch, "beam": w.k, "vocab": w.vocab, "logit_dtype": w.dtype, "decode_steps_per_step": T,
            "l2": f"inputs larger than L2: {T * w.rows * w.vocab * (2 if w.dtype != 'f32' else 4) / 1e9:.2f} GB of "
                  f"logits per benchmark step",
            "graph": f"one CUDA graph of the {T}-step loop and the end-of-search backtrack",
            "cache_refresh": "in place, copy on change (out-of-place figures under cache_refresh_out_of_place)",
            "parallelism": f"replicas x{world} (independent batches)"}


def moved_rows(par: np.ndarray, K: int) -> np.ndarray:
    """Rows the in-place refresh moves per step, from parents [steps, batch, k]: each changed beam
    is written once and each parent a changed beam needs is read once per batch."""
    steps, B = par.shape[:2]
    changed = par != np.arange(K)[None, None, :]
    needed = np.zeros((steps, B, K), bool)
    for j in range(K):
        needed[np.arange(steps)[:, None], np.arange(B)[None, :], par[:, :, j]] |= changed[:, :, j]
    return changed.sum(axis=(1, 2)) + needed.sum(axis=(1, 2))


def bench_kernel(args, w: synth.Workload):
    """Profiling driver: one kernel of the decode loop, alone, at the workload's last three decode
    steps (with --decode-steps N, steps N-2..N).  It walks the search's own trajectory with one step's logits on the device at a time
    (beam state carried from step to step as in the benchmark loop, so the parents are the loop's),
    then launches the kernel on those three steps: the beam step on their logits (3 x 82 MB at c5),
    the cache refresh at len = step on one seeded cache (in place, 805 MB) or two (out of place,
    1.6 GB).  Each of --warmup + --steps rounds launches the kernel once per step; the JSON line gives
    each step's event-timed microseconds and algorithmic bytes (one round is 3 launches, so
    `ncu -k <kernel> -s <launches before> -c 3` captures the three full-size launches)."""
    import torch

    import serving_ls_beam_gb300 as lsb
    from serving_ls_beam_gb300 import _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    _build.build()
    lsb.load_library()
    if args.kernel == "sample":
        return bench_kernel_sample(args, dev)
    B, K, V = w.batch, w.k, w.vocab
    es = 2 if w.dtype in ("f16", "bf16") else 4
    multi = w.steps > 1
    last = (min(w.steps, args.decode_steps) if args.decode_steps > 0 else w.steps) if multi else 0
    steps = list(range(max(1 if multi else 0, last - 2), last + 1))
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    bias_np = synth.bias(w)
    bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    fin_np = synth.finished(w)
    scores = [torch.from_numpy(synth.beam_scores(w, 0)).to(dev), torch.empty((B, K), dtype=torch.float32, device=dev)]
    fins = [torch.zeros((B, K), dtype=torch.uint8, device=dev) if fin_np is None
            else torch.from_numpy(fin_np).to(dev), torch.empty((B, K), dtype=torch.uint8, device=dev)]
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    ins, parents = [], []
    cur = 0
    for t in (range(1, last + 1) if multi else [0]):
        lg = torch.from_numpy(synth.logits(w, t)).to(dev)
        par = torch.empty((B, K), dtype=torch.int32, device=dev)
        if t in steps:
            ins.append((lg, scores[cur].clone(), fins[cur].clone()))
        lsb.check(lsb.ls_beam_step(lg, bias, scores[cur], fins[cur], w.eos_id, tok, par, scores[1 - cur],
                                   fins[1 - cur], ws), "ls_beam_step")
        if t in steps:
            parents.append(par)
        cur = 1 - cur
    torch.cuda.synchronize()
    lsb.check(lsb.ls_read_status(ws), "device status")
    sc = torch.empty((B, K), dtype=torch.float32, device=dev)
    fo = torch.empty((B, K), dtype=torch.uint8, device=dev)
    if args.kernel == "beam_step":
        nbytes = [(w.rows - int(f.sum())) * V * es + (V * 4 if bias is not None else 0) + w.rows * 13
                  for (_, _, f) in ins]

        def launch(i):
            lg, beam, fin = ins[i]
            return lsb.ls_beam_step(lg, bias, beam, fin, w.eos_id, tok, parents[i], sc, fo, ws)
    else:
        ins.clear()
        if w.kv_shape is None:
            raise SystemExit(f"bench.py: workload {w.name} has no cache")
        layers, heads, max_len, head_dim = w.kv_shape
        shape = (layers, w.rows, heads, max_len, head_dim)
        lens = [t if multi else max_len for t in steps]
        slabs = [layers * heads * n * head_dim * 2 for n in lens]
        caches = [torch.from_numpy(synth.kv_cache(shape, w.seed, which=i)).to(dev)
                  for i in range(1 if args.kernel == "cache_refresh_inplace" else 2)]
        if args.kernel == "cache_refresh_inplace":
            par_np = np.stack([p.cpu().numpy() for p in parents])
            nbytes = [int(m) * sl for m, sl in zip(moved_rows(par_np, K), slabs)]

            def launch(i):
                return lsb.ls_cache_refresh_inplace(caches[0], parents[i], lens[i], ws)
        else:
            nbytes = [2 * w.rows * sl for sl in slabs]

            def launch(i):
                return lsb.ls_cache_reorder(caches[i % 2], caches[1 - i % 2], parents[i], lens[i])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in steps]
    us = [[] for _ in steps]
    for rnd in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        torch.cuda._sleep(1 << 20)  # ~0.5 ms of GPU time, so every launch below is queued before it starts
        for i in range(len(steps)):
            ev[i][0].record()
            lsb.check(launch(i), args.kernel)
            ev[i][1].record()
        torch.cuda.synchronize()
        if rnd >= args.warmup:
            for i in range(len(steps)):
                us[i].append(ev[i][0].elapsed_time(ev[i][1]) * 1e3)
    lsb.check(lsb.ls_read_status(ws), "device status")
    peak, peak_src = hbm_peak()
    launches = []
    for i, t in enumerate(steps):
        u = statistics.median(us[i]) if us[i] else None
        launches.append({"decode_step": t, "us": u, "algorithmic_bytes": nbytes[i],
                         "gbs": None if not u else nbytes[i] / (u * 1e-6) / 1e9})
    return {"kernel": args.kernel, "workload": w.name, "warmup": args.warmup, "steps": args.steps,
            "peak": peak, "peak_source": peak_src, "launches": launches,
            "note": "each launch timed with CUDA events around it, the three launches of a round queued "
                    "back to back behind a GPU sleep (no host launch time inside); no L2 flush between "
                    "launches, each launch reads inputs larger than L2 or those of the previous step"}


def bench_kernel_sample(args, dev):
    """Profiling driver for sampling decoding: ls_sample on three of workload s1's logit sets
    (3 x 82 MB), each of --warmup + --steps rounds launching it once per set."""
    import torch

    import serving_ls_beam_gb300 as lsb

    w = synth.SAMPLE_WORKLOADS["s1"]
    ins = [synth.sample_inputs(w, step=i) for i in range(3)]
    rows, vocab, top_k, top_p = w.batch, w.vocab, ins[0]["top_k"], ins[0]["top_p"]
    lg = [torch.from_numpy(x["logits"]).to(dev) for x in ins]
    u = [torch.from_numpy(x["u"]).to(dev) for x in ins]
    tok = torch.empty(rows, dtype=torch.int32, device=dev)
    lp = torch.empty(rows, dtype=torch.float32, device=dev)
    ws = torch.empty(lsb.ls_sample_workspace_size(rows, top_k, vocab), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    nbytes = rows * vocab * 2
    us = [[] for _ in ins]
    for rnd in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        torch.cuda._sleep(1 << 20)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in ins]
        for i in range(len(ins)):
            ev[i][0].record()
            lsb.check(lsb.ls_sample(lg[i], None, u[i], top_k, top_p, tok, lp, ws), "ls_sample")
            ev[i][1].record()
        torch.cuda.synchronize()
        if rnd >= args.warmup:
            for i in range(len(ins)):
                us[i].append(ev[i][0].elapsed_time(ev[i][1]) * 1e3)
    lsb.check(lsb.ls_read_status(ws), "device status")
    peak, peak_src = hbm_peak()
    launches = []
    for i in range(len(ins)):
        t = statistics.median(us[i]) if us[i] else None
        launches.append({"call": i, "us": t, "algorithmic_bytes": nbytes,
                         "gbs": None if not t else nbytes / (t * 1e-6) / 1e9})
    return {"kernel": "sample", "workload": "s1", "warmup": args.warmup, "steps": args.steps, "peak": peak,
            "peak_source": peak_src, "launches": launches,
            "note": "each call timed with CUDA events around it, the three calls of a round queued back to back "
                    "behind a GPU sleep"}


def beam_step_kernels(w: synth.Workload, dev) -> int:
    """Kernels one ls_beam_step launches on this workload: 1 where the plan takes the
    one-kernel step K3 (k <= 8, every strip's stages within 32, two batches per SM at most),
    else 2 (K1 + K2).  Mirrors the plan in csrc/api.cu."""
    import torch

    if os.environ.get("LS_BEAM_DEBUG"):
        flags = os.environ["LS_BEAM_DEBUG"].split(",")
        if "nofused" in flags:
            return 2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    es = 2 if w.dtype in ("f16", "bf16") else 4
    vpl = 4 if (es == 4 or w.bias_var) else 8
    parts = max(0, 8 // w.k)
    if w.k > 8 or parts < 1:
        return 2
    ns = ((15 + w.vocab * es + 15) // 16 + 32 * vpl - 1) // (32 * vpl)
    return 1 if (ns + parts - 1) // parts <= 32 and 2 * w.batch >= sms else 2


def bench_gpu(args, w: synth.Workload, world: int, rank: int, local: int):
    import torch

    import serving_ls_beam_gb300 as lsb
    from serving_ls_beam_gb300 import _build
    from serving_ls_beam_gb300.loop import BeamSearchLoop

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    lsb.load_library()
    wr = shard_workload(w, rank)
    T = min(wr.steps, args.decode_steps) if args.decode_steps > 0 else wr.steps
    B, K, V = wr.batch, wr.k, wr.vocab
    es = 2 if wr.dtype in ("f16", "bf16") else 4
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[wr.dtype]

    # ---- inputs, resident in HBM
    t0 = time.time()
    host_logits = np.empty((T, B, K, V), np.float16 if wr.dtype == "f16" else np.float32)
    for t in range(T):
        host_logits[t] = synth.logits(wr, t + 1 if wr.steps > 1 else 0)
    d_logits = torch.from_numpy(host_logits).to(dev)
    bias_np = synth.bias(wr)
    d_bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    beam0 = torch.from_numpy(synth.beam_scores(wr, 0)).to(dev)
    fin_np = synth.finished(wr)
    fin0 = None if fin_np is None else torch.from_numpy(fin_np).to(dev)
    caches = None
    if wr.kv_shape is not None:
        layers, heads, max_len, head_dim = wr.kv_shape
        shape = (layers, wr.rows, heads, max_len, head_dim)
        caches = [torch.from_numpy(synth.kv_cache(shape, wr.seed, which=i)).to(dev) for i in range(2)]
    # the headline loop refreshes the cache in place (copy on change); the out-of-place
    # (ping-pong) refresh of the same search is timed too and reported beside it
    loop = BeamSearchLoop(B, K, V, wr.eos_id, kv_shape=wr.kv_shape, device=dev, caches=caches, max_steps=T,
                          inplace=True)
    loop_oop = None
    if caches is not None:
        loop_oop = BeamSearchLoop(B, K, V, wr.eos_id, kv_shape=wr.kv_shape, device=dev, caches=caches, max_steps=T)
    setup_s = time.time() - t0

    def lens(t):  # cache positions refreshed at decode step t (1-based)
        return t if wr.steps > 1 else (wr.kv_shape[2] if wr.kv_shape else 0)

    stream = torch.cuda.Stream(device=dev)
    try:  # events inside a captured graph must be "external" record nodes to be timed
        ev_k = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)] for _ in range(T + 1)]
        graph_events = True
    except TypeError:
        ev_k = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(T + 1)]
        graph_events = False

    def run_all(lp, instrument: bool):
        lp.reset(beam0, fin0)
        for t in range(T):
            if instrument:
                ev_k[t][0].record()
            s, n = lp.cur, 1 - lp.cur
            tok, par = lp.token_out(t + 1), lp.parent_out(t + 1)
            lsb.check(lsb.ls_beam_step(d_logits[t], d_bias, lp.scores[s], lp.finished[s], wr.eos_id,
                                       tok, par, lp.scores[n], lp.finished[n], lp.workspace), "ls_beam_step")
            if instrument:
                ev_k[t][1].record()
            if lp.cache is not None:
                if lp.inplace:
                    lsb.check(lsb.ls_cache_refresh_inplace(lp.cache[0], par, lens(t + 1), lp.workspace),
                              "ls_cache_refresh_inplace")
                else:
                    lsb.check(lsb.ls_cache_reorder(lp.cache[s], lp.cache[n], par, lens(t + 1)), "ls_cache_reorder")
            if instrument:
                ev_k[t][2].record()
            lp.cur = n
        # end of the search: every final beam's token sequence from the parent history
        if instrument:
            ev_k[T][0].record()
        lp.finalize(T)
        if instrument:
            ev_k[T][1].record()

    def capture(lp):
        # warm the library's per-device setup outside capture, then capture both graphs
        with torch.cuda.stream(stream):
            run_all(lp, False)
        torch.cuda.synchronize()
        lsb.check(lsb.ls_read_status(lp.workspace, stream), "device status")
        gp, gi = torch.cuda.CUDAGraph(), None
        with torch.cuda.graph(gp, stream=stream):
            run_all(lp, False)
        if graph_events:
            gi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gi, stream=stream):
                run_all(lp, True)
        torch.cuda.synchronize()
        return gp, gi

    def time_graphs(lp, gp, gi):
        """ms for args.steps replays of gp, then per-kernel ms per search from gi (K1+K2, K4, backtrack)."""
        for _ in range(args.warmup):
            gp.replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(args.steps):
                gp.replay()
            e1.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = e0.elapsed_time(e1)
        k1, k4, bt = 0.0, 0.0, 0.0
        reps = max(1, min(args.steps, 3))
        with torch.cuda.stream(stream):
            for _ in range(reps):
                if gi is not None:
                    gi.replay()
                else:
                    run_all(lp, True)
                torch.cuda.synchronize()
                for t in range(T):
                    k1 += ev_k[t][0].elapsed_time(ev_k[t][1])
                    if lp.cache is not None:
                        k4 += ev_k[t][1].elapsed_time(ev_k[t][2])
                bt += ev_k[T][0].elapsed_time(ev_k[T][1])
        lsb.check(lsb.ls_read_status(lp.workspace, stream), "device status")
        return ms, k1 / reps, k4 / reps, bt / reps

    def time_alone(lp):
        """us per launch of the beam step and of the cache refresh, each timed in a graph of the
        search's launches of that kernel alone (chained with programmatic dependent launch, no
        events between them; the refreshes use the parents the loop recorded)."""
        def beams():
            lp.reset(beam0, fin0)
            for t in range(T):
                s, n = lp.cur, 1 - lp.cur
                lsb.check(lsb.ls_beam_step(d_logits[t], d_bias, lp.scores[s], lp.finished[s], wr.eos_id,
                                           lp.token_out(t + 1), lp.parent_out(t + 1), lp.scores[n], lp.finished[n],
                                           lp.workspace), "ls_beam_step")
                lp.cur = n

        def refreshes():
            for t in range(T):
                par = lp.parent_out(t + 1)
                if lp.inplace:
                    lsb.check(lsb.ls_cache_refresh_inplace(lp.cache[0], par, lens(t + 1), lp.workspace),
                              "ls_cache_refresh_inplace")
                else:
                    lsb.check(lsb.ls_cache_reorder(lp.cache[t % 2], lp.cache[1 - t % 2], par, lens(t + 1)),
                              "ls_cache_reorder")

        out = {}
        for name, fn in (("beam_step", beams), ("refresh", refreshes)):
            if name == "refresh" and lp.cache is None:
                continue
            with torch.cuda.stream(stream):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            torch.cuda.synchronize()
            ts = []
            with torch.cuda.stream(stream):
                for r in range(4):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    g.replay()
                    b.record()
                    torch.cuda.synchronize()
                    if r > 0:
                        ts.append(a.elapsed_time(b) * 1e3 / T)
            del g
            out[name] = statistics.median(ts)
        lsb.check(lsb.ls_read_status(lp.workspace, stream), "device status")
        return out

    # kernels per decode step: the beam step (K3 alone, or K1 + K2) and the cache refresh; plus the backtrack
    launches_per_step = T * (beam_step_kernels(wr, dev) + (1 if loop.cache is not None else 0)) + 1
    g_plain, g_inst = capture(loop)
    with ClockSampler(local) as clk:
        ms_plain, k1_ms, k4_ms, bt_ms = time_graphs(loop, g_plain, g_inst)
        parents_run = loop.parent_hist.cpu().numpy() if loop.cache is not None else None
        alone = time_alone(loop)
        oop = None
        if loop_oop is not None:
            del g_plain, g_inst
            go_plain, go_inst = capture(loop_oop)
            oop = time_graphs(loop_oop, go_plain, go_inst)
            del go_plain, go_inst
    ms_total = max_over_ranks(ms_plain, world, dev)
    ms_per_step = ms_total / args.steps
    decode_steps = T * args.steps * world
    value = decode_steps / (ms_total / 1e3)

    # ---- algorithmic bytes
    fin_rows = 0 if fin_np is None else int(fin_np.sum())
    logit_bytes_launch = (wr.rows - fin_rows) * V * es + (V * 4 if bias_np is not None else 0) + wr.rows * 13
    k1_bytes = logit_bytes_launch * T
    k4_bytes, k4_dense_bytes = 0, 0
    if loop.cache is not None:
        layers, heads, max_len, head_dim = wr.kv_shape
        # in place: each batch reads the slabs of the parents its changed beams need and writes
        # the changed beams (exact, from the run's parents); out of place: every row both ways
        moved = moved_rows(parents_run.reshape(T, B, K), K)
        for t in range(1, T + 1):
            slab = layers * heads * lens(t) * head_dim * 2
            k4_bytes += int(moved[t - 1]) * slab
            k4_dense_bytes += 2 * wr.rows * slab
    peak, peak_src = hbm_peak()
    k1_gbs = k1_bytes / (k1_ms / 1e3) / 1e9
    def alone_fields(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us_per_launch_alone": us, "achieved_alone": gbs, "frac_alone": gbs / peak}

    kern = {"beam_step": {"bound": "hbm", "achieved": k1_gbs, "peak": peak, "unit": "GB/s", "frac": k1_gbs / peak,
                          "traffic": recorded_traffic("beam_step", wr.name),
                          "us_per_launch": k1_ms * 1e3 / T,
                          "algorithmic_bytes_per_launch": k1_bytes / T,
                          **alone_fields(alone["beam_step"], k1_bytes / T)}}
    oop_line = None
    if loop.cache is not None:
        k4_gbs = k4_bytes / (k4_ms / 1e3) / 1e9
        kern["cache_refresh_inplace"] = {
            "bound": "hbm", "achieved": k4_gbs, "peak": peak, "unit": "GB/s", "frac": k4_gbs / peak,
            "traffic": recorded_traffic("cache_refresh_inplace", wr.name), "us_per_launch": k4_ms * 1e3 / T,
            "algorithmic_bytes_per_launch": k4_bytes / T,
            "note": "copy on change: bytes of the parents read and the beams written, from the run's parents; "
                    f"{k4_dense_bytes / T:.0f} B per launch if every row were moved",
            **alone_fields(alone["refresh"], k4_bytes / T)}
        if oop is not None:
            o_ms, o_k1, o_k4, o_bt = oop
            o_ms = max_over_ranks(o_ms, world, dev)
            o_gbs = k4_dense_bytes / (o_k4 / 1e3) / 1e9
            oop_line = {"value": T * args.steps * world / (o_ms / 1e3), "unit": UNIT, "ms_per_step": o_ms / args.steps,
                        "cache_reorder": {"bound": "hbm", "achieved": o_gbs, "peak": peak, "unit": "GB/s",
                                          "frac": o_gbs / peak,
                                          "traffic": recorded_traffic("cache_reorder", wr.name),
                                          "us_per_launch": o_k4 * 1e3 / T,
                                          "algorithmic_bytes_per_launch": k4_dense_bytes / T,
                                          "note": "algorithmic bytes count every row both ways; a parent "
                                                  "shared by several beams is read again from L2, so frac "
                                                  "may exceed 1 (traffic is the DRAM bytes moved)"},
                        "beam_step_us_per_launch": o_k1 * 1e3 / T,
                        "note": "the same search with the out-of-place (ping-pong) cache refresh"}
    bt_bytes = 2 * T * B * K * 4 + B * K * (T + 1) * 4  # history read, sequences and lengths written
    bt_gbs = bt_bytes / (bt_ms / 1e3) / 1e9 if bt_ms > 0 else 0.0
    kern["backtrack"] = {"bound": "latency", "achieved": bt_gbs, "peak": peak, "unit": "GB/s", "frac": bt_gbs / peak,
                         "traffic": None, "us_per_launch": bt_ms * 1e3, "algorithmic_bytes_per_launch": bt_bytes,
                         "launches_per_step": 1}
    dominant = max((n for n in kern if n != "backtrack"), key=lambda n: kern[n]["us_per_launch"])
    roof = {key: kern[dominant][key] for key in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = dominant
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback"
    step_gbs = (k1_bytes + k4_bytes) / (ms_plain / args.steps / 1e3) / 1e9

    # ---- candidate statistics of the last decode step of the timed search (read after timing)
    _, _, ncand, path = lsb.ls_read_row_stats(loop.workspace, B, K, V)
    live = ncand >= 0
    cand = {"per_beam_mean": float(ncand[live].mean()) if live.any() else None,
            "per_batch_mean": float(np.where(live, ncand, 0).sum(axis=1).mean()),
            "exact_path_batches": int((path != 0).sum()), "batches": int(B),
            "note": "survivors of each beam's R-top-k at the last decode step (the queue the fine rank sorts)"}

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(args, wr, loop, host_logits, bias_np, beam0, fin0, lens, dev, world)

    sampling = None
    if not args.no_sampling:
        sampling = bench_sampling(dev, peak)

    projection = None
    if not args.no_projection:
        projection = bench_projection(dev)

    clocks = clk.summary()
    cfg = workload_config(wr, T, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wr.dtype, "data": "synthetic (seeded generators, workload recipe in synth/)", "config": cfg,
        "logit_gbs": k1_gbs, "step_gbs": step_gbs, "step_roofline_frac": step_gbs / peak,
        "roofline": roof, "roofline_kernels": kern,
        "roofline_kernels_note": "us_per_launch and frac: a second, event-instrumented graph of the same search "
                                 "(an event between every two kernels, so each kernel's time includes a launch "
                                 "gap and its frac reads low); us_per_launch_alone and frac_alone: a graph of the "
                                 "search's launches of that kernel alone, chained with programmatic dependent "
                                 "launch, events only around the graph; value comes from the plain graph",
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "e2e": e2e, "sampling": sampling, "projection_step": projection,
        "cache_refresh_out_of_place": oop_line,
        "candidates": cand,
        "setup_s": round(setup_s, 1),
    }
    return line


def bench_sampling(dev, peak, calls: int = 16):
    """Sampling decoding (ls_sample: the one-kernel sampler for top_k <= 8, else K1 then K5) on
    workload s1: one CUDA graph of `calls` calls over as many distinct logit sets (1.3 GB in all,
    larger than L2), timed with CUDA events."""
    import torch

    import serving_ls_beam_gb300 as lsb

    w = synth.SAMPLE_WORKLOADS["s1"]
    ins = [synth.sample_inputs(w, step=i) for i in range(calls)]
    rows, vocab, top_k, top_p = w.batch, w.vocab, ins[0]["top_k"], ins[0]["top_p"]
    lg = [torch.from_numpy(d["logits"]).to(dev) for d in ins]
    u = [torch.from_numpy(d["u"]).to(dev) for d in ins]
    tok = torch.empty((calls, rows), dtype=torch.int32, device=dev)
    lp = torch.empty((calls, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(lsb.ls_sample_workspace_size(rows, top_k, vocab), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    stream = torch.cuda.Stream(device=dev)

    def run():
        for i in range(calls):
            lsb.check(lsb.ls_sample(lg[i], None, u[i], top_k, top_p, tok[i], lp[i], ws), "ls_sample")

    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    lsb.check(lsb.ls_read_status(ws), "device status")
    us = e0.elapsed_time(e1) * 1e3 / (reps * calls)
    nbytes = rows * vocab * 2 + rows * 12  # logits once; uniform in, token and log-probability out
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"s1: {rows} rows, vocab {vocab}, f16 logits N(0,2), top_k {top_k}, top_p {top_p}",
            "us_per_call": us, "rows_per_s": rows / (us * 1e-6), "achieved": gbs, "peak": peak, "unit": "GB/s",
            "frac": gbs / peak, "algorithmic_bytes_per_call": nbytes,
            # the one-kernel sampler for top_k <= 8 with rows enough to fill the GPU, else K1 then K5
            "launches_per_call": 1 if top_k <= 8 and 2 * ((rows + 3) // 4) >= torch.cuda.get_device_properties(
                dev).multi_processor_count else 2,
            "l2": f"{calls} distinct logit sets per graph ({calls * rows * vocab * 2 / 1e9:.2f} GB)"}


def bench_projection(dev, calls: int = 12, copies: int = 3):
    """The beam step fused into the output projection (ls_logits_beam_step: K0 then K2) on workload p5:
    one CUDA graph of `calls` calls over `copies` copies of the projection (82 MB each, 246 MB in all,
    larger than L2) and `calls` sets of decoder states, timed with CUDA events.  For comparison the same
    step unfused: a cuBLAS bf16 GEMM (torch.mm) that writes bf16 logits, then ls_beam_step on them."""
    import torch

    import serving_ls_beam_gb300 as lsb

    w = synth.PROJ_WORKLOADS["p5"]
    dim = int(w.extra["dim"])
    B, K, V, rows = w.batch, w.k, w.vocab, w.rows
    tpeak, tsrc = tensor_peak()

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.int16).view(torch.bfloat16).to(dev)

    w0 = bf16(synth.projection(w, dim))
    wts = [w0] + [w0.clone() for _ in range(copies - 1)]
    hs = [bf16(synth.hidden_states(w, dim, step=i)) for i in range(calls)]
    beam = torch.from_numpy(synth.beam_scores(w)).to(dev)
    tok = torch.empty((calls, B, K), dtype=torch.int32, device=dev)
    par = torch.empty_like(tok)
    sc = torch.empty((calls, B, K), dtype=torch.float32, device=dev)
    of = torch.empty((calls, B, K), dtype=torch.uint8, device=dev)
    ws = torch.empty(lsb.ls_beam_step_workspace_size(B, K, V), dtype=torch.uint8, device=dev)
    lsb.check(lsb.ls_workspace_init(ws))
    logits = torch.empty((rows, V), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def fused():
        for i in range(calls):
            lsb.check(lsb.ls_logits_beam_step(hs[i], wts[i % copies], None, beam, None, w.eos_id, tok[i], par[i],
                                              sc[i], of[i], ws), "ls_logits_beam_step")

    def unfused():
        for i in range(calls):
            torch.mm(hs[i].view(rows, dim), wts[i % copies].t(), out=logits)
            lsb.check(lsb.ls_beam_step(logits.view(B, K, V), None, beam, None, w.eos_id, tok[i], par[i], sc[i], of[i],
                                       ws), "ls_beam_step")

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        torch.cuda.synchronize()
        lsb.check(lsb.ls_read_status(ws), "device status")
        return e0.elapsed_time(e1) * 1e3 / (reps * calls)

    us = timed(fused)
    fused_tok = tok.clone()
    us_unfused = timed(unfused)
    flops = 2.0 * rows * V * dim
    tf = flops / (us * 1e-6) / 1e12
    # the two paths select from logits that differ only by rounding (f32 accumulators vs bf16 logits)
    agree = float((fused_tok == tok).float().mean().item())
    return {"workload": f"p5: batch {B}, beam {K}, vocab {V}, hidden {dim}, bf16 decoder states and projection",
            "bound": "tensor", "us_per_call": us, "achieved": tf, "peak": tpeak, "unit": "TFLOP/s",
            "frac": tf / tpeak, "peak_source": f"{tsrc} (MEASURED_PEAKS.json bf16_tflops)" if tsrc == "measured"
            else "fallback", "flops_per_call": flops, "launches_per_call": 2,
            "decode_steps_per_s": 1e6 / us, "unfused_us_per_call": us_unfused,
            "unfused": "cuBLAS bf16 GEMM writing bf16 logits (torch.mm) + ls_beam_step on them",
            "token_agreement_with_unfused": agree,
            "note": "the unfused arm selects from bf16-rounded logits, the fused one from f32 accumulators, so "
                    "near-ties can resolve differently; the fused path is checked against the fp64 oracle in "
                    "the GPU tests",
            "l2": f"{copies} projection copies ({copies * V * dim * 2 / 1e6:.0f} MB) and {calls} decoder-state sets "
                  "per graph"}


def bench_e2e(args, wr, loop, host_logits, bias_np, beam0, fin0, lens, dev, world):
    """Logits copied from pinned host memory each decode step (copy stream, NBUF device buffers),
    outputs read back each step; the all-finished stop is checked LAG steps behind, so the copy of
    a step's logits overlaps the compute of the steps before it."""
    import torch

    import serving_ls_beam_gb300 as lsb

    T = host_logits.shape[0]
    pinned = torch.from_numpy(host_logits).pin_memory()
    NBUF, LAG = 3, 2
    bufs = [torch.empty(pinned.shape[1:], dtype=pinned.dtype, device=dev) for _ in range(NBUF)]
    d_bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    out_host = {key: torch.empty((T,) + tuple(loop.token[0].shape), dtype=dt).pin_memory()
                for key, dt in (("token", torch.int32), ("parent", torch.int32), ("score", torch.float32),
                                ("finished", torch.uint8))}
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(NBUF)]
    buf_free = [torch.cuda.Event() for _ in range(NBUF)]
    d2h_done = [torch.cuda.Event() for _ in range(T)]
    seq_host = torch.empty(wr.batch * wr.k * T, dtype=torch.int32).pin_memory()
    len_host = torch.empty((wr.batch, wr.k), dtype=torch.int32).pin_memory()

    def one_run():
        loop.reset(beam0, fin0)
        stop = T
        for t in range(T):
            i = t % NBUF
            with torch.cuda.stream(copy):
                if t >= NBUF:
                    copy.wait_event(buf_free[i])
                bufs[i].copy_(pinned[t], non_blocking=True)
                h2d_done[i].record(copy)
            comp.wait_event(h2d_done[i])
            idx = loop.step(bufs[i], lens(t + 1), bias=d_bias)
            buf_free[i].record(comp)
            o = loop.outputs(idx)
            for key in out_host:
                out_host[key][t].copy_(o[key], non_blocking=True)
            d2h_done[t].record(comp)
            if t >= LAG:
                d2h_done[t - LAG].synchronize()
                if bool(out_host["finished"][t - LAG].all()):
                    stop = t + 1  # the steps already enqueued have run
                    break
        # the search's result: every final beam's token sequence, read back to the host
        seq, ln = loop.finalize(stop)
        seq_host[: seq.numel()].copy_(seq.reshape(-1), non_blocking=True)
        len_host.copy_(ln, non_blocking=True)
        torch.cuda.synchronize()
        return stop

    for _ in range(max(1, args.warmup)):
        one_run()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    steps_done = 0
    for _ in range(args.e2e_steps):
        steps_done += one_run()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    dt = max_over_ranks(dt, world, dev)
    lsb.check(lsb.ls_read_status(loop.workspace), "device status")
    h2d = int(pinned[0].numel() * pinned.element_size())
    d2h = int(sum(v[0].numel() * v.element_size() for v in out_host.values()))
    d2h_final = (wr.batch * wr.k * T + wr.batch * wr.k) * 4
    return {"value": steps_done * world / dt, "unit": UNIT, "h2d_bytes_per_step": h2d * T,
            "d2h_bytes_per_step": d2h * T + d2h_final, "decode_steps_run": steps_done,
            "note": "per benchmark step (all decode steps): logits H2D from pinned memory every decode step "
                    "(3 device buffers, copy stream), outputs D2H every decode step, the all-finished stop checked "
                    "2 steps behind, final token sequences D2H at the end, wall clock"}


def bench_reference(args, w: synth.Workload):
    """The oracle timed on the host cores; each benchmark step = one bounded sample (2 batch-steps)."""
    import oracle

    oracle.build()
    T = w.steps
    for i in range(args.warmup):
        time_oracle_sample(w, [i % w.batch], [1], True)
    total, bs = 0.0, 0
    for i in range(args.steps):
        dt, n = time_oracle_sample(w, [(2 * i) % w.batch, (2 * i + 1) % w.batch], [1 + (i % T)], True)
        total += dt
        bs += n
    per = total / bs
    value = 1.0 / (per * w.batch)
    sample = (f"{args.steps} samples of 2 batches x 1 decode step of {w.name} (beam step + cache refresh), "
              f"single thread; {per * 1e3:.1f} ms per batch-step, scaled to all {w.batch} batches and "
              f"{T} decode steps (extrapolated)")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * w.batch * T * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generators)", "impl": "reference",
            "config": workload_config(w, T, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count() or 1,
                             "kind": "oracle", "sample": sample, "extrapolated": True},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world, rank, local = dist_env()
    w = synth.WORKLOADS[args.workload]
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(bench_reference(args, w)))
            return
        if args.kernel:
            if rank == 0:
                print(json.dumps(bench_kernel(args, w)))
            return
        line = bench_gpu(args, w, world, rank, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(w)
            print(json.dumps(line))
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
