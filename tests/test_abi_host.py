"""Host-side checks of the C ABI library (no GPU needed): it loads, exports every
symbol include/ls_beam.h declares, and answers the host-only calls; arguments it
must reject are rejected before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from serving_ls_beam_gb300 import _build

    _build.build()
    import serving_ls_beam_gb300 as lsb

    return lsb.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"LS_API\s+[\w\s\*]+?\b(ls_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"ls_beam_step", "ls_cache_reorder", "ls_beam_step_workspace_size", "ls_read_status",
            "ls_status_string", "ls_workspace_init", "ls_read_row_stats"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    import serving_ls_beam_gb300 as lsb

    for code in range(6):
        assert lsb.ls_status_string(code)
    assert lsb.ls_status_string(99) == "unknown status"


def test_workspace_size(lib):
    import serving_ls_beam_gb300 as lsb

    assert lsb.ls_beam_step_workspace_size(4, 4, 1024) > 0
    assert lsb.ls_beam_step_workspace_size(4, 0, 1024) == 0
    assert lsb.ls_beam_step_workspace_size(4, 65, 1024) == 0
    assert lsb.ls_beam_step_workspace_size(4, 8, 7) == 0
    assert lsb.ls_beam_step_workspace_size(1, 64, 1 << 26) == 0  # k * vocab >= 2^31
    a = lsb.ls_beam_step_workspace_size(32, 4, 40000)
    b = lsb.ls_beam_step_workspace_size(64, 4, 40000)
    assert 0 < a < b
    assert lsb.ls_beam_step_workspace_size(0, 4, 40000) > 0


def test_host_argument_checks(lib):
    """Shape errors return LS_ERR_INVALID_ARG from host checks alone (no device touched)."""
    E = 1
    p = ctypes.c_void_p(16)  # never dereferenced: the shape checks fail first
    assert lib.ls_beam_step(p, 0, None, p, None, 2, 0, 100, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 0, None, p, None, 2, 65, 100, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 0, None, p, None, 2, 4, 3, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 0, None, p, None, 2, 4, 100, 100, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 7, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 0, None, p, None, -1, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(None, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E
    assert lib.ls_beam_step(p, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 10, None) == E  # tiny workspace
    assert lib.ls_beam_step(None, 0, None, None, None, 0, 4, 100, 0, None, None, None, None, None, 0, None) == 0
    assert lib.ls_cache_reorder(p, p, 1, p, 1, 1, 1, 1, 4, 5, 8, None, None) == E  # len > max_len
    assert lib.ls_cache_reorder(p, p, 1, p, 1, 1, 0, 1, 4, 2, 8, None, None) == E  # k = 0
    assert lib.ls_cache_reorder(p, p, 1, p, 1, 1, 2, 1, 4, 2, 8, None, None) == E  # src == dst
    assert lib.ls_cache_reorder(None, None, 1, None, 1, 1, 2, 1, 4, 0, 8, None, None) == 0  # len 0 no-op
    assert lib.ls_backtrack(p, p, -1, 2, 3, 0, p, p, None, None) == E  # steps < 0
    # the projection-fused step: f16 / bf16 operands, dim a multiple of 8, 16-byte aligned operands
    F = lib.ls_logits_beam_step
    F.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + \
        [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p]
    q = ctypes.c_void_p(24)  # 8-byte aligned only
    assert F(p, p, 0, 64, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E  # f32 operands
    assert F(p, p, 2, 60, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E  # dim % 8
    assert F(p, p, 2, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E  # dim 0
    assert F(q, p, 2, 64, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E  # misaligned hidden
    assert F(p, q, 2, 64, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1 << 20, None) == E  # misaligned weight
    assert F(p, p, 2, 64, None, p, None, 2, 4, 100, 100, p, p, p, None, p, 1 << 20, None) == E  # eos
    assert F(p, p, 2, 64, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 10, None) == E  # tiny workspace
    assert F(p, p, 2, 64, None, p, None, 2, 33, 100, 0, p, p, p, None, p, 1 << 30, None) == 2  # k > 32
    assert F(None, None, 2, 64, None, None, None, 0, 4, 100, 0, None, None, None, None, None, 0, None) == 0
    assert lib.ls_backtrack(p, p, 4, 2, 0, 0, p, p, None, None) == E  # k = 0
    assert lib.ls_backtrack(p, p, 4, 2, 65, 0, p, p, None, None) == E  # k > 64
    assert lib.ls_backtrack(None, p, 4, 2, 3, 0, p, p, None, None) == E  # no history
    assert lib.ls_backtrack(None, None, 0, 2, 3, 0, None, None, None, None) == 0  # no steps: no-op
    # the step followed by the in-place refresh: the refresh's checks run before anything is queued
    R = lib.ls_beam_step_refresh_inplace
    R.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + \
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert R(p, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 1, 1, 1, 4, 5, 8, p, 1 << 20, None) == E  # len
    assert R(p, 0, None, p, None, 2, 4, 100, 0, p, None, p, None, p, 1, 1, 1, 4, 2, 8, p, 1 << 20, None) == E
    assert R(p, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, p, 7, 1, 1, 4, 2, 8, p, 1 << 20, None) == E  # dtype
    assert R(p, 0, None, p, None, 2, 4, 100, 0, p, p, p, None, None, 1, 1, 1, 4, 2, 8, p, 1 << 20, None) == E
    assert lib.ls_read_status(None, None) == E
    assert lib.ls_workspace_init(None, 0, None) == E


def test_fast_division_method():
    """The cache gather divides by an invariant with a multiply-high (Granlund & Montgomery 1994).
    Check the round-up multiplier rule against integer division on many divisors and dividends."""
    import numpy as np

    g = np.random.default_rng(0)
    for d in list(range(1, 300)) + [511, 512, 513, 1023, 1024, 4096, 65535, 65536, 1 << 20, (1 << 30) - 1]:
        s = 0
        while (1 << s) < d:
            s += 1
        m = ((1 << 32) * ((1 << s) - d)) // d + 1
        assert m < (1 << 32)
        ns = np.concatenate([np.arange(0, 2000), g.integers(0, 1 << 31, 3000), [(1 << 31) - 1]]).astype(np.uint64)
        q = ((((ns * np.uint64(m)) >> np.uint64(32)) + ns) >> np.uint64(s))
        assert np.array_equal(q, ns // np.uint64(d)), d
