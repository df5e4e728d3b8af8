"""GPU parity of ls_cache_reorder: bitwise equality with the oracle's host gather."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import serving_ls_beam_gb300 as lsb  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lsb.load_library()
    return torch.device("cuda:0")


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("dtype,shape,length", [
    (torch.float16, (2, 3, 4, 3, 17, 64), 17),
    (torch.float16, (2, 3, 4, 3, 17, 64), 5),
    (torch.float16, (1, 2, 4, 2, 9, 7), 3),       # 14-byte rows: 2-byte copy units
    (torch.float32, (3, 2, 3, 5, 8, 12), 8),
    (torch.bfloat16, (2, 4, 2, 2, 64, 64), 64),
    (torch.float16, (6, 8, 4, 16, 64, 64), 33),
])
def test_reorder_matches_oracle(dev, oracle_mod, dtype, shape, length):
    layers, batch, k, heads, max_len, head_dim = shape
    g = np.random.default_rng(sum(shape) + length)
    src = torch.from_numpy(g.standard_normal((layers, batch * k, heads, max_len, head_dim)).astype(np.float32)).to(dtype)
    parent = torch.from_numpy(synth.parents(batch, k, seed=length))
    d_src = src.to(dev)
    d_dst = torch.full_like(d_src, 7.0)
    lsb.check(lsb.ls_cache_reorder(d_src, d_dst, parent.to(dev), length))
    torch.cuda.synchronize()
    exp = oracle_mod.cache_reorder(_bits(src), parent.numpy(), length, dst=_bits(torch.full_like(src, 7.0)))
    assert np.array_equal(_bits(d_dst), exp)


def test_reorder_workload_c3_full(dev, oracle_mod):
    """Full-size c3 cache [6, 512, 16, 64, 64] fp16 (805 MB moved); every row checked bitwise
    against the oracle's gather of the whole cache."""
    w = synth.WORKLOADS["c3"]
    layers, heads, max_len, head_dim = w.kv_shape
    shape = (layers, w.rows, heads, max_len, head_dim)
    parent = synth.parents(w.batch, w.k, seed=w.seed)
    d_src = torch.from_numpy(synth.kv_cache(shape, w.seed)).to(dev)
    d_dst = torch.empty_like(d_src)
    lsb.check(lsb.ls_cache_reorder(d_src, d_dst, torch.from_numpy(parent).to(dev), max_len))
    torch.cuda.synchronize()
    src = d_src.cpu().numpy()
    del d_src
    exp = oracle_mod.cache_reorder(src, parent, max_len)
    got = d_dst.cpu().numpy()
    assert np.array_equal(got.view(np.int16), exp.view(np.int16))


def test_reorder_bad_parent_and_overlap(dev):
    src = torch.randn(2, 4, 2, 8, 16, device=dev, dtype=torch.float16)
    dst = torch.zeros_like(src)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    parent = torch.tensor([[0, 1], [2, 1]], dtype=torch.int32, device=dev)  # 2 is out of range for k=2
    assert lsb.ls_cache_reorder(src, dst, parent, 8, workspace=ws) == lsb.LS_OK
    assert lsb.ls_read_status(ws) == lsb.LS_ERR_INTERNAL
    assert (dst[:, 2] == 0).all()                         # the bad row is left unwritten
    assert torch.equal(dst[:, 3], src[:, 3])              # b=1, j=1 -> parent 1 -> row 3
    assert lsb.ls_read_status(ws) == lsb.LS_OK            # reading clears the status
    assert lsb.ls_cache_reorder(src, src, parent, 8) == lsb.LS_ERR_INVALID_ARG
    flat = torch.zeros(src.numel() * 2, dtype=torch.float16, device=dev)
    a, b = flat[: src.numel()].view(src.shape), flat[src.numel() // 2: src.numel() // 2 + src.numel()].view(src.shape)
    assert lsb.ls_cache_reorder(a, b, parent, 8) == lsb.LS_ERR_INVALID_ARG
    good = torch.tensor([[0, 1], [1, 1]], dtype=torch.int32, device=dev)
    assert lsb.ls_cache_reorder(src, dst, good, 0) == lsb.LS_OK  # len 0: no-op
