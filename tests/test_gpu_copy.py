"""GPU tests of the host staging copy (gf_copy, gf_prepare_copy): host <-> device and
device <-> device by a kernel, bit for bit, with and without programmatic dependent
launch; and a decode step recorded as one graph of upload, GEMV and download, checked
against the fp64 oracle."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, gemv_bound
from oracle import gemv as ogemv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0


def words(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(-2**31, 2**31, n, dtype=np.int64)
                            .astype(np.int32))


@pytest.mark.parametrize("n", [4, 1028, 262144, 2621444])  # 16 B .. 10 MB, grid-stride beyond 4 MB
@pytest.mark.parametrize("pdl", [False, True])
def test_copy_each_direction_bitwise(G, n, pdl):
    src_h = words(n, seed=n).pin_memory()
    mid_d = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    mid2_d = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    back_h = torch.full((n,), -1, dtype=torch.int32).pin_memory()
    G.copy(mid_d, src_h, 4 * n, pdl=pdl)           # host -> device
    G.copy(mid2_d, mid_d, 4 * n, pdl=pdl)          # device -> device
    G.copy(back_h, mid2_d, 4 * n, pdl=pdl)         # device -> host
    torch.cuda.synchronize()
    assert torch.equal(mid_d.cpu(), src_h)
    assert torch.equal(back_h, src_h)


def test_copy_refuses_pageable_host_memory(G):
    """Plain (pageable) host memory is refused before any launch, in either direction."""
    n = 4096
    src = words(n, seed=5)
    dst = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert G.copy(dst, src, 4 * n, check=False) == G.ERR_INVALID
    assert G.copy(src, dst, 4 * n, check=False) == G.ERR_INVALID
    assert G.prepare_copy(dst, src, 4 * n, check=False) == G.ERR_INVALID
    torch.cuda.synchronize()
    assert int(dst.abs().sum()) == 0


def test_decode_step_with_host_staging_in_one_graph(G):
    """Upload x and the residual, the GEMV with its in-place add, download the result:
    one graph launch per step, every step with new host inputs."""
    M, K = 4096, 4096
    raw = synth.weights(synth.F16, M, K, seed=90)
    Wd = dev_tensor(raw)
    x_h = torch.empty(K, dtype=torch.float32).pin_memory()
    r_h = torch.empty(M, dtype=torch.float32).pin_memory()
    y_h = torch.empty(M, dtype=torch.float32).pin_memory()
    x_d = torch.empty(K, device="cuda")
    r_d = torch.empty(M, device="cuda")
    calls = [G.prepare_copy(x_d, x_h, 4 * K, pdl=True), G.prepare_copy(r_d, r_h, 4 * M, pdl=True),
             G.prepare(Wd, synth.F16, x_d, M, K, ogemv.EPI_ADD, r_d, r_d, pdl=True),
             G.prepare_copy(y_h, r_d, 4 * M, pdl=True)]
    graph = G.Graph(calls)
    s = torch.cuda.Stream()
    for step in range(3):
        x = synth.normal(K, seed=91 + step)
        r = synth.normal(M, seed=95 + step)
        x_h.copy_(torch.from_numpy(x.astype(np.float32)))
        r_h.copy_(torch.from_numpy(r.astype(np.float32)))
        graph.launch(stream=s)
        s.synchronize()
        want = ogemv.gemv(raw, synth.F16, x.reshape(1, K), M, K, ogemv.EPI_ADD, r.reshape(1, M))
        assert_within(y_h.numpy().astype(np.float64).reshape(1, M), want,
                      gemv_bound(raw, synth.F16, x.reshape(1, K), M, K), "step %d" % step)
