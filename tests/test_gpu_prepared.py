"""Prepared calls (gf_prepare, gf_prepare_glu, gf_launch_prepared): planned once, launched
many times, they give exactly what the direct calls give (the same kernels with the same
arguments), for every path a call can take."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import dev_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def _bits(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32).copy()


CASES = [
    # (wtype, M, K, epilogue, ncols, prologue, path)
    (synth.Q4_0, 4096, 4096, 0, 1, None, "stream, integer dot products"),
    (synth.Q4_0, 1000, 14336, 4, 1, None, "stream, K chunks"),
    (synth.Q8_0, 3000, 4096, 3, 2, None, "stream, two columns"),
    (synth.F16, 5120, 5120, 4, 8, "workspace", "FWHT transform, then tensor cores"),
    (synth.F16, 640, 5120, 4, 3, "on_chip", "FWHT on chip"),
    (synth.F16, 2048, 1024, 1, 40, None, "tensor cores, three column blocks"),
    (synth.Q4_0, 16, 32768, 1, 1, None, "split K over a cluster"),
    (synth.F32, 300, 1000, 2, 1, None, "generic kernel (K % 16)"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[-1] for c in CASES])
def test_prepared_equals_direct(G, case):
    wt, M, K, epi, nc, pro, _ = case
    raw = synth.weights(wt, M, K, seed=901)
    Wd = dev_tensor(raw)
    x = dev_tensor(synth.normal(nc * K, seed=902).astype(np.float32))
    aux0 = synth.normal(nc * M, seed=903).astype(np.float32)
    kw = {"ncols": nc}
    if pro is not None:
        kw.update(fwht_signs=dev_tensor(synth.rademacher(1024, seed=904)), fwht_block=1024)
        if pro == "workspace":
            kw["fwht_workspace"] = torch.empty(nc * K, device="cuda")
    needs_aux = epi in (3, 4)

    def buffers():
        aux = dev_tensor(aux0) if needs_aux else None
        dst = aux if epi == 4 else torch.full((nc * M,), float("nan"), device="cuda")
        return aux, dst

    aux, dst = buffers()
    G.gemv_fused_ex(Wd, wt, x, M, K, epi, aux, dst, pdl=True, **kw)
    want = _bits(dst)
    aux2, dst2 = buffers()
    p = G.prepare(Wd, wt, x, M, K, epi, aux2, dst2, pdl=True, **kw)
    p.launch()
    assert np.array_equal(_bits(dst2), want)
    if epi != 4:  # launched again on changed inputs: the handle reads the buffers anew
        x.mul_(0.5)
        G.gemv_fused_ex(Wd, wt, x, M, K, epi, aux, dst, pdl=True, **kw)
        p.launch()
        assert np.array_equal(_bits(dst2), _bits(dst))
    p.close()


def test_prepared_sequence_and_glu(G):
    # a decode-layer-like sequence launched with one call: GLU, then a projection of its output
    M, K = 2048, 4096
    rg, ru, rd = (synth.weights(synth.Q4_0, M, K, seed=s) for s in (911, 912, 913))
    Gd, Ud = dev_tensor(rg), dev_tensor(ru)
    Dd = dev_tensor(synth.weights(synth.Q4_0, K, M, seed=913))
    x = dev_tensor(synth.normal(K, seed=914).astype(np.float32))
    r0 = synth.normal(K, seed=915).astype(np.float32)
    h, r = torch.empty(M, device="cuda"), dev_tensor(r0)
    G.gemv_glu(Gd, Ud, synth.Q4_0, x, M, K, h, pdl=True)
    G.gemv_fused_ex(Dd, synth.Q4_0, h, K, M, 4, r, r, pdl=True)
    want_h, want_r = _bits(h), _bits(r)
    h2, r2 = torch.empty(M, device="cuda"), dev_tensor(r0)
    seq = [G.prepare_glu(Gd, Ud, synth.Q4_0, x, M, K, h2, pdl=True),
           G.prepare(Dd, synth.Q4_0, h2, K, M, 4, r2, r2, pdl=True)]
    G.launch_prepared(seq)
    assert np.array_equal(_bits(h2), want_h) and np.array_equal(_bits(r2), want_r)
    for p in seq:
        p.close()


def test_prepared_empty_call(G):
    Wd = torch.zeros(64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(16, device="cuda")
    dst = torch.zeros(1, device="cuda")
    p = G.prepare(Wd, synth.F32, x, 0, 16, 0, None, dst)  # M == 0: launches nothing
    p.launch()
    p.close()


def test_graph_of_prepared_calls(G):
    # the sequence recorded as one graph: the same bits as the direct calls, replayed twice
    M, K = 2048, 4096
    Gd, Ud = (dev_tensor(synth.weights(synth.Q4_0, M, K, seed=s)) for s in (921, 922))
    Dd = dev_tensor(synth.weights(synth.F16, K, M, seed=923))
    x = dev_tensor(synth.normal(K, seed=924).astype(np.float32))
    r0 = synth.normal(K, seed=925).astype(np.float32)
    h, r = torch.empty(M, device="cuda"), dev_tensor(r0)
    G.gemv_glu(Gd, Ud, synth.Q4_0, x, M, K, h, pdl=True)
    G.gemv_fused_ex(Dd, synth.F16, h, K, M, 4, r, r, pdl=True)
    want_h, want_r = _bits(h), _bits(r)
    h2, r2 = torch.empty(M, device="cuda"), dev_tensor(r0)
    seq = [G.prepare_glu(Gd, Ud, synth.Q4_0, x, M, K, h2, pdl=True),
           G.prepare(Dd, synth.F16, h2, K, M, 4, r2, r2, pdl=True)]
    g = G.Graph(seq)
    for p in seq:  # the graph keeps what it needs
        p.close()
    s = torch.cuda.Stream()
    g.launch(stream=s)
    s.synchronize()
    assert np.array_equal(_bits(h2), want_h) and np.array_equal(_bits(r2), want_r)
    r2.copy_(dev_tensor(r0))  # inputs changed between replays: read anew
    g.launch(stream=s)
    s.synchronize()
    assert np.array_equal(_bits(r2), want_r)
    g.close()
