"""GPU test of gemv_fused_fwht_noalloc, the allocation-free entry point.

Callers that cannot allocate a device workspace (a C host with no device allocator of
its own, or a serving process whose device memory is fixed at start-up) use this entry
point: the signed-FWHT prologue's scratch comes from a static device array inside the
library.  Two calls are issued back to back on one stream, with different inputs and
separate outputs and a single synchronisation after both (once without and once with
programmatic dependent launch): each result is checked against the oracle (the GEMV of
the oracle's signed FWHT of x, within the parity bound of the other tests) and bit for
bit against gemv_fused_ex with a caller-allocated workspace, the path it runs.  The
module is collected last and keeps no state between tests, so it passes alone in a
fresh process and after the rest of the suite."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, fwht_err_bound, gemv_bound
from oracle import fwht as ofwht
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


def _oracle(raw, wt, X, s, M, K, B, epi, aux):
    """The oracle's result and the parity bound for a GEMV on the transformed input."""
    ncols = X.shape[0]
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, wt, Xp, M, K, epi, aux)
    return want, gemv_bound(raw, wt, Xp, M, K, x_err=E)


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("wt,M,K,ncols,epi", [
    (synth.F16, 700, 5120, 3, ogemv.EPI_ADD),
    (synth.Q4_0, 333, 8192, 1, ogemv.EPI_SILU_MUL),
    (synth.F16, 5120, 5120, 8, ogemv.EPI_ADD),
])
def test_noalloc_two_calls_back_to_back(G, wt, M, K, ncols, epi, pdl):
    B = 1024
    raw = synth.weights(wt, M, K, seed=120)
    Wd = dev_tensor(raw)
    s = synth.rademacher(B, seed=121)
    sd = dev_tensor(s)
    st = torch.cuda.Stream()
    calls = []
    for seed in (130, 140):  # two calls, different inputs, separate outputs
        X = synth.normal(ncols * K, seed=seed).reshape(ncols, K)
        aux = synth.normal(ncols * M, seed=seed + 1).reshape(ncols, M)
        xd = dev_tensor(X.reshape(-1))
        auxd = dev_tensor(aux.reshape(-1))
        dst = auxd if epi == ogemv.EPI_ADD else torch.full((ncols * M,), float("nan"), device="cuda")
        calls.append((X, aux, xd, auxd, dst))
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for (X, aux, xd, auxd, dst) in calls:
            assert G.gemv_fused_fwht_noalloc(Wd, wt, xd, M, K, epi, auxd, dst, ncols, sd, B, pdl=pdl,
                                             stream=st) == G.OK
    st.synchronize()
    for i, (X, aux, xd, auxd, dst) in enumerate(calls):
        got = dst.cpu().numpy().astype(np.float64).reshape(ncols, M)
        assert np.all(np.isfinite(got)), "call %d left outputs unwritten" % i
        want, bound = _oracle(raw, wt, X, s, M, K, B, epi, aux)
        assert_within(got, want, bound, "no-alloc call %d" % i)
        # the path it reduces to: a caller-allocated workspace, the same kernels
        ref_aux = dev_tensor(aux.reshape(-1))
        ref_dst = ref_aux if epi == ogemv.EPI_ADD else torch.full((ncols * M,), float("nan"), device="cuda")
        ws = torch.empty(ncols * K, device="cuda")
        G.gemv_fused_ex(Wd, wt, xd, M, K, epi, ref_aux, ref_dst, ncols=ncols, fwht_signs=sd, fwht_block=B,
                        fwht_workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(dst.view(torch.int32), ref_dst.view(torch.int32)), "call %d differs from the workspace path" % i


def test_noalloc_rejects_oversize_and_missing_signs(G):
    # ncols*K above the static array: refused before anything is launched
    big_k = G.NOALLOC_MAX_WORKSPACE_FLOATS // 2 + 1024
    assert G.gemv_fused_fwht_noalloc(1 << 40, synth.F16, 2 << 40, 16, big_k, 0, None, 4 << 40, 2, 5 << 40, 1024,
                                     check=False) == G.ERR_UNSUPPORTED
    assert G.gemv_fused_fwht_noalloc(1 << 40, synth.F16, 2 << 40, 16, 1024, 0, None, 4 << 40, 1, None, 1024,
                                     nsigns=1024, check=False) == G.ERR_INVALID
