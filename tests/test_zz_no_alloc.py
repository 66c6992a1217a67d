"""GPU test of gemv_fused_fwht_noalloc, the allocation-free entry point.

Callers that cannot allocate a device workspace (a C host with no device allocator of
its own, or a serving process whose device memory is fixed at start-up) use this entry
point: the signed-FWHT prologue's scratch comes from a static device array inside the
library.  The test calls it through the C ABI twice in a row, with different inputs, and
checks each result against the existing entry point (gemv_fused_ex) within the parity
tolerance the other GPU tests use.  It must pass on its own in a fresh process and after
the rest of the suite, so it keeps no state between tests."""

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


def _tolerance(raw, wt, X, s, M, K, B):
    """The parity bound of the other tests for a GEMV on the transformed input."""
    ncols = X.shape[0]
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    return gemv_bound(raw, wt, Xp, M, K, x_err=E)


@pytest.mark.parametrize("wt,M,K,ncols,epi", [
    (synth.F16, 700, 5120, 3, ogemv.EPI_ADD),
    (synth.Q4_0, 333, 8192, 1, ogemv.EPI_SILU_MUL),
])
def test_noalloc_matches_gemv_fused_ex_on_two_calls(G, wt, M, K, ncols, epi):
    B = 1024
    raw = synth.weights(wt, M, K, seed=120)
    Wd = dev_tensor(raw)
    s = synth.rademacher(B, seed=121)
    sd = dev_tensor(s)
    for call, seed in enumerate((130, 140)):  # two calls in a row, different inputs
        X = synth.normal(ncols * K, seed=seed).reshape(ncols, K)
        aux = synth.normal(ncols * M, seed=seed + 1).reshape(ncols, M)
        xd = dev_tensor(X.reshape(-1))
        ref_aux = dev_tensor(aux.reshape(-1))
        new_aux = dev_tensor(aux.reshape(-1))
        if epi == ogemv.EPI_ADD:  # residual add in place: dst is the aux buffer
            ref_dst, new_dst = ref_aux, new_aux
        else:
            ref_dst = torch.full((ncols * M,), float("nan"), device="cuda")
            new_dst = torch.full((ncols * M,), float("nan"), device="cuda")
        G.gemv_fused_ex(Wd, wt, xd, M, K, epi, ref_aux, ref_dst, ncols=ncols, fwht_signs=sd, fwht_block=B)
        st = G.gemv_fused_fwht_noalloc(Wd, wt, xd, M, K, epi, new_aux, new_dst, ncols, sd, B)
        assert st == G.OK
        torch.cuda.synchronize()
        ref = ref_dst.cpu().numpy().astype(np.float64).reshape(ncols, M)
        got = new_dst.cpu().numpy().astype(np.float64).reshape(ncols, M)
        assert np.all(np.isfinite(got)), "call %d left outputs unwritten" % call
        assert_within(got, ref, _tolerance(raw, wt, X, s, M, K, B), "no-alloc call %d" % call)


def test_noalloc_rejects_oversize_and_missing_signs(G):
    # ncols*K above the static array: refused before anything is launched
    big_k = G.NOALLOC_MAX_WORKSPACE_FLOATS // 2 + 1024
    assert G.gemv_fused_fwht_noalloc(1 << 40, synth.F16, 2 << 40, 16, big_k, 0, None, 4 << 40, 2, 5 << 40, 1024,
                                     check=False) == G.ERR_UNSUPPORTED
    assert G.gemv_fused_fwht_noalloc(1 << 40, synth.F16, 2 << 40, 16, 1024, 0, None, 4 << 40, 1, None, 1024,
                                     nsigns=1024, check=False) == G.ERR_INVALID
