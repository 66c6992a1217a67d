"""Guard bands around every buffer a call touches (in place of a memory checker).

Each operand sits inside a larger allocation with 4 KiB on either side filled with the
byte 0xA5.  After ragged-shape calls through every entry point the bands must be
untouched: no kernel reads its way into a write past the end (or before the start) of
dst, aux, the FWHT workspace or the multi / dual-GEMV outputs, and none writes into W,
x, the signs or the RMS weight.  The outputs are also checked against the oracle so a
band cannot stay clean because nothing was written."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, fwht_err_bound, gemv_bound, glu_bound
from oracle import fwht as ofwht
from oracle import gemv as ogemv
from oracle import quant as oquant

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GUARD = 4096
PAT = 0xA5


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


class Guarded:
    """A device tensor of n elements between two 4 KiB bands of PAT bytes."""

    def __init__(self, arr=None, n=None, dtype=torch.float32, fill=None):
        if arr is not None:
            arr = np.ascontiguousarray(arr)
            dtype = {np.dtype(np.float32): torch.float32, np.dtype(np.uint8): torch.uint8}[arr.dtype]
            n = arr.size
        isz = torch.tensor([], dtype=dtype).element_size()
        self.g = GUARD // isz
        self.n = n
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(PAT)
        self.t = self.buf[self.g:self.g + n]
        if arr is not None:
            self.t.copy_(torch.from_numpy(arr))
        elif fill is not None:
            self.t.fill_(fill)

    def intact(self):
        b = self.buf.view(torch.uint8)
        gb = self.g * self.buf.element_size()
        lo, hi = b[:gb], b[b.numel() - gb:]
        return bool(torch.all(lo == PAT).item()) and bool(torch.all(hi == PAT).item())

    def host(self):
        return self.t.cpu().numpy().astype(np.float64)


def check_all(*bufs):
    torch.cuda.synchronize()
    for i, b in enumerate(bufs):
        assert b.intact(), "guard band of operand %d was written" % i


# (format, M, K): rows from one to 65536, K from one unit and a ragged tail to 14336
SHAPES = [
    (synth.F32, 1, 33), (synth.F32, 611, 32), (synth.F32, 65536, 33), (synth.F32, 611, 14336),
    (synth.F16, 1, 14336), (synth.F16, 611, 33), (synth.F16, 65536, 32), (synth.F16, 611, 14336),
    (synth.Q8_0, 1, 32), (synth.Q8_0, 611, 14336), (synth.Q8_0, 65536, 32),
    (synth.Q4_0, 1, 14336), (synth.Q4_0, 611, 32), (synth.Q4_0, 65536, 64), (synth.Q4_0, 611, 14336),
    (synth.Q4_K, 611, 256), (synth.Q4_K, 1, 14336), (synth.Q4_K, 65536, 256),
]


@pytest.mark.parametrize("wt,M,K", SHAPES)
def test_gemv_fused_guard_bands(G, wt, M, K):
    raw = synth.weights(wt, M, K, seed=900 + M % 97 + K % 89)
    x = synth.normal(K, seed=901)
    r = synth.normal(M, seed=902)
    W, X = Guarded(raw), Guarded(x)
    for epi in (ogemv.EPI_SILU_MUL, ogemv.EPI_ADD):
        aux = Guarded(r)
        dst = aux if epi == ogemv.EPI_ADD else Guarded(n=M, fill=float("nan"))
        G.gemv_fused(W.t, wt, X.t, M, K, epi, aux.t, dst.t)
        check_all(W, X, aux, dst)
        want = ogemv.gemv(raw, wt, x, M, K, epi, r)
        assert_within(dst.host().reshape(1, M), want, gemv_bound(raw, wt, x, M, K), "guarded %d %dx%d" % (wt, M, K))


@pytest.mark.parametrize("wt,M,K,ncols", [(synth.F16, 611, 1024, 3), (synth.F16, 611, 1024, 8),
                                           (synth.F16, 611, 1024, 12), (synth.F16, 8200, 1024, 13),
                                           (synth.Q4_0, 611, 2048, 5), (synth.F32, 65, 33, 2)])
def test_batch_and_fwht_workspace_guard_bands(G, wt, M, K, ncols):
    B = 1024 if K % 1024 == 0 else 0
    raw = synth.weights(wt, M, K, seed=910)
    X = synth.normal(ncols * K, seed=911).reshape(ncols, K)
    r = synth.normal(ncols * M, seed=912).reshape(ncols, M)
    W, Xd, aux = Guarded(raw), Guarded(X.reshape(-1)), Guarded(r.reshape(-1))
    if B:
        s = synth.rademacher(B, seed=913)
        S = Guarded(s)
        ws = Guarded(n=ncols * K, fill=0.0)
        G.gemv_fused_ex(W.t, wt, Xd.t, M, K, ogemv.EPI_ADD, aux.t, aux.t, ncols=ncols, fwht_signs=S.t,
                        fwht_block=B, fwht_workspace=ws.t)
        check_all(W, Xd, aux, S, ws)
        Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
        E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
        want = ogemv.gemv(raw, wt, Xp, M, K, ogemv.EPI_ADD, r)
        bound = gemv_bound(raw, wt, Xp, M, K, x_err=E)
    else:
        G.gemv_fused_ex(W.t, wt, Xd.t, M, K, ogemv.EPI_ADD, aux.t, aux.t, ncols=ncols)
        check_all(W, Xd, aux)
        want = ogemv.gemv(raw, wt, X, M, K, ogemv.EPI_ADD, r)
        bound = gemv_bound(raw, wt, X, M, K)
    assert_within(aux.host().reshape(ncols, M), want, bound, "guarded batch")


@pytest.mark.parametrize("wt,M,K", [(synth.Q4_0, 611, 4096), (synth.Q4_0, 1, 14336), (synth.F16, 33, 32),
                                     (synth.Q4_K, 611, 4096)])
def test_glu_and_rms_guard_bands(G, wt, M, K):
    rg, ru = synth.weights(wt, M, K, seed=920), synth.weights(wt, M, K, seed=921)
    x = synth.normal(K, seed=922)
    gamma = (1.0 + 0.1 * synth.normal(K, seed=923)).astype(np.float32)
    Wg, Wu, X, GM = Guarded(rg), Guarded(ru), Guarded(x), Guarded(gamma)
    dst = Guarded(n=M, fill=float("nan"))
    G.gemv_glu(Wg.t, Wu.t, wt, X.t, M, K, dst.t)
    check_all(Wg, Wu, X, dst)
    assert_within(dst.host().reshape(1, M), ogemv.gemv_glu(rg, ru, wt, x, M, K), glu_bound(rg, ru, wt, x, M, K), "glu")
    dst2 = Guarded(n=M, fill=float("nan"))
    G.gemv_fused_ex(Wg.t, wt, X.t, M, K, ogemv.EPI_NONE, None, dst2.t, rms_norm_weight=GM.t, rms_norm_eps=1e-6)
    check_all(Wg, X, GM, dst2)
    assert np.all(np.isfinite(dst2.host()))


def test_multi_guard_bands(G):
    K = 4096
    shapes = [(611, ogemv.EPI_NONE), (1, ogemv.EPI_ADD), (4096, ogemv.EPI_SILU_MUL), (32, ogemv.EPI_SIGMOID)]
    raws = [synth.weights(synth.Q4_0, M, K, seed=930 + i) for i, (M, _) in enumerate(shapes)]
    x = synth.normal(K, seed=935)
    Ws = [Guarded(r) for r in raws]
    X = Guarded(x)
    auxs = [Guarded(synth.normal(M, seed=940 + i)) for i, (M, _) in enumerate(shapes)]
    dsts = [auxs[i] if e == ogemv.EPI_ADD else Guarded(n=M, fill=float("nan")) for i, (M, e) in enumerate(shapes)]
    aux_np = [a.host() for a in auxs]
    items = [(Ws[i].t, M, e, auxs[i].t if e in ogemv.NEEDS_AUX else None, dsts[i].t) for i, (M, e) in enumerate(shapes)]
    G.gemv_multi(items, synth.Q4_0, X.t, K)
    check_all(X, *Ws, *auxs, *dsts)
    for i, (M, e) in enumerate(shapes):
        want = ogemv.gemv(raws[i], synth.Q4_0, x, M, K, e, aux_np[i].reshape(1, M))
        assert_within(dsts[i].host().reshape(1, M), want, gemv_bound(raws[i], synth.Q4_0, x, M, K), "multi %d" % i)


@pytest.mark.parametrize("n,B", [(1024, 1024), (5 * 1024 * 3, 1024), (64, 2), (96, 32)])
def test_fwht_and_elementwise_guard_bands(G, n, B):
    x = synth.normal(n, seed=950)
    s = synth.rademacher(B, seed=951)
    X, S = Guarded(x), Guarded(s)
    dst = Guarded(n=n, fill=float("nan"))
    G.fwht_signed(X.t, S.t, dst.t, n, B)
    check_all(X, S, dst)
    want = ofwht.fwht_signed(x, s, B)
    assert_within(dst.host(), want, fwht_err_bound(x, B), "fwht")
    out = Guarded(n=n, fill=float("nan"))
    G.elementwise(G.EW_MUL, X.t, S.t, out.t, n, nb=B)
    check_all(X, S, out)
    assert np.array_equal(out.host(), (x.reshape(-1, B) * s).reshape(-1).astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("wt,M,K", [(synth.Q4_0, 611, 96), (synth.Q8_0, 1, 14336), (synth.Q4_K, 33, 512),
                                     (synth.F16, 65, 33)])
def test_dequantize_guard_bands(G, wt, M, K):
    raw = synth.weights(wt, M, K, seed=960)
    W = Guarded(raw)
    out = Guarded(n=M * K, fill=float("nan"))
    G.dequantize(W.t, wt, M, K, out.t)
    check_all(W, out)
    want = oquant.dequantize(raw, wt, M, K).astype(np.float32)
    assert np.array_equal(out.t.cpu().numpy().reshape(M, K).view(np.uint32), want.view(np.uint32))


def test_noalloc_guard_bands(G):
    M, K, ncols, B = 611, 5120, 3, 1024
    raw = synth.weights(synth.F16, M, K, seed=970)
    X = synth.normal(ncols * K, seed=971).reshape(ncols, K)
    r = synth.normal(ncols * M, seed=972).reshape(ncols, M)
    s = synth.rademacher(B, seed=973)
    W, Xd, aux, S = Guarded(raw), Guarded(X.reshape(-1)), Guarded(r.reshape(-1)), Guarded(s)
    assert G.gemv_fused_fwht_noalloc(W.t, synth.F16, Xd.t, M, K, ogemv.EPI_ADD, aux.t, aux.t, ncols, S.t, B) == G.OK
    check_all(W, Xd, aux, S)
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, synth.F16, Xp, M, K, ogemv.EPI_ADD, r)
    assert_within(aux.host().reshape(ncols, M), want, gemv_bound(raw, synth.F16, Xp, M, K, x_err=E), "noalloc")


@pytest.mark.parametrize("nbytes", [16, 4112, 1 << 20])
def test_copy_guard_bands(G, nbytes):
    """The staging copy writes exactly its range of a device buffer and reads exactly its
    range of another; host to device and device to host."""
    n = nbytes // 4
    src = np.random.default_rng(nbytes).standard_normal(n).astype(np.float32)
    host_in = torch.from_numpy(src).pin_memory()
    dst = Guarded(n=n, fill=0.0)
    assert G.copy(dst.t, host_in, nbytes) == G.OK
    check_all(dst)
    assert np.array_equal(dst.t.cpu().numpy(), src)
    srcd = Guarded(src)
    host_out = torch.zeros(n, dtype=torch.float32).pin_memory()
    assert G.copy(host_out, srcd.t, nbytes) == G.OK
    check_all(srcd)
    assert np.array_equal(host_out.numpy(), src)
