"""GPU parity of the Q4_K format through the C ABI against the fp64 oracle: decoded
weights bit-exact (each value d*sc*q - dmin*m has one rounding), GEMV outputs within
2e-5 * sum_k (|d sc q| + |dmin m|) |x_k| + 1e-6 (the kernel adds the min term through a
per-unit sum of x), on every tail, batch, prologue and kernel path."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, gemv_bound, glu_bound, norm_bound, TOL_NORM_REL
from oracle import gemv as ogemv
from oracle import norm as onorm
from oracle import quant as oquant

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

Q4K = synth.Q4_K
EPIS = [ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD]


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def _nan(n):
    return torch.full((n,), float("nan"), device="cuda")


@pytest.mark.parametrize("M,K,offset", [(64, 4096, 0), (3, 256, 0), (5, 768, 2)])
def test_q4_k_dequantize_bit_exact(G, M, K, offset):
    raw = synth.weights(Q4K, M, K, seed=500)
    if offset:  # 2-byte-aligned rows go through 16-bit loads
        buf = torch.zeros(raw.size + 16, dtype=torch.uint8, device="cuda")
        Wd = buf[offset:offset + raw.size]
        Wd.copy_(dev_tensor(raw))
    else:
        Wd = dev_tensor(raw)
    out = torch.empty(M * K, device="cuda")
    G.dequantize(Wd, Q4K, M, K, out)
    torch.cuda.synchronize()
    want = oquant.dequantize(raw, Q4K, M, K).astype(np.float32)
    assert np.array_equal(out.cpu().numpy().reshape(M, K).view(np.uint32), want.view(np.uint32))


def test_q4_k_dequantize_golden_block(G):
    from conftest import read_golden
    gd = read_golden("q4_k_block.txt")
    raw = np.array([int(t, 16) for t in gd["bytes"][0]], dtype=np.uint8)
    out = torch.empty(256, device="cuda")
    G.dequantize(dev_tensor(raw), Q4K, 1, 256, out)
    torch.cuda.synchronize()
    want = np.concatenate([[float(v) for v in row] for row in gd["values"]])
    assert np.array_equal(out.cpu().numpy().astype(np.float64), want)


def run(G, raw, X, M, K, epi, aux=None, ncols=1, w_offset=0, **kw):
    if w_offset:
        buf = torch.zeros(raw.size + 32, dtype=torch.uint8, device="cuda")
        Wd = buf[w_offset:w_offset + raw.size]
        Wd.copy_(dev_tensor(raw))
    else:
        Wd = dev_tensor(raw)
    xd = dev_tensor(np.asarray(X, dtype=np.float32).reshape(-1))
    auxd = dev_tensor(np.asarray(aux, dtype=np.float32).reshape(-1)) if aux is not None else None
    dst = auxd if epi == ogemv.EPI_ADD else _nan(ncols * M)
    path, info = G.plan(Wd, Q4K, xd, M, K, epi, auxd, dst, ncols=ncols, **kw)
    G.gemv_fused_ex(Wd, Q4K, xd, M, K, epi, auxd if epi in ogemv.NEEDS_AUX else None, dst, ncols=ncols, **kw)
    torch.cuda.synchronize()
    return dst.cpu().numpy().astype(np.float64).reshape(ncols, M), path, info


@pytest.mark.parametrize("epi", EPIS)
@pytest.mark.parametrize("M,K", [(333, 4096), (1000, 1024), (7, 256)])
def test_q4_k_tails_and_ragged_rows(G, epi, M, K):
    raw = synth.weights(Q4K, M, K, seed=510)
    X = synth.normal(K, seed=511).reshape(1, K)
    aux = synth.normal(M, seed=512).reshape(1, M)
    got, path, _ = run(G, raw, X, M, K, epi, aux)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, Q4K, X, M, K, epi, aux)
    assert_within(got, want, gemv_bound(raw, Q4K, X, M, K), "q4_k epi %d %dx%d" % (epi, M, K))


@pytest.mark.parametrize("ncols", [2, 3, 8])
def test_q4_k_batch(G, ncols):
    M, K = 517, 4096
    raw = synth.weights(Q4K, M, K, seed=520)
    X = synth.normal(ncols * K, seed=521).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=522).reshape(ncols, M)
    got, _, _ = run(G, raw, X, M, K, ogemv.EPI_ADD, aux, ncols=ncols)
    want = ogemv.gemv(raw, Q4K, X, M, K, ogemv.EPI_ADD, aux)
    assert_within(got, want, gemv_bound(raw, Q4K, X, M, K), "q4_k batch")


def test_q4_k_generic_path(G):
    M, K = 90, 1024
    raw = synth.weights(Q4K, M, K, seed=530)
    X = synth.normal(2 * K, seed=531).reshape(2, K)
    aux = synth.normal(2 * M, seed=532).reshape(2, M)
    got, path, _ = run(G, raw, X, M, K, ogemv.EPI_SILU_MUL, aux, ncols=2, w_offset=2)
    assert path == G.PATH_GENERIC
    want = ogemv.gemv(raw, Q4K, X, M, K, ogemv.EPI_SILU_MUL, aux)
    assert_within(got, want, gemv_bound(raw, Q4K, X, M, K), "q4_k generic")


def test_q4_k_long_rows_k_chunks_and_split(G):
    for M, K in ((64, 28672), (8, 65536)):
        raw = synth.weights(Q4K, M, K, seed=540)
        X = synth.normal(K, seed=541).reshape(1, K)
        for split in (True, False):
            got, _, info = run(G, raw, X, M, K, ogemv.EPI_NONE, split_k=split)
            if not split:
                assert info["split"] == 1
            want = ogemv.gemv(raw, Q4K, X, M, K)
            assert_within(got, want, gemv_bound(raw, Q4K, X, M, K), "q4_k %dx%d split=%s" % (M, K, split))
    assert info is not None


def test_q4_k_glu_and_rms_norm(G):
    M, K, eps = 700, 4096, 1e-6
    rg, ru = synth.weights(Q4K, M, K, seed=550), synth.weights(Q4K, M, K, seed=551)
    X = (synth.normal(K, seed=552) * 2.0).reshape(1, K)
    gamma = 1.0 + 0.1 * synth.normal(K, seed=553)
    Gd, Ud = dev_tensor(rg), dev_tensor(ru)
    xd, gd = dev_tensor(X.astype(np.float32).reshape(-1)), dev_tensor(gamma.astype(np.float32))
    dst = _nan(M)
    G.gemv_glu(Gd, Ud, Q4K, xd, M, K, dst, rms_norm_weight=gd, rms_norm_eps=eps)
    torch.cuda.synchronize()
    Xn = onorm.rms_norm(X, gamma, eps, K)
    want = ogemv.gemv_glu(rg, ru, Q4K, Xn, M, K)
    got = dst.cpu().numpy().astype(np.float64).reshape(1, M)
    assert_within(got, want, glu_bound(rg, ru, Q4K, Xn, M, K, extra_rel=TOL_NORM_REL), "q4_k glu + rms")
    d2 = _nan(M)
    G.gemv_fused_ex(Gd, Q4K, xd, M, K, ogemv.EPI_NONE, None, d2, rms_norm_weight=gd, rms_norm_eps=eps)
    torch.cuda.synchronize()
    want2 = ogemv.gemv(rg, Q4K, Xn, M, K)
    assert_within(d2.cpu().numpy().astype(np.float64).reshape(1, M), want2, norm_bound(rg, Q4K, Xn, M, K),
                  "q4_k rms")


def test_q4_k_full_ffn_down_every_row(G):
    # the FFN down projection of a decode layer in Q4_K: 4096 x 14336, residual add in place
    M, K = 4096, 14336
    raw = synth.weights(Q4K, M, K, seed=560)
    X = synth.normal(K, seed=561).reshape(1, K)
    r = synth.normal(M, seed=562).reshape(1, M)
    got, path, _ = run(G, raw, X, M, K, ogemv.EPI_ADD, r, pdl=True)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, Q4K, X, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, gemv_bound(raw, Q4K, X, M, K), "q4_k full down")
