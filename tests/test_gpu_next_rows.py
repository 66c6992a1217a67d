"""GPU parity of the rows beyond the single-GEMV path, through the C ABI against the
fp64 oracle: the gated dual GEMV (gemv_glu), the RMS-normalisation prologue and
split-K over a cluster of CTAs for GEMVs with few rows.  Tolerances: the literal
per-GEMV bound 2e-5 * sum_k |W_ik x'_k| + 1e-6, propagated through silu(g) * u for
the dual GEMV, plus the 1/rms term for the normalisation (tests/gpu_util.py)."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import (assert_within, dev_tensor, fwht_err_bound, gemv_bound, glu_bound, norm_bound,
                      TOL_NORM_REL)
from oracle import fwht as ofwht
from oracle import gemv as ogemv
from oracle import norm as onorm

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ALL_WT = [synth.F32, synth.F16, synth.Q8_0, synth.Q4_0]
EPIS = [ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD]


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def _upload_w(raw, offset=0):
    if not offset:
        return dev_tensor(raw)
    buf = torch.zeros(raw.size + 64, dtype=torch.uint8, device="cuda")
    w = buf[offset:offset + raw.size]
    w.copy_(dev_tensor(raw))
    return w


def _nan_out(n):
    return torch.full((n,), float("nan"), device="cuda")


def _cpu(t, ncols, M):
    return t.cpu().numpy().astype(np.float64).reshape(ncols, M)


def run_glu(G, rg, ru, wt, X, M, K, ncols=1, up_offset=0, **kw):
    Gd, Ud = dev_tensor(rg), _upload_w(ru, up_offset)
    xd = dev_tensor(np.asarray(X, dtype=np.float32).reshape(-1))
    dst = _nan_out(ncols * M)
    path, info = G.plan_glu(Gd, Ud, wt, xd, M, K, dst, ncols=ncols, **kw)
    G.gemv_glu(Gd, Ud, wt, xd, M, K, dst, ncols=ncols, **kw)
    torch.cuda.synchronize()
    return _cpu(dst, ncols, M), path, info


# ----------------------------------------------------------------------------- gated dual GEMV

@pytest.mark.parametrize("wt", ALL_WT)
@pytest.mark.parametrize("M,K", [(333, 4096), (1000, 1024), (8, 512), (2, 2048)])
def test_glu_formats_and_ragged_rows(G, wt, M, K):
    rg, ru = synth.weights(wt, M, K, seed=200 + wt), synth.weights(wt, M, K, seed=210 + wt)
    X = synth.normal(K, seed=220).reshape(1, K)
    got, path, _ = run_glu(G, rg, ru, wt, X, M, K)
    assert path == G.PATH_STREAM
    want = ogemv.gemv_glu(rg, ru, wt, X, M, K)
    assert_within(got, want, glu_bound(rg, ru, wt, X, M, K), "glu wt %d %dx%d" % (wt, M, K))


@pytest.mark.parametrize("wt", [synth.F16, synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("ncols", [2, 3, 8])
def test_glu_batch(G, wt, ncols):
    M, K = 517, 2048
    rg, ru = synth.weights(wt, M, K, seed=230), synth.weights(wt, M, K, seed=231)
    X = synth.normal(ncols * K, seed=232).reshape(ncols, K)
    got, _, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=ncols)
    assert_within(got, ogemv.gemv_glu(rg, ru, wt, X, M, K), glu_bound(rg, ru, wt, X, M, K), "glu batch")


@pytest.mark.parametrize("wt,K,up_offset", [(synth.F16, 40, 0), (synth.F16, 1024, 2), (synth.Q4_0, 96, 0),
                                            (synth.F32, 12, 0)])
def test_glu_generic_path(G, wt, K, up_offset):
    M = 70
    rg, ru = synth.weights(wt, M, K, seed=240), synth.weights(wt, M, K, seed=241)
    X = synth.normal(2 * K, seed=242).reshape(2, K)
    got, path, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=2, up_offset=up_offset)
    assert path == G.PATH_GENERIC
    assert_within(got, ogemv.gemv_glu(rg, ru, wt, X, M, K), glu_bound(rg, ru, wt, X, M, K), "glu generic")


@pytest.mark.parametrize("wt", [synth.F16, synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("ncols", [1, 4])
def test_glu_equals_unfused_bitwise(G, wt, ncols):
    # gate and up rows of the dual kernel are reduced exactly like the plain kernel's
    # rows, so silu(gate) * up equals GEMV(up), then GEMV(gate) with the SILU_MUL tail
    M, K = 1536, 4096
    rg, ru = synth.weights(wt, M, K, seed=250), synth.weights(wt, M, K, seed=251)
    X = synth.normal(ncols * K, seed=252).reshape(ncols, K)
    got, _, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=ncols)
    Gd, Ud = dev_tensor(rg), dev_tensor(ru)
    xd = dev_tensor(X.astype(np.float32).reshape(-1))
    u, g = _nan_out(ncols * M), _nan_out(ncols * M)
    # the plain kernels the dual one is built from (not the tensor-core path)
    G.gemv_fused_ex(Ud, wt, xd, M, K, ogemv.EPI_NONE, None, u, ncols=ncols, tensor_cores=False)
    G.gemv_fused_ex(Gd, wt, xd, M, K, ogemv.EPI_SILU_MUL, u, g, ncols=ncols, tensor_cores=False)
    torch.cuda.synchronize()
    assert np.array_equal(got.astype(np.float32), _cpu(g, ncols, M).astype(np.float32))


def test_glu_with_fwht_prologue_on_chip_and_workspace(G):
    wt, M, K, B, ncols = synth.F16, 640, 5120, 1024, 3
    rg, ru = synth.weights(wt, M, K, seed=260), synth.weights(wt, M, K, seed=261)
    X = synth.normal(ncols * K, seed=262).reshape(ncols, K)
    s = synth.rademacher(B, seed=263)
    sd = dev_tensor(s)
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv_glu(rg, ru, wt, Xp, M, K)
    bound = glu_bound(rg, ru, wt, Xp, M, K, x_err=E)
    on_chip, _, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=ncols, fwht_signs=sd, fwht_block=B)
    assert_within(on_chip, want, bound, "glu + fwht on chip")
    ws = torch.empty(ncols * K, device="cuda")
    via_ws, _, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=ncols, fwht_signs=sd, fwht_block=B, fwht_workspace=ws)
    assert_within(via_ws, want, bound, "glu + fwht workspace")


def test_full_q4_0_ffn_gate_up_every_row(G):
    # the FFN gate/up pair of the Q4_0 decode layer (d_model 4096, ffn 14336) in one launch
    wt, M, K = synth.Q4_0, 14336, 4096
    rg, ru = synth.weights(wt, M, K, seed=270), synth.weights(wt, M, K, seed=271)
    X = synth.normal(K, seed=272).reshape(1, K)
    got, path, info = run_glu(G, rg, ru, wt, X, M, K, pdl=True)
    assert path == G.PATH_STREAM and info["grid"] == torch.cuda.get_device_properties(0).multi_processor_count
    want = ogemv.gemv_glu(rg, ru, wt, X, M, K)
    assert_within(got, want, glu_bound(rg, ru, wt, X, M, K), "full glu")


# ----------------------------------------------------------------------------- RMS normalisation prologue

def run_norm(G, raw, wt, X, gamma, eps, M, K, epi, aux=None, ncols=1, gamma_offset=0, **kw):
    Wd = dev_tensor(raw)
    xd = dev_tensor(np.asarray(X, dtype=np.float32).reshape(-1))
    if gamma_offset:
        gbuf = torch.zeros(K + 16, device="cuda")
        gd = gbuf[gamma_offset:gamma_offset + K]
        gd.copy_(dev_tensor(np.asarray(gamma, dtype=np.float32)))
    else:
        gd = dev_tensor(np.asarray(gamma, dtype=np.float32))
    auxd = dev_tensor(np.asarray(aux, dtype=np.float32).reshape(-1)) if aux is not None else None
    dst = auxd if epi == ogemv.EPI_ADD else _nan_out(ncols * M)
    path, info = G.plan(Wd, wt, xd, M, K, epi, auxd, dst, ncols=ncols, rms_norm_weight=gd, rms_norm_eps=eps, **kw)
    G.gemv_fused_ex(Wd, wt, xd, M, K, epi, auxd if epi in ogemv.NEEDS_AUX else None, dst, ncols=ncols,
                    rms_norm_weight=gd, rms_norm_eps=eps, **kw)
    torch.cuda.synchronize()
    return _cpu(dst, ncols, M), path, info


def _norm_case(wt, M, K, ncols, seed, x_scale=3.0):
    raw = synth.weights(wt, M, K, seed=seed)
    X = (synth.normal(ncols * K, seed=seed + 1) * x_scale).reshape(ncols, K)
    gamma = 1.0 + 0.1 * synth.normal(K, seed=seed + 2)
    aux = synth.normal(ncols * M, seed=seed + 3).reshape(ncols, M)
    return raw, X, gamma, aux


@pytest.mark.parametrize("wt", ALL_WT)
@pytest.mark.parametrize("epi", EPIS)
def test_rms_norm_prologue_formats_and_tails(G, wt, epi):
    M, K, eps = 700, 4096, 1e-6
    raw, X, gamma, aux = _norm_case(wt, M, K, 1, 300 + wt)
    got, path, _ = run_norm(G, raw, wt, X, gamma, eps, M, K, epi, aux)
    assert path == G.PATH_STREAM
    Xn = onorm.rms_norm(X, gamma, eps, K)
    want = ogemv.gemv(raw, wt, Xn, M, K, epi, aux)
    assert_within(got, want, norm_bound(raw, wt, Xn, M, K), "rms wt %d epi %d" % (wt, epi))


@pytest.mark.parametrize("ncols,eps,x_scale", [(3, 1e-5, 1.0), (8, 0.0, 50.0), (1, 10.0, 0.01)])
def test_rms_norm_batch_and_eps(G, ncols, eps, x_scale):
    wt, M, K = synth.F16, 1100, 5120
    raw, X, gamma, aux = _norm_case(wt, M, K, ncols, 320, x_scale)
    got, _, _ = run_norm(G, raw, wt, X, gamma, eps, M, K, ogemv.EPI_ADD, aux, ncols=ncols)
    Xn = onorm.rms_norm(X, gamma, eps, K)
    want = ogemv.gemv(raw, wt, Xn, M, K, ogemv.EPI_ADD, aux)
    assert_within(got, want, norm_bound(raw, wt, Xn, M, K), "rms batch")


@pytest.mark.parametrize("wt,K,gamma_offset", [(synth.F16, 4096, 1), (synth.F16, 36, 0), (synth.Q4_0, 96, 0)])
def test_rms_norm_generic_path(G, wt, K, gamma_offset):
    M = 90
    raw, X, gamma, aux = _norm_case(wt, M, K, 2, 330)
    got, path, _ = run_norm(G, raw, wt, X, gamma, 1e-6, M, K, ogemv.EPI_SILU_MUL, aux, ncols=2,
                            gamma_offset=gamma_offset)
    assert path == G.PATH_GENERIC
    Xn = onorm.rms_norm(X, gamma, 1e-6, K)
    want = ogemv.gemv(raw, wt, Xn, M, K, ogemv.EPI_SILU_MUL, aux)
    assert_within(got, want, norm_bound(raw, wt, Xn, M, K), "rms generic")


def test_rms_norm_with_glu(G):
    wt, M, K, eps = synth.Q4_0, 900, 4096, 1e-6
    rg, ru = synth.weights(wt, M, K, seed=340), synth.weights(wt, M, K, seed=341)
    X = (synth.normal(2 * K, seed=342) * 2.0).reshape(2, K)
    gamma = 1.0 + 0.1 * synth.normal(K, seed=343)
    gd = dev_tensor(gamma.astype(np.float32))
    got, path, _ = run_glu(G, rg, ru, wt, X, M, K, ncols=2, rms_norm_weight=gd, rms_norm_eps=eps)
    assert path == G.PATH_STREAM
    Xn = onorm.rms_norm(X, gamma, eps, K)
    want = ogemv.gemv_glu(rg, ru, wt, Xn, M, K)
    assert_within(got, want, glu_bound(rg, ru, wt, Xn, M, K, extra_rel=TOL_NORM_REL), "rms + glu")


# ----------------------------------------------------------------------------- split K

@pytest.mark.parametrize("wt", ALL_WT)
@pytest.mark.parametrize("M,K", [(1, 32768), (7, 65536), (32, 32768), (76, 32768), (19, 40960), (32, 4096)])
def test_split_k_matches_oracle(G, wt, M, K):
    raw = synth.weights(wt, M, K, seed=400 + wt)
    x = synth.normal(K, seed=401)
    aux = synth.normal(M, seed=402)
    Wd, xd = dev_tensor(raw), dev_tensor(x)
    outs = {}
    for split in (True, False):
        r = dev_tensor(aux)
        _, info = G.plan(Wd, wt, xd, M, K, ogemv.EPI_ADD, r, r, split_k=split)
        outs[split] = info["split"]
        G.gemv_fused_ex(Wd, wt, xd, M, K, ogemv.EPI_ADD, r, r, split_k=split, pdl=split)
        torch.cuda.synchronize()
        got = r.cpu().numpy().astype(np.float64)
        want = ogemv.gemv(raw, wt, x, M, K, ogemv.EPI_ADD, aux)[0]
        assert_within(got, want, gemv_bound(raw, wt, x, M, K)[0], "split=%s wt %d %dx%d" % (split, wt, M, K))
    assert outs[False] == 1
    assert outs[True] > 1 or K * 4 < 128 * 1024  # split only with >= 128 KB of x per CTA


@pytest.mark.parametrize("epi", EPIS)
def test_split_k_tails_and_batch(G, epi):
    wt, M, K, ncols = synth.Q4_0, 32, 16384, 3
    raw = synth.weights(wt, M, K, seed=410)
    X = synth.normal(ncols * K, seed=411).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=412).reshape(ncols, M)
    Wd, xd = dev_tensor(raw), dev_tensor(X.reshape(-1))
    auxd = dev_tensor(aux.reshape(-1))
    dst = auxd if epi == ogemv.EPI_ADD else _nan_out(ncols * M)
    _, info = G.plan(Wd, wt, xd, M, K, epi, auxd, dst, ncols=ncols)
    assert info["split"] == 4
    G.gemv_fused_ex(Wd, wt, xd, M, K, epi, auxd if epi in ogemv.NEEDS_AUX else None, dst, ncols=ncols)
    torch.cuda.synchronize()
    want = ogemv.gemv(raw, wt, X, M, K, epi, aux)
    assert_within(_cpu(dst, ncols, M), want, gemv_bound(raw, wt, X, M, K), "split tails")


def test_split_k_with_fwht_on_chip(G):
    wt, M, K, B = synth.F16, 32, 40960, 1024
    raw = synth.weights(wt, M, K, seed=420)
    x = synth.normal(K, seed=421)
    s = synth.rademacher(B, seed=422)
    Wd, xd, sd = dev_tensor(raw), dev_tensor(x), dev_tensor(s)
    dst = _nan_out(M)
    _, info = G.plan(Wd, wt, xd, M, K, 0, None, dst, fwht_signs=sd, fwht_block=B)
    assert info["split"] == 4
    G.gemv_fused_ex(Wd, wt, xd, M, K, 0, None, dst, fwht_signs=sd, fwht_block=B)
    torch.cuda.synchronize()
    xp = ofwht.fwht_signed(x, s, B)
    want = ogemv.gemv(raw, wt, xp, M, K)
    bound = gemv_bound(raw, wt, xp, M, K, x_err=fwht_err_bound(x, B))
    assert_within(_cpu(dst, 1, M), want, bound, "split + fwht")


def test_split_k_glu_and_rms_norm(G):
    wt, M, K, eps = synth.Q8_0, 24, 32768, 1e-5
    rg, ru = synth.weights(wt, M, K, seed=430), synth.weights(wt, M, K, seed=431)
    X = synth.normal(K, seed=432).reshape(1, K)
    gamma = 1.0 + 0.1 * synth.normal(K, seed=433)
    got, _, info = run_glu(G, rg, ru, wt, X, M, K, rms_norm_weight=dev_tensor(gamma.astype(np.float32)),
                           rms_norm_eps=eps)
    assert info["split"] > 1  # the largest split whose clusters all fit (5 or 6 here)
    Xn = onorm.rms_norm(X, gamma, eps, K)
    want = ogemv.gemv_glu(rg, ru, wt, Xn, M, K)
    assert_within(got, want, glu_bound(rg, ru, wt, Xn, M, K, extra_rel=TOL_NORM_REL), "split glu rms")


def test_split_k_deterministic(G):
    wt, M, K = synth.Q4_0, 32, 32768
    raw = synth.weights(wt, M, K, seed=440)
    x = synth.normal(K, seed=441)
    Wd, xd = dev_tensor(raw), dev_tensor(x)
    outs = []
    for _ in range(3):
        d = _nan_out(M)
        G.gemv_fused_ex(Wd, wt, xd, M, K, ogemv.EPI_SIGMOID, None, d, pdl=True)
        torch.cuda.synchronize()
        outs.append(d.cpu().numpy())
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


# ----------------------------------------------------------------------------- batches wider than 8

@pytest.mark.parametrize("wt,ncols", [(synth.F16, 9), (synth.Q4_0, 16), (synth.Q8_0, 33), (synth.Q4_K, 12)])
def test_wide_batch_add_in_place(G, wt, ncols):
    M, K = 300, 2048
    raw = synth.weights(wt, M, K, seed=600 + ncols)
    X = synth.normal(ncols * K, seed=601).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=602).reshape(ncols, M)
    Wd, xd, r = dev_tensor(raw), dev_tensor(X.reshape(-1)), dev_tensor(aux.reshape(-1))
    G.gemv_fused_ex(Wd, wt, xd, M, K, ogemv.EPI_ADD, r, r, ncols=ncols, pdl=True)
    torch.cuda.synchronize()
    want = ogemv.gemv(raw, wt, X, M, K, ogemv.EPI_ADD, aux)
    assert_within(_cpu(r, ncols, M), want, gemv_bound(raw, wt, X, M, K), "wide batch %d" % ncols)


def test_wide_batch_fwht_workspace_and_glu_rms(G):
    wt, M, K, B, ncols = synth.F16, 256, 5120, 1024, 20
    raw = synth.weights(wt, M, K, seed=610)
    X = synth.normal(ncols * K, seed=611).reshape(ncols, K)
    s = synth.rademacher(B, seed=612)
    xd, sd = dev_tensor(X.reshape(-1)), dev_tensor(s)
    ws = torch.empty(ncols * K, device="cuda")
    dst = _nan_out(ncols * M)
    G.gemv_fused_ex(dev_tensor(raw), wt, xd, M, K, ogemv.EPI_SIGMOID, None, dst, ncols=ncols, fwht_signs=sd,
                    fwht_block=B, fwht_workspace=ws)
    torch.cuda.synchronize()
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, wt, Xp, M, K, ogemv.EPI_SIGMOID)
    assert_within(_cpu(dst, ncols, M), want, gemv_bound(raw, wt, Xp, M, K, x_err=E), "wide fwht ws")
    # gated dual GEMV with the RMS prologue over 11 columns
    rg, ru = synth.weights(synth.Q4_0, M, 4096, seed=613), synth.weights(synth.Q4_0, M, 4096, seed=614)
    X2 = synth.normal(11 * 4096, seed=615).reshape(11, 4096)
    gamma = 1.0 + 0.1 * synth.normal(4096, seed=616)
    got, _, _ = run_glu(G, rg, ru, synth.Q4_0, X2, M, 4096, ncols=11,
                        rms_norm_weight=dev_tensor(gamma.astype(np.float32)), rms_norm_eps=1e-6)
    Xn = onorm.rms_norm(X2, gamma, 1e-6, 4096)
    want = ogemv.gemv_glu(rg, ru, synth.Q4_0, Xn, M, 4096)
    assert_within(got, want, glu_bound(rg, ru, synth.Q4_0, Xn, M, 4096, extra_rel=TOL_NORM_REL), "wide glu rms")
