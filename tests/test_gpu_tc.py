"""GPU parity of the tensor-core GEMV (F16 weights, batches of 3..16 columns per launch)
through the C ABI against the fp64 oracle, within 2e-5 * sum_k |W_ik x_k| + 1e-6: x
enters as scaled f16 hi + lo parts (about 2^-22 relative), f16 products are exact and
the accumulation is fp32.  Covers ragged tiles, split K, every tail, wide dynamic
ranges of x (the per-column power-of-two scale), determinism, the transform-once
prologue and agreement with the CUDA-core kernels."""

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

F16 = synth.F16
EPIS = [ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD]


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def run(G, raw, X, M, K, epi, aux=None, expect_path=None, **kw):
    ncols = X.shape[0]
    Wd = dev_tensor(raw)
    xd = dev_tensor(X.astype(np.float32).reshape(-1))
    auxd = dev_tensor(aux.astype(np.float32).reshape(-1)) if aux is not None else None
    dst = auxd if epi == ogemv.EPI_ADD else torch.full((ncols * M,), float("nan"), device="cuda")
    path, info = G.plan(Wd, F16, xd, M, K, epi, auxd, dst, ncols=ncols, **kw)
    if expect_path is not None:
        assert path == expect_path, (path, info)
    G.gemv_fused_ex(Wd, F16, xd, M, K, epi, auxd if epi in ogemv.NEEDS_AUX else None, dst, ncols=ncols, **kw)
    torch.cuda.synchronize()
    return dst.cpu().numpy().astype(np.float64).reshape(ncols, M), info


@pytest.mark.parametrize("M,K,ncols", [(128, 64, 4), (100, 4096, 8), (333, 1024, 5), (1000, 2048, 16), (200, 2048, 3),
                                       (4096, 512, 8), (640, 8192, 64), (257, 4096, 36)])
def test_tc_shapes(G, M, K, ncols):
    raw = synth.weights(F16, M, K, seed=700 + ncols)
    X = synth.normal(ncols * K, seed=701).reshape(ncols, K)
    got, info = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC)
    want = ogemv.gemv(raw, F16, X, M, K)
    assert_within(got, want, gemv_bound(raw, F16, X, M, K), "tc %dx%d n%d split %d" % (M, K, ncols, info["split"]))


@pytest.mark.parametrize("epi", EPIS)
def test_tc_tails(G, epi):
    M, K, ncols = 700, 2048, 8
    raw = synth.weights(F16, M, K, seed=710)
    X = synth.normal(ncols * K, seed=711).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=712).reshape(ncols, M)
    got, _ = run(G, raw, X, M, K, epi, aux, expect_path=G.PATH_TC, view=(7, 100) if epi == ogemv.EPI_ADD else None)
    want = ogemv.gemv(raw, F16, X, M, K, epi, aux)
    assert_within(got, want, gemv_bound(raw, F16, X, M, K), "tc tail %d" % epi)


def test_tc_dynamic_range_of_x(G):
    # per column: all zero, huge, tiny, mixed magnitudes, a single spike
    M, K, ncols = 384, 4096, 6
    raw = synth.weights(F16, M, K, seed=720)
    base = synth.normal(ncols * K, seed=721).reshape(ncols, K)
    X = np.zeros((ncols, K))
    X[1] = base[1] * 3.0e4
    X[2] = base[2] * 1.0e-20
    X[3] = base[3] * np.where(np.arange(K) % 7 == 0, 1e3, 1e-3)
    X[4, 1234] = 77.0
    X[5] = base[5]
    got, _ = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC)
    want = ogemv.gemv(raw, F16, X, M, K)
    assert_within(got, want, gemv_bound(raw, F16, X, M, K), "tc dynamic range")
    assert np.all(got[0] == 0.0)


def test_tc_split_matches_unsplit_and_cuda_cores(G):
    M, K, ncols = 512, 8192, 8
    raw = synth.weights(F16, M, K, seed=730)
    X = synth.normal(ncols * K, seed=731).reshape(ncols, K)
    want = ogemv.gemv(raw, F16, X, M, K)
    bound = gemv_bound(raw, F16, X, M, K)
    got_split, info = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC)
    assert info["split"] > 1
    got_one, info1 = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC, split_k=False)
    got_cc, _ = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_STREAM, tensor_cores=False)
    for got, what in ((got_split, "split"), (got_one, "one CTA per tile"), (got_cc, "cuda cores")):
        assert_within(got, want, bound, what)


def test_tc_deterministic(G):
    M, K, ncols = 5120, 5120, 8
    raw = synth.weights(F16, M, K, seed=740)
    X = synth.normal(ncols * K, seed=741).reshape(ncols, K)
    a, _ = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC, pdl=True)
    b, _ = run(G, raw, X, M, K, ogemv.EPI_NONE, expect_path=G.PATH_TC)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("ncols", [3, 4, 8, 12, 16])  # 12, 16: x by one 2-D copy per stage
def test_tc_full_fwht_f16_5120_workspace(G, ncols):
    M, K, B = 5120, 5120, 1024
    raw = synth.weights(F16, M, K, seed=750)
    X = synth.normal(ncols * K, seed=751).reshape(ncols, K)
    r = synth.normal(ncols * M, seed=752).reshape(ncols, M)
    s = synth.rademacher(B, seed=753)
    ws = torch.empty(ncols * K, device="cuda")
    got, _ = run(G, raw, X, M, K, ogemv.EPI_ADD, r, expect_path=G.PATH_TC, fwht_signs=dev_tensor(s), fwht_block=B,
                 fwht_workspace=ws, pdl=True)
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, F16, Xp, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, gemv_bound(raw, F16, Xp, M, K, x_err=E), "tc fwht ws")


def test_tc_wide_batch_blocks_of_16(G):
    M, K, ncols = 256, 1024, 100
    raw = synth.weights(F16, M, K, seed=760)
    X = synth.normal(ncols * K, seed=761).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=762).reshape(ncols, M)
    got, _ = run(G, raw, X, M, K, ogemv.EPI_SILU_MUL, aux, expect_path=G.PATH_TC)
    want = ogemv.gemv(raw, F16, X, M, K, ogemv.EPI_SILU_MUL, aux)
    assert_within(got, want, gemv_bound(raw, F16, X, M, K), "tc 100 columns")


@pytest.mark.parametrize("ncols", [3, 8, 13, 16])
@pytest.mark.parametrize("epi", [ogemv.EPI_ADD, ogemv.EPI_SILU_MUL])
def test_tc_every_split_width(G, ncols, epi):
    """Row counts that give every cluster size the planner can pick (1..8 CTAs splitting K;
    ragged last tiles), each with the batch widths whose column owners (column c belongs
    to rank c % S) wrap differently: the split-K exchange and the per-rank tails."""
    K = 1024
    seen = set()
    for M in (10240, 8192, 5184, 4196, 3800, 3100, 2600, 1000):
        raw = synth.weights(F16, M, K, seed=770 + M % 97)
        X = synth.normal(ncols * K, seed=771 + M % 89).reshape(ncols, K)
        aux = synth.normal(ncols * M, seed=772 + M % 83).reshape(ncols, M)
        got, info = run(G, raw, X, M, K, epi, aux, expect_path=G.PATH_TC)
        seen.add(info["split"])
        want = ogemv.gemv(raw, F16, X, M, K, epi, aux)
        assert_within(got, want, gemv_bound(raw, F16, X, M, K),
                      "tc %dx%d n%d split %d epi %d" % (M, K, ncols, info["split"], epi))
    assert {1, 2, 8} <= seen and len(seen) >= 5, seen


def test_tc_with_staging_copies_through_launch_prepared(G):
    """Upload, the 8-column tensor-core call with its transform, download: issued with
    gf_launch_prepared (no graph), twice with new host inputs."""
    M, K, B, nc = 1000, 4096, 1024, 8
    raw = synth.weights(F16, M, K, seed=780)
    Wd = dev_tensor(raw)
    s = synth.rademacher(B, seed=781)
    sd = dev_tensor(s)
    xh = torch.empty(nc * K, dtype=torch.float32).pin_memory()
    rh = torch.empty(nc * M, dtype=torch.float32).pin_memory()
    yh = torch.empty(nc * M, dtype=torch.float32).pin_memory()
    xd, rd, ws = (torch.empty(nc * K, device="cuda"), torch.empty(nc * M, device="cuda"),
                  torch.empty(nc * K, device="cuda"))
    calls = [G.prepare_copy(xd, xh, 4 * nc * K), G.prepare_copy(rd, rh, 4 * nc * M, pdl=True),
             G.prepare(Wd, F16, xd, M, K, ogemv.EPI_ADD, rd, rd, ncols=nc, fwht_signs=sd, fwht_block=B,
                       fwht_workspace=ws, pdl=True),
             G.prepare_copy(yh, rd, 4 * nc * M, pdl=True)]
    for step in range(2):
        X = synth.normal(nc * K, seed=782 + step).reshape(nc, K)
        R = synth.normal(nc * M, seed=784 + step).reshape(nc, M)
        xh.copy_(torch.from_numpy(X.astype(np.float32).reshape(-1)))
        rh.copy_(torch.from_numpy(R.astype(np.float32).reshape(-1)))
        G.launch_prepared(calls)
        torch.cuda.synchronize()
        Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(nc)])
        E = np.stack([fwht_err_bound(X[c], B) for c in range(nc)])
        want = ogemv.gemv(raw, F16, Xp, M, K, ogemv.EPI_ADD, R)
        assert_within(yh.numpy().astype(np.float64).reshape(nc, M), want,
                      gemv_bound(raw, F16, Xp, M, K, x_err=E), "step %d" % step)
