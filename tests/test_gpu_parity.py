"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by
element, on seeded inputs.  Bit-exact for decoded weights; within
2e-5 * sum_k |W_ik x_k| + 1e-6 for outputs (plus the propagated prologue error where
the signed FWHT runs on chip)."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, fwht_err_bound, gemv_bound, glu_bound
from oracle import chain as ochain
from oracle import fwht as ofwht
from oracle import gemv as ogemv
from oracle import quant as oquant

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

WT_NAMES = {synth.F32: "f32", synth.F16: "f16", synth.Q8_0: "q8_0", synth.Q4_0: "q4_0"}
EPIS = [ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD]


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def run_gemv(G, raw, wt, x, M, K, epi, aux=None, ncols=1, signs=None, block=0, view=None,
             w_offset=0, pdl=False, tensor_cores=True):
    """Upload, call gemv_fused_ex, return dst as float64 [ncols, M] and the plan path."""
    if w_offset:
        buf = torch.zeros(raw.size + 64, dtype=torch.uint8, device="cuda")
        Wd = buf[w_offset:w_offset + raw.size]
        Wd.copy_(dev_tensor(raw))
    else:
        Wd = dev_tensor(raw)
    xd = dev_tensor(np.asarray(x, dtype=np.float32).reshape(-1))
    auxd = dev_tensor(np.asarray(aux, dtype=np.float32).reshape(-1)) if aux is not None else None
    if epi == ogemv.EPI_ADD:
        dst = auxd  # residual add in place
    else:
        dst = torch.full((ncols * M,), float("nan"), device="cuda")
    sd = dev_tensor(signs) if signs is not None else None
    path, _ = G.plan(Wd, wt, xd, M, K, epi, auxd, dst, ncols=ncols, fwht_signs=sd, fwht_block=block,
                     tensor_cores=tensor_cores)
    G.gemv_fused_ex(Wd, wt, xd, M, K, epi, auxd if epi in ogemv.NEEDS_AUX else None, dst,
                    ncols=ncols, fwht_signs=sd, fwht_block=block, view=view, pdl=pdl, tensor_cores=tensor_cores)
    torch.cuda.synchronize()
    return dst.cpu().numpy().astype(np.float64).reshape(ncols, M), path


# ----------------------------------------------------------------------------- decoders

@pytest.mark.parametrize("wt,M,K", [
    (synth.Q4_0, 64, 4096), (synth.Q4_0, 3, 96), (synth.Q4_0, 1, 32),
    (synth.Q8_0, 64, 4096), (synth.Q8_0, 5, 160),
    (synth.F16, 8, 4096), (synth.F16, 3, 33),
    (synth.F32, 4, 512), (synth.F32, 4, 12),
])
def test_dequantize_bit_exact(G, wt, M, K):
    raw = synth.weights(wt, M, K, seed=10 + wt)
    out = torch.empty(M * K, device="cuda")
    G.dequantize(dev_tensor(raw), wt, M, K, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().reshape(M, K)
    want = oquant.dequantize(raw, wt, M, K).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequantize_golden_blocks(G):
    from conftest import read_golden
    g = read_golden("q4_0_block.txt")
    raw = np.concatenate([np.array([int(t, 16) for t in b], dtype=np.uint8) for b in g["bytes"]])
    out = torch.empty(96, device="cuda")
    G.dequantize(dev_tensor(raw), synth.Q4_0, 1, 96, out)
    torch.cuda.synchronize()
    want = np.concatenate([[float(t) for t in v] for v in g["values"]]).astype(np.float32)
    assert np.array_equal(out.cpu().numpy(), want)


# ----------------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("epi", EPIS)
def test_small_f32_all_epilogues(G, epi):
    """f32 M=256, K=512: W ~ U(+-1/sqrt K), x, m, r ~ N(0,1), seed 0; each tail."""
    M, K = 256, 512
    raw = synth.weights(synth.F32, M, K, seed=0)
    x = synth.normal(K, seed=1)
    aux = synth.normal(M, seed=2)
    got, path = run_gemv(G, raw, synth.F32, x, M, K, epi, aux)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, synth.F32, x, M, K, epi, aux)
    assert_within(got, want, gemv_bound(raw, synth.F32, x, M, K), "f32 epi %d" % epi)


@pytest.mark.parametrize("wt", [synth.F32, synth.F16, synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("epi", EPIS)
def test_formats_tiles_and_ragged_rows(G, wt, epi):
    """M = 611 rows spread over 152 CTAs (4-5 rows each, ragged last tile), K = 1024."""
    M, K = 611, 1024
    raw = synth.weights(wt, M, K, seed=20 + wt)
    x = synth.normal(K, seed=30)
    aux = synth.normal(M, seed=31)
    got, path = run_gemv(G, raw, wt, x, M, K, epi, aux)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, wt, x, M, K, epi, aux)
    assert_within(got, want, gemv_bound(raw, wt, x, M, K), "%s epi %d" % (WT_NAMES[wt], epi))


@pytest.mark.parametrize("wt,M,K,w_offset,expect_path", [
    (synth.F32, 37, 33, 0, 2),       # ragged K
    (synth.F16, 19, 36, 0, 2),       # K % 8 != 0
    (synth.F16, 45, 1024, 2, 2),     # W only 2-byte aligned
    (synth.Q4_0, 29, 96, 0, 2),      # row bytes 54, not a multiple of 16
    (synth.Q8_0, 13, 224, 0, 2),     # row bytes 238
    (synth.Q4_0, 1, 4096, 0, 1),     # a single row
    (synth.F32, 5, 16, 0, 1),        # smallest K of the streamed kernel
    (synth.F32, 5, 8, 0, 2),         # below one 16-weight unit
    (synth.Q4_0, 300, 32, 0, 2),     # one block per row
])
def test_edge_shapes_and_paths(G, wt, M, K, w_offset, expect_path):
    raw = synth.weights(wt, M, K, seed=40)
    x = synth.normal(K, seed=41)
    aux = synth.normal(M, seed=42)
    for epi in (ogemv.EPI_NONE, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD):
        got, path = run_gemv(G, raw, wt, x, M, K, epi, aux, w_offset=w_offset)
        assert path == expect_path
        want = ogemv.gemv(raw, wt, x, M, K, epi, aux)
        assert_within(got, want, gemv_bound(raw, wt, x, M, K), "%s %dx%d" % (WT_NAMES[wt], M, K))


def test_k_zero_gives_tail_of_zero(G):
    M = 40
    aux = synth.normal(M, seed=43)
    for epi in EPIS:
        got, _ = run_gemv(G, np.zeros(0, np.uint8), synth.F16, np.zeros(0, np.float32), M, 0, epi, aux)
        want = ogemv.apply_epilogue(np.zeros((1, M)), epi, aux.reshape(1, M).astype(np.float64)
                                    if epi in ogemv.NEEDS_AUX else None)
        assert_within(got, want, np.full((1, M), 1e-6), "K=0 epi %d" % epi)


def test_m_zero_launches_nothing(G):
    assert G.gemv_fused(None, synth.F16, None, 0, 4096, ogemv.EPI_NONE, None, None) == 0


def test_many_rows_per_cta_row_chunks(G):
    """M = 65536, K = 256: 431 rows per CTA, more than one finalize chunk."""
    M, K = 65536, 256
    raw = synth.weights(synth.F16, M, K, seed=44)
    x = synth.normal(K, seed=45)
    r = synth.normal(M, seed=46)
    got, path = run_gemv(G, raw, synth.F16, x, M, K, ogemv.EPI_ADD, r)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, synth.F16, x, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, gemv_bound(raw, synth.F16, x, M, K), "row chunks")


def test_k_chunks_f32_long_rows(G):
    """f32 K = 14336 (57 KB rows) is streamed in two K chunks."""
    M, K = 300, 14336
    raw = synth.weights(synth.F32, M, K, seed=47)
    x = synth.normal(K, seed=48)
    m = synth.normal(M, seed=49)
    got, path = run_gemv(G, raw, synth.F32, x, M, K, ogemv.EPI_SILU_MUL, m)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, synth.F32, x, M, K, ogemv.EPI_SILU_MUL, m)
    assert_within(got, want, gemv_bound(raw, synth.F32, x, M, K), "f32 K chunks")


@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("wt", [synth.F16, synth.Q4_0])
def test_ncols_batch(G, ncols, wt):
    M, K = 333, 2048
    raw = synth.weights(wt, M, K, seed=50)
    X = synth.normal(ncols * K, seed=51).reshape(ncols, K)
    aux = synth.normal(ncols * M, seed=52).reshape(ncols, M)
    want = ogemv.gemv(raw, wt, X, M, K, ogemv.EPI_SILU_MUL, aux)
    for tc in (True, False):  # F16 batches default to the tensor cores
        got, path = run_gemv(G, raw, wt, X, M, K, ogemv.EPI_SILU_MUL, aux, ncols=ncols, tensor_cores=tc)
        assert path == (G.PATH_TC if tc and wt == synth.F16 and ncols >= 3 else G.PATH_STREAM)
        assert_within(got, want, gemv_bound(raw, wt, X, M, K), "ncols %d tc %s" % (ncols, tc))


# ----------------------------------------------------------------------------- signed FWHT

@pytest.mark.parametrize("n,block,nsigns", [(5120, 1024, 1024), (40960, 1024, 1024), (4096, 64, 64),
                                             (1024, 1024, 256), (12, 4, 4), (8, 1, 1), (16384, 16384, 16384),
                                             (8192, 2, 2)])
def test_fwht_signed_standalone(G, n, block, nsigns):
    x = synth.normal(n, seed=60)
    s = synth.rademacher(nsigns, seed=61)
    out = torch.empty(n, device="cuda")
    G.fwht_signed(dev_tensor(x), dev_tensor(s), out, n, block, nsigns)
    torch.cuda.synchronize()
    want = ofwht.fwht_signed(x, s, block)
    assert_within(out.cpu().numpy(), want, fwht_err_bound(x, block), "fwht n=%d B=%d" % (n, block))


def test_fwht_in_place_and_unsigned(G):
    n, B = 8192, 1024
    x = synth.normal(n, seed=62)
    xd = dev_tensor(x)
    G.fwht_signed(xd, None, xd, n, B)
    torch.cuda.synchronize()
    assert_within(xd.cpu().numpy(), ofwht.fwht_signed(x, None, B), fwht_err_bound(x, B), "in place")


def test_fwht_golden_worked_example(G):
    from conftest import read_golden
    g = read_golden("fwht_signed_b4.txt")
    f = lambda k: np.array([float(t) for t in g[k][0]], dtype=np.float32)
    out = torch.empty(8, device="cuda")
    G.fwht_signed(dev_tensor(f("x2")), dev_tensor(f("signs")), out, 8, 4, 4)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), f("out2"))


@pytest.mark.parametrize("ncols", [1, 2, 5, 8])
def test_fused_fwht_prologue(G, ncols):
    """x' = H (x*s)/sqrt(B) per 1024 block on chip, then F16 GEMV + in-place residual."""
    M, K, B = 400, 5120, 1024
    raw = synth.weights(synth.F16, M, K, seed=70)
    X = synth.normal(ncols * K, seed=71).reshape(ncols, K)
    s = synth.rademacher(B, seed=72)
    r = synth.normal(ncols * M, seed=73).reshape(ncols, M)
    got, path = run_gemv(G, raw, synth.F16, X, M, K, ogemv.EPI_ADD, r, ncols=ncols, signs=s, block=B)
    assert path == G.PATH_STREAM
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, synth.F16, Xp, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, gemv_bound(raw, synth.F16, Xp, M, K, x_err=E), "fwht+gemv ncols %d" % ncols)


@pytest.mark.parametrize("ncols", [1, 3, 8])
def test_fwht_workspace_path_matches_on_chip_prologue(G, ncols):
    """The transform-once path (stand-alone signed FWHT into a workspace, then the GEMV,
    chained with programmatic dependent launch) gives the same x' and therefore, on the
    same CUDA-core kernel, the same outputs as the on-chip prologue, bit for bit; with
    the tensor cores (batches) it passes the oracle bound."""
    M, K, B = 700, 5120, 1024
    raw = synth.weights(synth.F16, M, K, seed=90)
    X = synth.normal(ncols * K, seed=91).reshape(ncols, K)
    s = synth.rademacher(B, seed=92)
    r = synth.normal(ncols * M, seed=93).reshape(ncols, M)
    Wd, xd, sd = dev_tensor(raw), dev_tensor(X.reshape(-1)), dev_tensor(s)
    ws = torch.full((ncols * K,), float("nan"), device="cuda")
    d_chip = dev_tensor(r.reshape(-1))
    d_ws = dev_tensor(r.reshape(-1))
    G.gemv_fused_ex(Wd, synth.F16, xd, M, K, ogemv.EPI_ADD, d_chip, d_chip, ncols=ncols, fwht_signs=sd, fwht_block=B)
    d_tc = dev_tensor(r.reshape(-1))
    G.gemv_fused_ex(Wd, synth.F16, xd, M, K, ogemv.EPI_ADD, d_ws, d_ws, ncols=ncols, fwht_signs=sd, fwht_block=B,
                    fwht_workspace=ws, tensor_cores=False)
    G.gemv_fused_ex(Wd, synth.F16, xd, M, K, ogemv.EPI_ADD, d_tc, d_tc, ncols=ncols, fwht_signs=sd, fwht_block=B,
                    fwht_workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(d_chip.view(torch.int32), d_ws.view(torch.int32))
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    assert_within(ws.cpu().numpy().reshape(ncols, K), Xp, E, "workspace x'")
    want = ogemv.gemv(raw, synth.F16, Xp, M, K, ogemv.EPI_ADD, r)
    for d, what in ((d_ws, "workspace path"), (d_tc, "workspace path, default kernel")):
        got = d.cpu().numpy().astype(np.float64).reshape(ncols, M)
        assert_within(got, want, gemv_bound(raw, synth.F16, Xp, M, K, x_err=E), "%s ncols %d" % (what, ncols))


@pytest.mark.parametrize("wt,block,nsigns", [(synth.Q4_0, 256, 256), (synth.F32, 64, 32), (synth.F16, 8192, 8192),
                                             (synth.Q8_0, 1, 1)])
def test_fused_fwht_other_blocks(G, wt, block, nsigns):
    M, K = 150, 8192
    raw = synth.weights(wt, M, K, seed=74)
    x = synth.normal(K, seed=75)
    s = synth.rademacher(nsigns, seed=76)
    got, _ = run_gemv(G, raw, wt, x, M, K, ogemv.EPI_NONE, None, signs=s, block=block)
    xp = ofwht.fwht_signed(x, s, block)
    want = ogemv.gemv(raw, wt, xp, M, K)
    assert_within(got, want, gemv_bound(raw, wt, xp, M, K, x_err=fwht_err_bound(x, block)),
                  "fwht B=%d" % block)


# ----------------------------------------------------------------------------- fused vs unfused

def _unfused(G, Wd, wt, xd, M, K, epi, auxd):
    y = torch.empty(M, device="cuda")
    G.gemv_fused(Wd, wt, xd, M, K, ogemv.EPI_NONE, None, y)
    out = torch.empty(M, device="cuda")
    if epi == ogemv.EPI_NONE:
        out.copy_(y)
    elif epi == ogemv.EPI_SIGMOID:
        G.elementwise(G.EW_SIGMOID, y, None, out, M)
    elif epi == ogemv.EPI_SILU:
        G.elementwise(G.EW_SILU, y, None, out, M)
    elif epi == ogemv.EPI_SILU_MUL:
        G.elementwise(G.EW_SILU, y, None, out, M)
        G.elementwise(G.EW_MUL, out, auxd, out, M)
    else:
        G.elementwise(G.EW_ADD, y, auxd, out, M)
    return out


@pytest.mark.parametrize("wt", [synth.F16, synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("epi", EPIS)
def test_fused_equals_unfused_bitwise(G, wt, epi):
    """The fused tail reads the same values the separate passes would: bit-identical."""
    M, K = 1000, 2048
    Wd = dev_tensor(synth.weights(wt, M, K, seed=80))
    xd = dev_tensor(synth.normal(K, seed=81))
    auxd = dev_tensor(synth.normal(M, seed=82))
    ref = _unfused(G, Wd, wt, xd, M, K, epi, auxd)
    dst = auxd.clone() if epi == ogemv.EPI_ADD else torch.empty(M, device="cuda")
    G.gemv_fused(Wd, wt, xd, M, K, epi, dst if epi == ogemv.EPI_ADD else auxd, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst.view(torch.int32), ref.view(torch.int32))


def test_signed_fwht_fused_equals_unfused_bitwise(G):
    """Sign multiply then plain FWHT (two kernels) == signed FWHT (one) == on-chip prologue."""
    M, K, B = 500, 5120, 1024
    Wd = dev_tensor(synth.weights(synth.F16, M, K, seed=83))
    x = dev_tensor(synth.normal(K, seed=84))
    s = dev_tensor(synth.rademacher(B, seed=85))
    t = torch.empty(K, device="cuda")
    G.elementwise(G.EW_MUL, x, s, t, K, nb=B)
    xp_unfused = torch.empty(K, device="cuda")
    G.fwht_signed(t, None, xp_unfused, K, B)
    xp = torch.empty(K, device="cuda")
    G.fwht_signed(x, s, xp, K, B)
    torch.cuda.synchronize()
    assert torch.equal(xp.view(torch.int32), xp_unfused.view(torch.int32))
    y_two = torch.empty(M, device="cuda")
    G.gemv_fused(Wd, synth.F16, xp, M, K, ogemv.EPI_NONE, None, y_two)
    y_one = torch.empty(M, device="cuda")
    G.gemv_fused_ex(Wd, synth.F16, x, M, K, ogemv.EPI_NONE, None, y_one, fwht_signs=s, fwht_block=B)
    torch.cuda.synchronize()
    assert torch.equal(y_one.view(torch.int32), y_two.view(torch.int32))


def test_deterministic_and_stream_argument(G):
    M, K = 4096, 4096
    Wd = dev_tensor(synth.weights(synth.Q4_0, M, K, seed=86))
    xd = dev_tensor(synth.normal(K, seed=87))
    s = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        o = torch.empty(M, device="cuda")
        with torch.cuda.stream(s):
            G.gemv_fused(Wd, synth.Q4_0, xd, M, K, ogemv.EPI_SIGMOID, None, o, stream=s)
        outs.append(o)
    s.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ----------------------------------------------------------------------------- full sizes

def test_full_f16_4096_add_view_in_place_and_sigmoid(G):
    """f16 4096x4096, W ~ N(0, 0.02), x ~ N(0,1); residual add through a [32,128] view
    into r in place; and the sigmoid tail.  Every row against the oracle."""
    M = K = 4096
    raw = synth.weights(synth.F16, M, K, seed=0)
    x = synth.normal(K, seed=1)
    r = synth.normal(M, seed=2)
    bound = gemv_bound(raw, synth.F16, x, M, K)
    got, path = run_gemv(G, raw, synth.F16, x, M, K, ogemv.EPI_ADD, r, view=(32, 128))
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, synth.F16, x, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, bound, "f16 add view")
    got, _ = run_gemv(G, raw, synth.F16, x, M, K, ogemv.EPI_SIGMOID, None)
    want = ogemv.gemv(raw, synth.F16, x, M, K, ogemv.EPI_SIGMOID)
    assert_within(got, want, bound, "f16 sigmoid")


def test_full_q8_0_swiglu_gate(G):
    """Q8_0 11008x4096, q ~ U{-127..127}, d ~ U(0.001, 0.01); silu(y) * m."""
    M, K = 11008, 4096
    raw = synth.weights(synth.Q8_0, M, K, seed=0)
    x = synth.normal(K, seed=1)
    m = synth.normal(M, seed=2)
    got, path = run_gemv(G, raw, synth.Q8_0, x, M, K, ogemv.EPI_SILU_MUL, m)
    assert path == G.PATH_STREAM
    want = ogemv.gemv(raw, synth.Q8_0, x, M, K, ogemv.EPI_SILU_MUL, m)
    assert_within(got, want, gemv_bound(raw, synth.Q8_0, x, M, K), "q8_0 gate")


@pytest.mark.parametrize("ncols", [1, 3, 8])
def test_full_fwht_f16_5120(G, ncols):
    """signed FWHT(1024) prologue + f16 5120x5120 + in-place residual, ncols columns."""
    M = K = 5120
    B = 1024
    raw = synth.weights(synth.F16, M, K, seed=0)
    X = synth.normal(ncols * K, seed=1).reshape(ncols, K)
    s = synth.rademacher(B, seed=2)
    r = synth.normal(ncols * M, seed=3).reshape(ncols, M)
    got, path = run_gemv(G, raw, synth.F16, X, M, K, ogemv.EPI_ADD, r, ncols=ncols, signs=s, block=B)
    assert path == G.PATH_STREAM
    Xp = np.stack([ofwht.fwht_signed(X[c], s, B) for c in range(ncols)])
    E = np.stack([fwht_err_bound(X[c], B) for c in range(ncols)])
    want = ogemv.gemv(raw, synth.F16, Xp, M, K, ogemv.EPI_ADD, r)
    assert_within(got, want, gemv_bound(raw, synth.F16, Xp, M, K, x_err=E), "fwht f16 ncols %d" % ncols)


_CHAIN_CACHE = {}


def _chain_weights():
    if not _CHAIN_CACHE:
        for i, name in enumerate(ochain.LAYER_ORDER):
            M, K = CHAIN_SHAPES[name]
            _CHAIN_CACHE[name] = (synth.weights(synth.Q4_0, M, K, seed=100 + i), synth.Q4_0, M, K)
    return _CHAIN_CACHE


CHAIN_SHAPES = {"q": (4096, 4096), "k": (4096, 4096), "v": (4096, 4096), "o": (4096, 4096),
                "up": (14336, 4096), "gate": (14336, 4096), "down": (4096, 14336), "beta": (32, 4096)}


def test_full_q4_0_decode_layer_four_launches(G):
    """The same layer as the bench step runs it: q, k, v and the sigmoid head sharing x in
    one gemv_multi, o + residual add, gate and up in one gemv_glu, down + residual add.
    Each launch's outputs, every row, against the oracle on the inputs it saw."""
    w = _chain_weights()
    dev = {name: dev_tensor(w[name][0]) for name in ochain.LAYER_ORDER}
    x = synth.normal(4096, seed=210)
    a = synth.normal(4096, seed=211)
    r = synth.normal(4096, seed=212)
    xd, ad, rd = dev_tensor(x), dev_tensor(a), dev_tensor(r)
    outs = {n: torch.full((CHAIN_SHAPES[n][0],), float("nan"), device="cuda") for n in ("q", "k", "v", "gate", "beta")}
    G.gemv_multi([(dev["q"], 4096, 0, None, outs["q"]), (dev["k"], 4096, 0, None, outs["k"]),
                  (dev["v"], 4096, 0, None, outs["v"]), (dev["beta"], 32, ogemv.EPI_SIGMOID, None, outs["beta"])],
                 synth.Q4_0, xd, 4096, pdl=True)
    G.gemv_fused_ex(dev["o"], synth.Q4_0, ad, 4096, 4096, ogemv.EPI_ADD, rd, rd, pdl=True)
    torch.cuda.synchronize()
    r1 = rd.cpu().numpy().astype(np.float64)
    G.gemv_glu(dev["gate"], dev["up"], synth.Q4_0, rd, 14336, 4096, outs["gate"], pdl=True)
    G.gemv_fused_ex(dev["down"], synth.Q4_0, outs["gate"], 4096, 14336, ogemv.EPI_ADD, rd, rd, pdl=True)
    torch.cuda.synchronize()
    h = {k: v.cpu().numpy().astype(np.float64) for k, v in outs.items()}
    r2 = rd.cpu().numpy().astype(np.float64)

    def check(name, vec_in, epi, aux, got):
        raw, wt, M, K = w[name]
        want = ogemv.gemv(raw, wt, vec_in, M, K, epi, aux)
        assert_within(got, want[0], gemv_bound(raw, wt, vec_in, M, K)[0], name)

    for n in ("q", "k", "v"):
        check(n, x, 0, None, h[n])
    check("beta", x, ogemv.EPI_SIGMOID, None, h["beta"])
    check("o", a, ogemv.EPI_ADD, r, r1)
    # silu(gate r1) * (up r1): the oracle's gated dual GEMV on the same rows
    rg, _, M, K = w["gate"]
    ru = w["up"][0]
    r1f = r1.astype(np.float32)
    want = ogemv.gemv_glu(rg, ru, synth.Q4_0, r1f, M, K)
    assert_within(h["gate"], want[0], glu_bound(rg, ru, synth.Q4_0, r1f, M, K)[0], "gate*up")
    check("down", h["gate"].astype(np.float32), ogemv.EPI_ADD, r1, r2)


@pytest.mark.parametrize("pdl", [False, True])
def test_full_q4_0_decode_layer_chain(G, pdl):
    """Q4_0 layer (d_model 4096, ffn 14336): 8 fused launches.  Each step is checked
    against the oracle on the GPU's own input for that step (every row), and the
    PDL-chained run must equal the serial one bit for bit."""
    w = _chain_weights()
    dev = {name: dev_tensor(w[name][0]) for name in ochain.LAYER_ORDER}
    x = synth.normal(4096, seed=200)
    a = synth.normal(4096, seed=201)
    r = synth.normal(4096, seed=202)
    xd, ad, rd = dev_tensor(x), dev_tensor(a), dev_tensor(r)
    outs = {n: torch.empty(CHAIN_SHAPES[n][0], device="cuda") for n in ("q", "k", "v", "up", "gate", "beta")}
    snap = {}

    def mv(name, vec, epi, aux, dst):
        M, K = CHAIN_SHAPES[name]
        G.gemv_fused_ex(dev[name], synth.Q4_0, vec, M, K, epi, aux, dst, pdl=pdl)

    mv("q", xd, 0, None, outs["q"])
    mv("k", xd, 0, None, outs["k"])
    mv("v", xd, 0, None, outs["v"])
    mv("o", ad, ogemv.EPI_ADD, rd, rd)
    snap["r1"] = rd.clone()
    mv("up", rd, 0, None, outs["up"])
    mv("gate", rd, ogemv.EPI_SILU_MUL, outs["up"], outs["gate"])
    mv("down", outs["gate"], ogemv.EPI_ADD, rd, rd)
    mv("beta", xd, ogemv.EPI_SIGMOID, None, outs["beta"])
    torch.cuda.synchronize()
    h = {k: v.cpu().numpy().astype(np.float64) for k, v in outs.items()}
    r1 = snap["r1"].cpu().numpy().astype(np.float64)
    r2 = rd.cpu().numpy().astype(np.float64)

    def check(name, vec_in, epi, aux, got):
        raw, wt, M, K = w[name]
        want = ogemv.gemv(raw, wt, vec_in, M, K, epi, aux)
        assert_within(got, want[0], gemv_bound(raw, wt, vec_in, M, K)[0], name)

    check("q", x, 0, None, h["q"])
    check("k", x, 0, None, h["k"])
    check("v", x, 0, None, h["v"])
    check("o", a, ogemv.EPI_ADD, r, r1)
    check("up", r1.astype(np.float32), 0, None, h["up"])
    check("gate", r1.astype(np.float32), ogemv.EPI_SILU_MUL, h["up"], h["gate"])
    check("down", h["gate"].astype(np.float32), ogemv.EPI_ADD, r1, r2)
    check("beta", x, ogemv.EPI_SIGMOID, None, h["beta"])
    if pdl:
        test_full_q4_0_decode_layer_chain.pdl_result = r2
    else:
        test_full_q4_0_decode_layer_chain.serial_result = r2
    both = [getattr(test_full_q4_0_decode_layer_chain, k, None) for k in ("serial_result", "pdl_result")]
    if all(b is not None for b in both):
        assert np.array_equal(both[0], both[1])
