"""Dynamic range of x for the single-column Q4_0, Q8_0 and Q4_K kernels.

Those kernels take integer dot products against x rounded to 24-bit integers that share
one exponent per 16-element unit, and hand a unit to fp32 products when that rounding
could be coarse next to its values (an outlier, a sparse unit) or when a value is NaN or
infinite.  Every case here is gated on the workload's literal bound
|gpu - oracle| <= 2e-5 * sum_k |W_ik x_k| + 1e-6 (for Q4_K the scale of each weight is
|d sc q| + |dmin m|), through gemv_fused, gemv_multi, gemv_glu, the split-K kernel and the
RMS prologue, at the decode layer's sizes.  Non-finite outputs must be NaN exactly where
the oracle's are NaN and the same infinity where the oracle's are infinite."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import TOL_ABS, TOL_REL, assert_within, dev_tensor, int_rounding_scale
from oracle import gemv as ogemv
from oracle import norm as onorm
from oracle import quant as oquant

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

NONE, SIG, SILU_MUL, ADD = ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD
FORMATS = {"q4_0": synth.Q4_0, "q8_0": synth.Q8_0, "q4_k": synth.Q4_K}


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


# ----------------------------------------------------------------------------- inputs

SPIKE_COLS = (5, 600, 601, 2060, 3900)  # 600 and 601 share a unit in every format


def zero_weight_columns(raw, wt, M, K, cols):
    """A copy of the packed weights whose elements in columns `cols` are exactly zero in
    every row: Q4_0 code 8, Q8_0 code 0, Q4_K code 0 with the sub-block's min zeroed (cols
    of Q4_K must lie in sub-blocks 0..3 of their super-block, whose mins sit in the low
    six bits of scale bytes 4..7)."""
    rb = oquant.row_bytes(wt, K)
    w = raw.copy().reshape(M, rb)
    for k in cols:
        if wt == synth.Q4_0:
            b, j = divmod(k, 32)
            byte = 18 * b + 2 + (j % 16)
            if j < 16:
                w[:, byte] = (w[:, byte] & 0xF0) | 8
            else:
                w[:, byte] = (w[:, byte] & 0x0F) | 0x80
        elif wt == synth.Q8_0:
            b, j = divmod(k, 32)
            w[:, 34 * b + 2 + j] = 0
        else:
            sb, e = divmod(k, 256)
            j, t = divmod(e, 32)
            assert j < 4, "Q4_K spike columns must sit in sub-blocks 0..3"
            base = 144 * sb
            w[:, base + 4 + 4 + j] &= 0xC0                  # m[j] = 0 (keep sc[j + 4]'s top bits)
            code = base + 16 + 32 * (j // 2) + t
            w[:, code] &= 0xF0 if j % 2 == 0 else 0x0F       # q = 0
    out = w.reshape(-1)
    deq = oquant.dequantize(out, wt, M, K)
    assert np.all(deq[:, list(cols)] == 0.0)
    return out


def x_case(name, K, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    base = g.standard_normal(K)
    if name == "zeros":
        x = np.zeros(K)
    elif name == "scale_3e4":
        x = 3e4 * base
    elif name == "scale_1e-20":
        x = 1e-20 * base
    elif name == "mixed_1e3_1e-3":  # every unit holds eight values near 1e3 and eight near 1e-3
        x = base * np.where(np.arange(K) % 2 == 0, 1e3, 1e-3)
    elif name.startswith("spike_"):  # N(0,1) with spikes on the columns whose weights are zero
        x = base.copy()
        x[list(SPIKE_COLS)] = float(name.split("_")[1]) * np.array([1.0, -1.0, 1.0, -1.0, 1.0])
    elif name == "heavy_tail":  # cubes of N(0,1): units often hold one value far above the rest
        x = base ** 3
    elif name == "sparse":  # one value in 64 non-zero, magnitudes over six decades
        x = np.where(g.random(K) < 1.0 / 64, base * 10.0 ** g.uniform(-3, 3, K), 0.0)
    else:
        raise ValueError(name)
    return x.astype(np.float32)


# spike_3e2 stays on the integer path (its spikes are below 1024 times the mean of their
# units' other values); the larger spikes send their units to the fp32 products
FINITE_CASES = ["zeros", "scale_3e4", "scale_1e-20", "mixed_1e3_1e-3", "spike_3e2", "spike_1e4", "spike_1e6",
                "heavy_tail", "sparse"]


# cases whose units the integer path must hand to the fp32 repair, and ones it must carry
REPAIRED = ("spike_1e4", "spike_1e6")
NOT_REPAIRED = ("zeros", "scale_3e4", "scale_1e-20", "mixed_1e3_1e-3", "spike_3e2", "heavy_tail")


def case_weights(wt, M, K, seed):
    raw = synth.weights(wt, M, K, seed=seed)
    return zero_weight_columns(raw, wt, M, K, SPIKE_COLS)


def literal_bound(raw, wt, x, M, K, rows=None):
    """The literal bound 2e-5 * sum_k |W_ik x_k| + 1e-6."""
    return TOL_REL * ogemv.abs_dot(raw, wt, x, M, K, rows) + TOL_ABS


def scaled_bound(raw, wt, x, M, K, want):
    """A stricter companion for inputs far below 1, where the literal bound's 1e-6 alone
    would pass anything: its absolute term scaled by max |x|, plus the rounding of the
    stored fp32 output itself (2^-24 of it: with a residual add the output is about r)."""
    xmax = float(np.max(np.abs(x))) if np.size(x) else 0.0
    return (TOL_REL * ogemv.abs_dot(raw, wt, x, M, K)[0] + TOL_ABS * min(1.0, xmax)
            + 2.0 ** -24 * np.abs(want))


def report_ratio(got, want, raw, wt, x, M, K):
    """Max error over the scale a shared-exponent rounding of every unit would have (2^-23
    of max|x| per block times sum |w| per block): printed, never gated."""
    scale = 2.0 ** -23 * int_rounding_scale(raw, wt, x, M, K)
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(scale > 0, err / scale, 0.0)
    print("max err / (2^-23 * block-max scale) = %.3g" % float(np.max(r)))


def assert_classes(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "%s: NaN pattern differs" % what
    inf = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf), "%s: Inf pattern differs" % what
    assert np.array_equal(got[inf], want[inf]), "%s: sign of an infinity differs" % what
    fin = np.isfinite(want)
    return fin


# ----------------------------------------------------------------------------- gemv_fused

@pytest.mark.parametrize("fmt,M,K", [("q4_0", 4096, 4096), ("q8_0", 11008, 4096), ("q4_k", 4096, 4096)])
@pytest.mark.parametrize("case", FINITE_CASES)
def test_gemv_fused_dynamic_range(G, fmt, M, K, case):
    wt = FORMATS[fmt]
    raw = case_weights(wt, M, K, seed=500 + wt)
    x = x_case(case, K, seed=510)
    r = synth.normal(M, seed=511)
    Wd, xd = dev_tensor(raw), dev_tensor(x)
    for epi in (NONE, ADD):
        dst = dev_tensor(r) if epi == ADD else torch.full((M,), float("nan"), device="cuda")
        G.repair_count(reset=True)
        G.gemv_fused(Wd, wt, xd, M, K, epi, dst if epi == ADD else None, dst)
        torch.cuda.synchronize()
        repairs = G.repair_count()
        if case in REPAIRED:
            assert repairs > 0, "%s %s: the fp32 repair should have run" % (fmt, case)
        elif case in NOT_REPAIRED:
            assert repairs == 0, "%s %s: %d row chunks repaired" % (fmt, case, repairs)
        got = dst.cpu().numpy().astype(np.float64)
        want = ogemv.gemv(raw, wt, x, M, K, epi, r)[0]
        assert_within(got, want, literal_bound(raw, wt, x, M, K)[0], "%s %s epi %d" % (fmt, case, epi))
        if case != "zeros":
            assert_within(got, want, scaled_bound(raw, wt, x, M, K, want), "%s %s epi %d (scaled)" % (fmt, case, epi))
        if epi == NONE:
            report_ratio(got, want, raw, wt, x, M, K)


@pytest.mark.parametrize("fmt,M,K", [("q4_0", 4096, 4096), ("q8_0", 4096, 4096), ("q4_k", 4096, 4096)])
@pytest.mark.parametrize("bad", ["nan", "inf", "-inf", "inf_and_-inf"])
def test_gemv_fused_non_finite_x(G, fmt, M, K, bad):
    wt = FORMATS[fmt]
    raw = case_weights(wt, M, K, seed=520 + wt)
    x = x_case("heavy_tail", K, seed=521)
    if bad == "nan":
        x[1234] = np.nan
    elif bad == "inf":
        x[1234] = np.inf
    elif bad == "-inf":
        x[3000] = -np.inf
    else:
        x[1234], x[3000] = np.inf, -np.inf
    Wd, xd = dev_tensor(raw), dev_tensor(x)
    for epi in (NONE, SIG):
        dst = torch.zeros(M, device="cuda")
        G.repair_count(reset=True)
        G.gemv_fused(Wd, wt, xd, M, K, epi, None, dst)
        torch.cuda.synchronize()
        assert G.repair_count() > 0, "a non-finite x must go to the fp32 repair"
        got = dst.cpu().numpy().astype(np.float64)
        with np.errstate(invalid="ignore", over="ignore"):
            want = ogemv.gemv(raw, wt, x, M, K, epi)[0]
        fin = assert_classes(got, want, "%s %s epi %d" % (fmt, bad, epi))
        if np.any(fin):  # sigmoid of +-inf is finite: those must still be within the bound
            b = TOL_REL * 1.0 + TOL_ABS
            assert np.all(np.abs(got[fin] - want[fin]) <= b)


# ----------------------------------------------------------------------------- gemv_multi, gemv_glu

@pytest.mark.parametrize("case", ["spike_1e6", "mixed_1e3_1e-3", "heavy_tail", "nan", "inf"])
def test_gemv_multi_dynamic_range(G, case):
    """q, k, v and the sigmoid head sharing x, as the decode layer runs them."""
    K = 4096
    shapes = [(4096, NONE), (4096, NONE), (4096, NONE), (32, SIG)]
    raws = [case_weights(synth.Q4_0, M, K, seed=530 + i) for i, (M, _) in enumerate(shapes)]
    if case in ("nan", "inf"):
        x = x_case("heavy_tail", K, seed=535)
        x[2222] = np.nan if case == "nan" else np.inf
    else:
        x = x_case(case, K, seed=535)
    xd = dev_tensor(x)
    outs = [torch.full((M,), 7.0, device="cuda") for (M, _) in shapes]
    G.gemv_multi([(dev_tensor(raws[i]), M, e, None, outs[i]) for i, (M, e) in enumerate(shapes)], synth.Q4_0, xd, K)
    torch.cuda.synchronize()
    for i, (M, e) in enumerate(shapes):
        got = outs[i].cpu().numpy().astype(np.float64)
        with np.errstate(invalid="ignore", over="ignore"):
            want = ogemv.gemv(raws[i], synth.Q4_0, x, M, K, e)[0]
        if case in ("nan", "inf"):
            assert_classes(got, want, "multi %d %s" % (i, case))
        else:
            assert_within(got, want, literal_bound(raws[i], synth.Q4_0, x, M, K)[0], "multi %d %s" % (i, case))


@pytest.mark.parametrize("fmt", ["q4_0", "q4_k"])
@pytest.mark.parametrize("case", ["spike_1e6", "heavy_tail", "sparse", "inf"])
def test_gemv_glu_dynamic_range(G, fmt, case):
    """silu(W_gate x) * (W_up x), 14336 x 4096: each product against the oracle's."""
    wt = FORMATS[fmt]
    M, K = 14336, 4096
    rg = case_weights(wt, M, K, seed=540 + wt)
    ru = case_weights(wt, M, K, seed=541 + wt)
    if case == "inf":
        x = x_case("heavy_tail", K, seed=545)
        x[1111] = np.inf
    else:
        x = x_case(case, K, seed=545)
    dst = torch.full((M,), 7.0, device="cuda")
    G.gemv_glu(dev_tensor(rg), dev_tensor(ru), wt, dev_tensor(x), M, K, dst)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        want = ogemv.gemv_glu(rg, ru, wt, x, M, K)[0]
    if case == "inf":
        assert_classes(got, want, "glu %s inf" % fmt)
        return
    gv = ogemv.gemv(rg, wt, x, M, K)[0]
    uv = ogemv.gemv(ru, wt, x, M, K)[0]
    bg = literal_bound(rg, wt, x, M, K)[0]
    bu = literal_bound(ru, wt, x, M, K)[0]
    sg = ogemv.silu(gv)
    bound = 1.1 * bg * (np.abs(uv) + bu) + np.abs(sg) * bu + 1e-6 * np.abs(sg * uv)
    assert_within(got, want, bound, "glu %s %s" % (fmt, case))


# ----------------------------------------------------------------------------- split K, RMS prologue

@pytest.mark.parametrize("case", ["spike_1e6", "heavy_tail", "nan"])
def test_split_k_dynamic_range(G, case):
    """Few rows, long K: a cluster of CTAs splits K (the integer path in every rank)."""
    M, K = 8, 65536
    wt = synth.Q4_0
    raw = case_weights(wt, M, K, seed=550)
    if case == "nan":
        x = x_case("heavy_tail", K, seed=551)
        x[40000] = np.nan
    else:
        x = x_case(case, K, seed=551)
    xd = dev_tensor(x)
    _, info = G.plan(dev_tensor(raw), wt, xd, M, K, NONE, None, torch.empty(M, device="cuda"))
    assert info["split"] > 1, "expected a split-K plan"
    dst = torch.full((M,), 7.0, device="cuda")
    G.gemv_fused(dev_tensor(raw), wt, xd, M, K, NONE, None, dst)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    with np.errstate(invalid="ignore"):
        want = ogemv.gemv(raw, wt, x, M, K)[0]
    if case == "nan":
        assert np.all(np.isnan(got)) and np.all(np.isnan(want))
    else:
        assert_within(got, want, literal_bound(raw, wt, x, M, K)[0], "split %s" % case)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_rms_prologue_with_spike(G, fmt):
    """RMS normalisation ahead of the GEMV, x with spikes on zero-weight columns: the
    kernel's x' = x * gamma carries the spikes into the integer conversion."""
    wt = FORMATS[fmt]
    M, K = 4096, 4096
    raw = case_weights(wt, M, K, seed=560 + wt)
    x = x_case("spike_1e4", K, seed=561)
    gamma = (1.0 + 0.1 * synth.normal(K, seed=562)).astype(np.float32)
    eps = 1e-6
    dst = torch.full((M,), 7.0, device="cuda")
    G.gemv_fused_ex(dev_tensor(raw), wt, dev_tensor(x), M, K, NONE, None, dst, rms_norm_weight=dev_tensor(gamma),
                    rms_norm_eps=eps)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    xn = onorm.rms_norm(x, gamma, eps, K)[0]
    want = ogemv.gemv(raw, wt, xn, M, K)[0]
    # the literal bound on x', plus the kernel's own 1/rms (under 2e-6 relative)
    bound = literal_bound(raw, wt, xn, M, K)[0] + 2e-6 * ogemv.abs_dot(raw, wt, xn, M, K)[0]
    assert_within(got, want, bound, "rms %s spike" % fmt)


# ----------------------------------------------------------------------------- on-chip FWHT prologue

@pytest.mark.parametrize("M,K", [(512, 5120), (300, 32768), (8, 32768)])
@pytest.mark.parametrize("bad", ["nan", "inf"])
def test_fwht_prologue_non_finite(G, M, K, bad):
    """Signed FWHT(1024) on chip ahead of a Q4_0 GEMV: one K chunk, several chunks, and
    split K (8 rows).  A non-finite x spreads over its whole transform block, so the rows
    are recomputed with x' rebuilt chunk by chunk; the non-finite pattern must match."""
    B = 1024
    wt = synth.Q4_0
    raw = synth.weights(wt, M, K, seed=570)
    x = x_case("heavy_tail", K, seed=571)
    x[K - 700] = np.nan if bad == "nan" else np.inf
    s = synth.rademacher(B, seed=572)
    xd, sd = dev_tensor(x), dev_tensor(s)
    dst = torch.full((M,), 7.0, device="cuda")
    G.gemv_fused_ex(dev_tensor(raw), wt, xd, M, K, NONE, None, dst, fwht_signs=sd, fwht_block=B)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    from oracle import fwht as ofwht
    with np.errstate(invalid="ignore", over="ignore"):
        xp = ofwht.fwht_signed(x, s, B)
        want = ogemv.gemv(raw, wt, xp, M, K)[0]
    assert_classes(got, want, "fwht %s %dx%d" % (bad, M, K))


@pytest.mark.parametrize("M,K", [(512, 5120), (300, 32768), (8, 32768)])
def test_fwht_prologue_after_repair_matches_oracle(G, M, K):
    """Finite x whose transform holds an outlier unit: x is chosen so that one 1024-block
    of x' = H (s x) / 32 is a single spike (x = the block's inverse transform of a
    one-hot, times 1e6) on top of N(0,1) elsewhere; the spike's column has zero weights.
    Its unit is repaired in fp32; every row within the literal bound on x'."""
    B = 1024
    wt = synth.Q4_0
    col = 1024 + 37
    raw = zero_weight_columns(synth.weights(wt, M, K, seed=580), wt, M, K, (col,))
    s = synth.rademacher(B, seed=581)
    from oracle import fwht as ofwht
    target = x_case("heavy_tail", K, seed=582).astype(np.float64)
    target[col] = 1e6
    # x with fwht_signed(x) == target: the normalised transform is its own inverse, then undo the signs
    blocks = target.reshape(-1, B)
    x = np.concatenate([ofwht.fwht_signed(b, np.ones(B), B) * s for b in blocks]).astype(np.float32)
    xp = ofwht.fwht_signed(x, s, B)
    dst = torch.full((M,), 7.0, device="cuda")
    G.gemv_fused_ex(dev_tensor(raw), wt, dev_tensor(x), M, K, NONE, None, dst, fwht_signs=dev_tensor(s),
                    fwht_block=B)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    want = ogemv.gemv(raw, wt, xp, M, K)[0]
    from gpu_util import fwht_err_bound
    E = fwht_err_bound(x, B).reshape(1, K)
    bound = literal_bound(raw, wt, xp, M, K)[0] + ogemv.abs_w_dot(raw, wt, E, M, K)[0]
    assert_within(got, want, bound, "fwht repaired %dx%d" % (M, K))
