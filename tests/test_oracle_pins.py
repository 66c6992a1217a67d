"""Pins for the fp64 oracle: closed forms, hand-worked fixtures, library special cases
and brute force.  None of these compares the oracle with itself.  The mutation tests at
the end plant plausible mistakes in copies of oracle functions and check that a pin
fails for each."""

import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
from oracle import chain, fwht, gemv, quant

F32, F16, Q8_0, Q4_0 = quant.WTYPE_F32, quant.WTYPE_F16, quant.WTYPE_Q8_0, quant.WTYPE_Q4_0


def _hexbytes(tokens):
    return np.array([int(t, 16) for t in tokens], dtype=np.uint8)


# ----------------------------------------------------------------------------- decoders

def check_f16_fixture(dequant_f16):
    g = read_golden("f16_values.txt")["rows"]
    raw = np.concatenate([np.array([int(h, 16) & 0xFF, int(h, 16) >> 8], dtype=np.uint8)
                          for h, _ in g])
    got = dequant_f16(raw, 1, len(g))[0]
    want = np.array([float(v) for _, v in g])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_f16_fixture():
    check_f16_fixture(quant.dequantize_f16)


def test_f16_all_patterns_match_numpy_float16():
    # library special case: numpy's binary16 conversion, every non-NaN pattern
    pats = np.arange(65536, dtype=np.uint32).astype("<u2")
    got = quant.dequantize_f16(pats.view(np.uint8), 1, 65536)[0]
    want = pats.view(np.float16).astype(np.float64)
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.all(np.isnan(got[~ok]))


def test_f32_bytes_roundtrip():
    v = np.array([1.5, -0.0, 3.4028234663852886e38, 1e-45, -7.25], dtype="<f4")
    got = quant.dequantize_f32(v.view(np.uint8), 1, v.size)[0]
    assert np.array_equal(got, v.astype(np.float64))


def check_q8_0_fixture(dequant):
    g = read_golden("q8_0_block.txt")
    raw = _hexbytes(g["bytes"][0])
    got = dequant(raw, 1, 32)[0]
    assert np.array_equal(got, np.array([float(v) for v in g["values"][0]]))


def test_q8_0_fixture():
    check_q8_0_fixture(quant.dequantize_q8_0)


def check_q4_0_fixture(dequant):
    g = read_golden("q4_0_block.txt")
    for b, v in zip(g["bytes"], g["values"]):
        got = dequant(_hexbytes(b), 1, 32)[0]
        assert np.array_equal(got, np.array([float(t) for t in v])), (b, got)
    # the three blocks as one row of K = 96 (block order along the row)
    raw = np.concatenate([_hexbytes(b) for b in g["bytes"]])
    got = dequant(raw, 1, 96)[0]
    want = np.concatenate([[float(t) for t in v] for v in g["values"]])
    assert np.array_equal(got, want)


def test_q4_0_fixture():
    check_q4_0_fixture(quant.dequantize_q4_0)


def test_row_bytes():
    assert quant.row_bytes(Q4_0, 4096) == 2304
    assert quant.row_bytes(Q8_0, 4096) == 4352
    assert quant.row_bytes(Q4_0, 14336) == 8064
    assert quant.row_bytes(F16, 5120) == 10240
    with pytest.raises(ValueError):
        quant.row_bytes(Q4_0, 33)


# ----------------------------------------------------------------------------- GEMV

def check_worked_example(gemv_fn):
    g = read_golden("gemv_worked.txt")
    W = np.array([float(t) for t in g["W"][0]], dtype="<f4")
    x = np.array([float(t) for t in g["x"][0]])
    y = gemv_fn(W.view(np.uint8), F32, x, 2, 3, gemv.EPI_NONE)[0]
    assert np.array_equal(y, np.array([float(t) for t in g["y"][0]]))
    r = np.array([float(t) for t in g["r"][0]])
    a = gemv_fn(W.view(np.uint8), F32, x, 2, 3, gemv.EPI_ADD, r)[0]
    assert np.array_equal(a, np.array([float(t) for t in g["add"][0]]))


def test_gemv_worked_example():
    check_worked_example(gemv.gemv)


def test_gemv_identity_f32():
    K = 8
    W = np.eye(K, dtype="<f4")
    x = np.arange(1, K + 1, dtype=np.float64) * 0.25
    assert np.array_equal(gemv.gemv(W.view(np.uint8), F32, x, K, K)[0], x)


def check_onehot_selects_column(gemv_fn):
    """x = e_j gives column j of W.  The rows of W are the hand-decoded Q4_0 blocks, so
    a transposed operand or a wrong element order fails."""
    g = read_golden("q4_0_block.txt")
    raw = np.concatenate([_hexbytes(b) for b in g["bytes"]])      # 3 rows of K = 32
    vals = np.array([[float(t) for t in v] for v in g["values"]])  # [3, 32]
    for j in (0, 5, 16, 31):
        x = np.zeros(32)
        x[j] = 1.0
        y = gemv_fn(raw, Q4_0, x, 3, 32, gemv.EPI_NONE)[0]
        assert np.array_equal(y, vals[:, j]), j


def test_gemv_onehot_selects_column():
    check_onehot_selects_column(gemv.gemv)


def test_gemv_onehot_q8_0():
    g = read_golden("q8_0_block.txt")
    raw = _hexbytes(g["bytes"][0])
    vals = [float(t) for t in g["values"][0]]
    for j in range(32):
        x = np.zeros(32)
        x[j] = 1.0
        assert gemv.gemv(raw, Q8_0, x, 1, 32)[0][0] == vals[j]


@pytest.mark.parametrize("M,K", [(1, 1), (2, 3), (3, 5), (8, 8), (5, 7)])
def test_gemv_brute_force_exact(M, K):
    # integer-valued f32 weights and inputs: exact in fp64; brute force with Fractions
    g = np.random.Generator(np.random.PCG64(100 + M * 10 + K))
    W = g.integers(-9, 10, size=(M, K)).astype("<f4")
    X = g.integers(-9, 10, size=(2, K)).astype(np.float64)
    got = gemv.gemv(W.view(np.uint8), F32, X, M, K)
    for c in range(2):
        for i in range(M):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(int(W[i, k])) * Fraction(int(X[c, k]))
            assert got[c, i] == float(acc)


def test_gemv_rows_subset_and_batch_layout():
    # x is [ncols][K]; aux/out are [ncols][M]; a row subset keeps row identity
    W = np.array([[1, 0], [0, 1], [2, 3]], dtype="<f4")
    X = np.array([[1.0, 10.0], [100.0, 1000.0]])
    full = gemv.gemv(W.view(np.uint8), F32, X, 3, 2)
    assert np.array_equal(full, np.array([[1, 10, 32], [100, 1000, 3200]], dtype=np.float64))
    sub = gemv.gemv(W.view(np.uint8), F32, X, 3, 2, rows=[2, 0])
    assert np.array_equal(sub, full[:, [2, 0]])


# ----------------------------------------------------------------------------- tails

def check_epilogue_closed_forms(apply):
    assert apply(np.array([0.0]), gemv.EPI_SIGMOID)[0] == 0.5
    assert apply(np.array([0.0]), gemv.EPI_SILU)[0] == 0.0
    # sigmoid(ln 3) = 3/4 and silu(ln 3) = 3/4 ln 3
    l3 = math.log(3.0)
    assert abs(apply(np.array([l3]), gemv.EPI_SIGMOID)[0] - 0.75) < 1e-15
    assert abs(apply(np.array([l3]), gemv.EPI_SILU)[0] - 0.75 * l3) < 1e-15
    assert abs(apply(np.array([-l3]), gemv.EPI_SIGMOID)[0] - 0.25) < 1e-15
    y = np.linspace(-30, 30, 121)
    s = apply(y, gemv.EPI_SIGMOID)
    assert np.allclose(s + apply(-y, gemv.EPI_SIGMOID), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(s) > 0)
    assert apply(np.array([800.0]), gemv.EPI_SIGMOID)[0] == 1.0
    assert apply(np.array([-800.0]), gemv.EPI_SIGMOID)[0] == 0.0
    assert apply(np.array([-800.0]), gemv.EPI_SILU)[0] == 0.0
    assert apply(np.array([60.0]), gemv.EPI_SILU)[0] == pytest.approx(60.0, rel=1e-20, abs=1e-12)
    m = np.array([2.0, -3.0, 0.5])
    y3 = np.array([l3, 0.0, -l3])
    assert np.allclose(apply(y3, gemv.EPI_SILU_MUL, m),
                       np.array([0.75 * l3 * 2.0, 0.0, -0.25 * l3 * 0.5]), rtol=0, atol=1e-15)
    r = np.array([1.0, -2.0, 0.25])
    assert np.array_equal(apply(np.array([1.0, 2.0, 3.0]), gemv.EPI_ADD, r),
                          np.array([2.0, 0.0, 3.25]))
    assert np.array_equal(apply(np.array([1.0, -2.0]), gemv.EPI_NONE), np.array([1.0, -2.0]))


def test_epilogue_closed_forms():
    check_epilogue_closed_forms(gemv.apply_epilogue)


def test_epilogue_special_cases_through_gemv():
    K, M = 64, 16
    g = np.random.Generator(np.random.PCG64(7))
    x = g.standard_normal(K)
    r = g.standard_normal(M)
    m = g.standard_normal(M)
    zero = np.zeros((M, K), dtype="<f4").view(np.uint8)
    # W = 0: ADD returns r exactly, SILU_MUL returns 0, SIGMOID returns 1/2
    assert np.array_equal(gemv.gemv(zero, F32, x, M, K, gemv.EPI_ADD, r)[0], r)
    assert np.array_equal(gemv.gemv(zero, F32, x, M, K, gemv.EPI_SILU_MUL, m)[0], np.zeros(M))
    assert np.array_equal(gemv.gemv(zero, F32, x, M, K, gemv.EPI_SIGMOID)[0], np.full(M, 0.5))
    # m = 1: SILU_MUL equals SILU
    W = g.standard_normal((M, K)).astype("<f4").view(np.uint8)
    a = gemv.gemv(W, F32, x, M, K, gemv.EPI_SILU_MUL, np.ones(M))
    b = gemv.gemv(W, F32, x, M, K, gemv.EPI_SILU)
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        gemv.apply_epilogue(np.zeros(3), gemv.EPI_ADD, np.zeros(4))


# ----------------------------------------------------------------------------- Hadamard

def check_hadamard(hfn):
    assert np.array_equal(hfn(1), np.array([[1.0]]))
    assert np.array_equal(hfn(2), np.array([[1.0, 1.0], [1.0, -1.0]]))
    rows = read_golden("hadamard4.txt")["rows"]
    assert np.array_equal(hfn(4), np.array([[float(t) for t in r] for r in rows]))
    H2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    n = 2
    while n <= 256:
        assert np.array_equal(hfn(2 * n), np.kron(H2, hfn(n)))
        n *= 2
    for n in (8, 64, 1024):
        H = hfn(n)
        assert np.array_equal(H @ H.T, n * np.eye(n))


def test_hadamard_sylvester():
    check_hadamard(fwht.hadamard)


def test_hadamard_matches_scipy():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    for n in (1, 2, 16, 128, 1024):
        assert np.array_equal(fwht.hadamard(n), scipy_linalg.hadamard(n).astype(np.float64))


def check_fwht_fixture(fn):
    g = read_golden("fwht_signed_b4.txt")
    f = lambda k: np.array([float(t) for t in g[k][0]])
    assert np.allclose(fn(f("x"), f("signs"), 4), f("out"), rtol=0, atol=1e-15)
    assert np.allclose(fn(f("x2"), f("signs"), 4), f("out2"), rtol=0, atol=1e-15)


def test_fwht_worked_example():
    check_fwht_fixture(fwht.fwht_signed)
    check_fwht_fixture(fwht.fwht_butterfly)


def check_fwht_closed_forms(fn):
    B = 1024
    e0 = np.zeros(B)
    e0[0] = 1.0
    ones = np.ones(B)
    assert np.allclose(fn(e0, None, B), np.full(B, 1.0 / 32.0), rtol=0, atol=1e-15)
    assert np.allclose(fn(ones, None, B), 32.0 * e0, rtol=0, atol=1e-12)
    g = np.random.Generator(np.random.PCG64(3))
    x = g.standard_normal(5 * B)
    s = np.where(g.integers(0, 2, B) == 0, -1.0, 1.0)
    y = fn(x, s, B)
    # Parseval per block (orthonormal transform; |s| = 1)
    assert np.allclose((y.reshape(5, B) ** 2).sum(1), (x.reshape(5, B) ** 2).sum(1), rtol=1e-12)
    # the normalised plain transform is an involution
    assert np.allclose(fn(fn(x, None, B), None, B), x, rtol=0, atol=1e-12)
    # signs are applied before the transform: undo with the plain transform then s
    assert np.allclose(fn(y, None, B) * np.tile(s, 5), x, rtol=0, atol=1e-12)
    # all +1 signs reduce to the plain transform; all -1 negate it
    assert np.array_equal(fn(x, np.ones(B), B), fn(x, None, B))
    assert np.allclose(fn(x, -np.ones(B), B), -fn(x, None, B), rtol=0, atol=0)
    # e_j with s_j = -1 gives -(1/sqrt(B)) H[:, j]
    j = 77
    ej = np.zeros(B)
    ej[j] = 1.0
    sj = np.ones(B)
    sj[j] = -1.0
    assert np.allclose(fn(ej, sj, B), -fwht.hadamard(B)[:, j] / 32.0, rtol=0, atol=1e-15)


def test_fwht_closed_forms_dense():
    check_fwht_closed_forms(fwht.fwht_signed)


def test_fwht_closed_forms_butterfly():
    check_fwht_closed_forms(fwht.fwht_butterfly)


@pytest.mark.parametrize("B", [1, 2, 4, 32, 256, 1024])
def test_fwht_butterfly_equals_dense(B):
    g = np.random.Generator(np.random.PCG64(B))
    x = g.standard_normal(3 * B)
    s = np.where(g.integers(0, 2, B) == 0, -1.0, 1.0)
    assert np.allclose(fwht.fwht_butterfly(x, s, B), fwht.fwht_signed(x, s, B), rtol=0, atol=1e-12)


def test_fwht_sign_broadcast_shorter_than_block():
    # signs of length 2 broadcast over a block of 4: element k uses s[k mod 2]
    x = np.array([1.0, 2.0, 3.0, 4.0])
    got = fwht.fwht_signed(x, np.array([1.0, -1.0]), 4)
    want = fwht.hadamard(4) @ np.array([1.0, -2.0, 3.0, -4.0]) / 2.0
    assert np.allclose(got, want, rtol=0, atol=0)


# ----------------------------------------------------------------------------- chain

def test_decode_layer_identity_weights():
    """With every weight the identity (f32, n x n) the chain reduces to element-wise
    closed forms: r1 = r + a, u = r1, g = silu(r1) * r1, r2 = r1 + g, beta = sigmoid(x)."""
    n = 16
    I = np.eye(n, dtype="<f4").view(np.uint8)
    w = {k: (I, F32, n, n) for k in chain.LAYER_ORDER}
    g = np.random.Generator(np.random.PCG64(11))
    x, a, r = g.standard_normal(n), g.standard_normal(n), g.standard_normal(n)
    out = chain.decode_layer(w, x, a, r)
    assert np.array_equal(out["q"], x) and np.array_equal(out["v"], x)
    assert np.array_equal(out["r1"], r + a)
    assert np.array_equal(out["u"], r + a)
    r1 = r + a
    silu_r1 = r1 / (1.0 + np.exp(-r1))
    assert np.allclose(out["g"], silu_r1 * r1, rtol=1e-15, atol=0)
    assert np.allclose(out["r2"], r1 + silu_r1 * r1, rtol=1e-15, atol=0)
    assert np.allclose(out["beta"], 1.0 / (1.0 + np.exp(-x)), rtol=1e-15, atol=0)


def test_decode_layer_order_gate_uses_up_output():
    # gate's multiplicand is up's output: scaling W_up by 2 doubles g (silu part fixed)
    n = 8
    I = np.eye(n, dtype="<f4")
    w = {k: (I.view(np.uint8), F32, n, n) for k in chain.LAYER_ORDER}
    w2 = dict(w)
    w2["up"] = ((2 * I).astype("<f4").view(np.uint8), F32, n, n)
    g = np.random.Generator(np.random.PCG64(12))
    x, a, r = g.standard_normal(n), g.standard_normal(n), g.standard_normal(n)
    o1 = chain.decode_layer(w, x, a, r)
    o2 = chain.decode_layer(w2, x, a, r)
    assert np.allclose(o2["g"], 2 * o1["g"], rtol=1e-15, atol=0)


# ----------------------------------------------------------------------------- mutations

def _expect_fail(check, fn):
    with pytest.raises(AssertionError):
        check(fn)


def test_mutation_swapped_nibbles_fails_pin():
    def bad(raw, M, K, rows=None):
        v = quant.dequantize_q4_0(raw, M, K, rows).reshape(M, K // 32, 32)
        return np.concatenate([v[:, :, 16:], v[:, :, :16]], axis=2).reshape(M, K)
    _expect_fail(check_q4_0_fixture, bad)


def test_mutation_interleaved_nibbles_fails_pin():
    # a plausible alternative layout: element 2j low nibble, element 2j+1 high nibble
    def bad(raw, M, K, rows=None):
        mat = np.asarray(raw).reshape(M, -1).reshape(M, K // 32, 18)
        d = quant._binary16_to_f64(mat[:, :, 0], mat[:, :, 1])
        qs = mat[:, :, 2:].astype(np.int64)
        codes = np.stack([qs & 15, qs >> 4], axis=-1).reshape(M, K // 32, 32)
        return (d[:, :, None] * (codes - 8)).reshape(M, K)
    _expect_fail(check_q4_0_fixture, bad)


def test_mutation_q8_unsigned_codes_fails_pin():
    def bad(raw, M, K, rows=None):
        mat = np.asarray(raw).reshape(M, K // 32, 34)
        d = quant._binary16_to_f64(mat[:, :, 0], mat[:, :, 1])
        return (d[:, :, None] * mat[:, :, 2:].astype(np.float64)).reshape(M, K)
    _expect_fail(check_q8_0_fixture, bad)


def test_mutation_transposed_weight_fails_pin():
    def bad(raw, wtype, x, M, K, epilogue=0, aux=None, rows=None):
        W = quant.dequantize(raw, wtype, M, K)
        y = np.asarray(x, dtype=np.float64).reshape(1, -1)[:, :M] @ W[:, :M]
        return gemv.apply_epilogue(y, epilogue, None if aux is None else np.asarray(aux).reshape(1, -1))
    _expect_fail(check_onehot_selects_column, bad)


def test_mutation_epilogue_sign_error_fails_pin():
    def bad(y, epilogue, aux=None):
        if epilogue == gemv.EPI_SIGMOID:
            return 1.0 / (1.0 + np.exp(np.asarray(y, dtype=np.float64)))
        return gemv.apply_epilogue(y, epilogue, aux)
    _expect_fail(check_epilogue_closed_forms, bad)


def test_mutation_silu_mul_order_fails_pin():
    def bad(y, epilogue, aux=None):
        if epilogue == gemv.EPI_SILU_MUL:
            return gemv.silu(np.asarray(y) * np.asarray(aux))
        return gemv.apply_epilogue(y, epilogue, aux)
    _expect_fail(check_epilogue_closed_forms, bad)


def test_mutation_sign_after_transform_fails_pin():
    def bad(x, signs, block):
        y = fwht.fwht_signed(x, None, block)
        return y if signs is None else y * np.tile(np.asarray(signs, float), y.size // len(signs))
    _expect_fail(check_fwht_fixture, bad)


def test_mutation_missing_normalisation_fails_pin():
    def bad(x, signs, block):
        return fwht.fwht_signed(x, signs, block) * np.sqrt(block)
    _expect_fail(check_fwht_fixture, bad)


def test_mutation_natural_order_hadamard_fails_pin():
    # a wrong matrix order (rows sorted by sequency instead of Sylvester's) must fail
    def bad(n):
        H = fwht.hadamard(n)
        if n < 4:
            return H
        seq = (np.diff(H, axis=1) != 0).sum(axis=1)
        return H[np.argsort(seq, kind="stable")]
    _expect_fail(check_hadamard, bad)
