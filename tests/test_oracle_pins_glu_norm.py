"""Pins for the oracle's gated dual GEMV and RMS normalisation prologue: hand-worked
fixtures, closed forms and limits; then mutation tests that plant plausible mistakes
in copies of the functions and check that a pin fails for each."""

import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import gemv, norm, quant

F32 = quant.WTYPE_F32


def _f32_raw(rows):
    return np.asarray(rows, dtype="<f4").reshape(-1).view(np.uint8)


def _floats(tokens):
    return np.array([float(t) for t in tokens])


# ----------------------------------------------------------------------------- gated dual GEMV

def check_glu_worked(glu):
    g = read_golden("glu_worked.txt")
    Wg, Wu, x = _floats(g["Wg"][0]), _floats(g["Wu"][0]), _floats(g["x"][0])
    got = glu(_f32_raw(Wg), _f32_raw(Wu), F32, x, 3, 2)[0]
    want = _floats(g["out"][0])
    assert np.allclose(got, want, rtol=1e-15, atol=0.0), got


def test_glu_worked_example():
    check_glu_worked(gemv.gemv_glu)


def check_glu_zero_and_onehot(glu):
    rng = np.random.default_rng(7)
    M, K = 5, 6
    Wg = rng.standard_normal((M, K))
    Wu = rng.standard_normal((M, K))
    x = rng.standard_normal(K)
    z = np.zeros((M, K))
    # silu(0) = 0: a zero gate zeroes the output; a zero up projection too
    assert np.all(glu(_f32_raw(z), _f32_raw(Wu), F32, x, M, K) == 0.0)
    assert np.all(glu(_f32_raw(Wg), _f32_raw(z), F32, x, M, K) == 0.0)
    # one-hot x = e_j picks column j of each weight: silu(Wg[:, j]) * Wu[:, j]
    Wg32, Wu32 = Wg.astype(np.float32).astype(np.float64), Wu.astype(np.float32).astype(np.float64)
    for j in range(K):
        e = np.zeros(K)
        e[j] = 1.0
        got = glu(_f32_raw(Wg), _f32_raw(Wu), F32, e, M, K)[0]
        gj = Wg32[:, j]
        want = gj / (1.0 + np.exp(-gj)) * Wu32[:, j]
        assert np.allclose(got, want, rtol=1e-15, atol=0.0)


def test_glu_zero_and_onehot():
    check_glu_zero_and_onehot(gemv.gemv_glu)


def test_glu_batch_columns_independent():
    rng = np.random.default_rng(8)
    M, K = 4, 8
    Wg, Wu = _f32_raw(rng.standard_normal((M, K))), _f32_raw(rng.standard_normal((M, K)))
    X = rng.standard_normal((3, K))
    both = gemv.gemv_glu(Wg, Wu, F32, X, M, K)
    for c in range(3):
        assert np.array_equal(both[c], gemv.gemv_glu(Wg, Wu, F32, X[c], M, K)[0])
    rows = [3, 0]
    assert np.array_equal(gemv.gemv_glu(Wg, Wu, F32, X, M, K, rows=rows), both[:, rows])


# ----------------------------------------------------------------------------- RMS normalisation

def check_rms_worked(fn):
    g = read_golden("rms_norm_worked.txt")
    x, gamma = _floats(g["x"][0]), _floats(g["gamma"][0])
    got = fn(x, gamma, float(g["eps"][0][0]), 2)[0]
    assert np.allclose(got, _floats(g["out"][0]), rtol=1e-15, atol=0.0), got
    got2 = fn(x, gamma, float(g["eps2"][0][0]), 2)[0]
    assert np.allclose(got2, _floats(g["out2"][0]), rtol=1e-15, atol=0.0), got2


def test_rms_worked_example():
    check_rms_worked(norm.rms_norm)


def check_rms_closed_forms(fn):
    rng = np.random.default_rng(9)
    K = 64
    x = rng.standard_normal(K) * 3.0
    ones = np.ones(K)
    # gamma = 1, eps = 0: unit mean square
    y = fn(x, ones, 0.0, K)[0]
    assert abs(np.mean(y * y) - 1.0) < 1e-14
    # scale invariance for alpha > 0 and oddness, eps = 0
    assert np.allclose(fn(x * 1024.0, ones, 0.0, K)[0], y, rtol=1e-14, atol=0.0)
    assert np.allclose(fn(-x, ones, 0.0, K)[0], -y, rtol=1e-15, atol=0.0)
    # a constant vector normalises to its sign
    assert np.allclose(fn(np.full(K, -2.5), ones, 0.0, K)[0], -ones, rtol=1e-15, atol=0.0)
    # gamma multiplies element-wise after the normalisation
    gam = rng.standard_normal(K)
    assert np.allclose(fn(x, gam, 0.0, K)[0], y * gam, rtol=1e-14, atol=0.0)
    # eps much larger than the mean square: x' ~ x * gamma / sqrt(eps)
    tiny = x * 1e-6
    assert np.allclose(fn(tiny, gam, 4.0, K)[0], tiny * gam / 2.0, rtol=1e-9, atol=0.0)


def test_rms_closed_forms():
    check_rms_closed_forms(norm.rms_norm)


def test_rms_columns_independent():
    rng = np.random.default_rng(10)
    K = 32
    X = rng.standard_normal((3, K))
    gam = rng.standard_normal(K)
    both = norm.rms_norm(X, gam, 1e-5, K)
    for c in range(3):
        assert np.array_equal(both[c], norm.rms_norm(X[c], gam, 1e-5, K)[0])


# ----------------------------------------------------------------------------- mutations

def _expect_fail(check, fn):
    with pytest.raises(AssertionError):
        check(fn)


def _bad_glu_swapped(raw_gate, raw_up, wtype, x, M, K, rows=None):
    # activation on the up projection instead of the gate
    return gemv.gemv_glu(raw_up, raw_gate, wtype, x, M, K, rows)


def _bad_glu_silu_of_product(raw_gate, raw_up, wtype, x, M, K, rows=None):
    g = gemv.gemv(raw_gate, wtype, x, M, K, rows=rows)
    u = gemv.gemv(raw_up, wtype, x, M, K, rows=rows)
    return gemv.silu(g * u)


def _bad_glu_sigmoid(raw_gate, raw_up, wtype, x, M, K, rows=None):
    g = gemv.gemv(raw_gate, wtype, x, M, K, rows=rows)
    u = gemv.gemv(raw_up, wtype, x, M, K, rows=rows)
    return gemv.sigmoid(g) * u


def test_mutation_glu_swapped_operands_fails_pin():
    _expect_fail(check_glu_worked, _bad_glu_swapped)


def test_mutation_glu_silu_of_product_fails_pin():
    _expect_fail(check_glu_worked, _bad_glu_silu_of_product)


def test_mutation_glu_sigmoid_for_silu_fails_pin():
    _expect_fail(check_glu_zero_and_onehot, _bad_glu_sigmoid)


def _bad_rms_sum(x, gamma, eps, K):  # sum of squares instead of the mean
    X = np.asarray(x, dtype=np.float64).reshape(-1, K)
    return np.stack([X[c] / math.sqrt(np.sum(X[c] ** 2) + eps) * gamma for c in range(X.shape[0])])


def _bad_rms_no_sqrt(x, gamma, eps, K):
    X = np.asarray(x, dtype=np.float64).reshape(-1, K)
    return np.stack([X[c] / (np.mean(X[c] ** 2) + eps) * gamma for c in range(X.shape[0])])


def _bad_rms_gamma_inside(x, gamma, eps, K):  # weight applied before the statistics
    X = np.asarray(x, dtype=np.float64).reshape(-1, K) * np.asarray(gamma, dtype=np.float64)
    return np.stack([X[c] / math.sqrt(np.mean(X[c] ** 2) + eps) for c in range(X.shape[0])])


def _bad_rms_eps_outside(x, gamma, eps, K):
    X = np.asarray(x, dtype=np.float64).reshape(-1, K)
    return np.stack([X[c] / (math.sqrt(np.mean(X[c] ** 2)) + eps) * gamma for c in range(X.shape[0])])


@pytest.mark.parametrize("bad", [_bad_rms_sum, _bad_rms_no_sqrt, _bad_rms_gamma_inside, _bad_rms_eps_outside])
def test_mutation_rms_fails_pin(bad):
    _expect_fail(check_rms_worked, bad)
