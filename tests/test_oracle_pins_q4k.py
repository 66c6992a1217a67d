"""Pins for the oracle's Q4_K decoder: a super-block packed by hand from chosen fields
(tests/golden/q4_k_block.txt), closed forms (zero codes, zero dmin), agreement with the
independently written packer of the seeded generator on random fields, and mutation
tests that plant plausible unpacking mistakes and check that a pin fails."""

import numpy as np
import pytest

from conftest import read_golden
from decode_gemv_epilogue_gb300 import synth
from oracle import gemv, quant

Q4_K = quant.WTYPE_Q4_K


def _block():
    g = read_golden("q4_k_block.txt")
    raw = np.array([int(t, 16) for t in g["bytes"][0]], dtype=np.uint8)
    want = np.concatenate([[float(v) for v in row] for row in g["values"]])
    return raw, want


def check_q4_k_fixture(dequant):
    raw, want = _block()
    assert raw.size == 144 and want.size == 256
    got = dequant(raw, 1, 256)[0]
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
    # two super-blocks in a row, and two rows
    raw2 = np.concatenate([raw, raw])
    assert np.array_equal(dequant(raw2, 1, 512)[0], np.concatenate([want, want]))
    assert np.array_equal(dequant(raw2, 2, 256), np.stack([want, want]))


def test_q4_k_fixture():
    check_q4_k_fixture(quant.dequantize_q4_k)


def test_q4_k_row_bytes():
    assert quant.row_bytes(Q4_K, 256) == 144 and quant.row_bytes(Q4_K, 4096) == 16 * 144
    with pytest.raises(ValueError):
        quant.row_bytes(Q4_K, 128)


def _fields(seed, M=3, nsb=2):
    g = np.random.default_rng(seed)
    K = 256 * nsb
    codes = g.integers(0, 16, size=(M, K))
    sc = g.integers(0, 64, size=(M, nsb, 8))
    mn = g.integers(0, 64, size=(M, nsb, 8))
    d = g.uniform(1e-3, 1.0, size=(M, nsb)).astype(np.float16)
    dmin = g.uniform(1e-3, 1.0, size=(M, nsb)).astype(np.float16)
    return codes, sc, mn, d, dmin, K


def _direct(codes, sc, mn, d, dmin):
    # value straight from the fields, element k in sub-block (k // 32) of super-block (k // 256)
    M, K = codes.shape
    k = np.arange(K)
    sb, j = k // 256, (k % 256) // 32
    dd = d.astype(np.float64)[:, sb]
    dm = dmin.astype(np.float64)[:, sb]
    return dd * sc[:, sb, j] * codes - dm * mn[:, sb, j]


def check_q4_k_fields(dequant):
    for seed in range(3):
        codes, sc, mn, d, dmin, K = _fields(seed)
        raw = synth.pack_q4_k(codes, sc, mn, d, dmin).reshape(-1)
        assert np.array_equal(dequant(raw, 3, K), _direct(codes, sc, mn, d, dmin))


def test_q4_k_random_fields_through_the_packer():
    check_q4_k_fields(quant.dequantize_q4_k)


def test_q4_k_closed_forms():
    codes, sc, mn, d, dmin, K = _fields(5)
    zero = np.zeros_like(codes)
    raw = synth.pack_q4_k(zero, sc, mn, d, dmin).reshape(-1)
    W = quant.dequantize_q4_k(raw, 3, K)
    k = np.arange(K)
    assert np.array_equal(W, -dmin.astype(np.float64)[:, k // 256] * mn[:, k // 256, (k % 256) // 32])
    raw = synth.pack_q4_k(codes, sc, mn, d, np.zeros_like(dmin)).reshape(-1)
    W = quant.dequantize_q4_k(raw, 3, K)
    assert np.array_equal(W, d.astype(np.float64)[:, k // 256] * sc[:, k // 256, (k % 256) // 32] * codes)


def test_q4_k_gemv_onehot_and_tolerance_scale():
    raw, want = _block()
    for j in (0, 37, 200, 255):
        e = np.zeros(256)
        e[j] = 1.0
        assert gemv.gemv(raw, Q4_K, e, 1, 256)[0, 0] == want[j]
    # the tolerance scale counts both terms of each weight: never below |W|
    x = np.ones(256)
    assert gemv.abs_dot(raw, Q4_K, x, 1, 256)[0, 0] >= np.sum(np.abs(want))


# ----------------------------------------------------------------------------- mutations

def _expect_fail(check, fn):
    with pytest.raises(AssertionError):
        check(fn)


def _mutant(scales_fn=None, codes_fn=None, combine=None, swap_d=False):
    def dequant(raw, M, K, rows=None):
        mat = np.ascontiguousarray(raw).reshape(M, -1)
        nsb = K // 256
        blk = mat.reshape(M, nsb, 144)
        lo, hi = (2, 0) if swap_d else (0, 2)
        d = quant._binary16_to_f64(blk[:, :, lo], blk[:, :, lo + 1])
        dmin = quant._binary16_to_f64(blk[:, :, hi], blk[:, :, hi + 1])
        sc, m = (scales_fn or quant.q4_k_scales_mins)(blk[:, :, 4:16])
        q = (codes_fn or quant.q4_k_codes)(blk[:, :, 16:]).astype(np.float64)
        a = (d[:, :, None] * sc).repeat(32, axis=2) * q
        b = (dmin[:, :, None] * m).repeat(32, axis=2)
        return (combine or (lambda a, b: a - b))(a, b).reshape(M, K)
    return dequant


def _scales_swapped(sb):  # scales and mins exchanged
    sc, m = quant.q4_k_scales_mins(sb)
    return m, sc


def _scales_no_high_bits(sb):  # upper sub-blocks without bits 4..5
    b = sb.astype(np.int64)
    sc, m = quant.q4_k_scales_mins(sb)
    for j in range(4):
        sc[..., j + 4] = b[..., 8 + j] & 15
        m[..., j + 4] = b[..., 8 + j] >> 4
    return sc, m


def _scales_high_bits_from_wrong_byte(sb):  # sc high bits taken from the min bytes
    b = sb.astype(np.int64)
    sc, m = quant.q4_k_scales_mins(sb)
    for j in range(4):
        sc[..., j + 4] = (b[..., 8 + j] & 15) | ((b[..., j + 4] >> 6) << 4)
        m[..., j + 4] = (b[..., 8 + j] >> 4) | ((b[..., j] >> 6) << 4)
    return sc, m


def _codes_interleaved(qs):  # element pairs sharing a byte instead of sub-block halves
    b = qs.astype(np.int64)
    out = np.empty(b.shape[:-1] + (256,), dtype=np.int64)
    out[..., 0::2] = b & 15
    out[..., 1::2] = b >> 4
    return out


def _codes_nibbles_swapped(qs):
    b = qs.astype(np.int64)
    out = quant.q4_k_codes(qs)
    for g in range(4):
        grp = b[..., 32 * g:32 * g + 32]
        out[..., 64 * g:64 * g + 32] = grp >> 4
        out[..., 64 * g + 32:64 * g + 64] = grp & 15
    return out


@pytest.mark.parametrize("mut", [
    _mutant(scales_fn=_scales_swapped), _mutant(scales_fn=_scales_no_high_bits),
    _mutant(scales_fn=_scales_high_bits_from_wrong_byte), _mutant(codes_fn=_codes_interleaved),
    _mutant(codes_fn=_codes_nibbles_swapped), _mutant(combine=lambda a, b: a + b), _mutant(swap_d=True),
])
def test_mutation_q4_k_fails_pin(mut):
    _expect_fail(check_q4_k_fixture, mut)


def test_unmutated_helper_passes():
    check_q4_k_fixture(_mutant())
    check_q4_k_fields(_mutant())
