"""Oracle weight decoders (fp64).  Test infrastructure only; see ``oracle/__init__``.

The weight formats F32, F16, Q8_0 and Q4_0 are the ones named in "ggml-cpu: fuse
element-wise epilogues (ADD, MUL, SILU) into ggml_compute_forward_mul_mat",
Correctness.  The page names them but does not print their layouts, so this module
states the reading it takes (the ggml block convention the pages' projects use):

* F32: little-endian IEEE binary32, row-major [M][K].
* F16: little-endian IEEE binary16, row-major [M][K]; value = the binary16 value.
* Q8_0: each row is K/32 blocks of 34 bytes: binary16 scale d, then 32 int8 codes q.
  value(j) = d * q[j].
* Q4_0: each row is K/32 blocks of 18 bytes: binary16 scale d, then 16 bytes qs.
  Byte j of qs holds element j in its low nibble and element j+16 in its high nibble.
  value = d * (nibble - 8).

Every decoded value is exact in float64 (and in float32: an 11-bit significand times
a code of at most 8 bits).  Decoding is written out by hand from the byte stream.
"""

import numpy as np

QK = 32  # elements per quant block
WTYPE_F32, WTYPE_F16, WTYPE_Q8_0, WTYPE_Q4_0 = 0, 1, 2, 3
BLOCK_BYTES = {WTYPE_Q8_0: 2 + QK, WTYPE_Q4_0: 2 + QK // 2}


def row_bytes(wtype, K):
    """Bytes of one weight row of K elements."""
    if wtype == WTYPE_F32:
        return 4 * K
    if wtype == WTYPE_F16:
        return 2 * K
    if K % QK:
        raise ValueError("quantised rows need K % 32 == 0")
    return (K // QK) * BLOCK_BYTES[wtype]


def _binary16_to_f64(lo, hi):
    """Decode little-endian binary16 (two byte arrays) to float64 by its definition:
    sign, 5-bit exponent (bias 15), 10-bit fraction; subnormals at exponent 0."""
    bits = lo.astype(np.int64) | (hi.astype(np.int64) << 8)
    sign = np.where(bits & 0x8000, -1.0, 1.0)
    exp = (bits >> 10) & 0x1F
    frac = (bits & 0x3FF).astype(np.float64)
    normal = sign * (1.0 + frac / 1024.0) * np.exp2(exp.astype(np.float64) - 15.0)
    sub = sign * (frac / 1024.0) * 2.0 ** -14
    special = np.where(frac == 0, sign * np.inf, np.nan)
    return np.where(exp == 0, sub, np.where(exp == 31, special, normal))


def _rows_view(raw, wtype, M, K, rows):
    rb = row_bytes(wtype, K)
    raw = np.ascontiguousarray(raw).view(np.uint8).reshape(-1)
    if raw.size != M * rb:
        raise ValueError("weight buffer has %d bytes, expected %d" % (raw.size, M * rb))
    mat = raw.reshape(M, rb)
    if rows is not None:
        mat = mat[np.asarray(rows, dtype=np.int64)]
    return mat


def dequantize_f32(raw, M, K, rows=None):
    mat = _rows_view(raw, WTYPE_F32, M, K, rows)
    return np.ascontiguousarray(mat).view("<f4").astype(np.float64)


def dequantize_f16(raw, M, K, rows=None):
    mat = _rows_view(raw, WTYPE_F16, M, K, rows)
    return _binary16_to_f64(mat[:, 0::2], mat[:, 1::2])


def dequantize_q8_0(raw, M, K, rows=None):
    mat = _rows_view(raw, WTYPE_Q8_0, M, K, rows)
    blocks = mat.reshape(mat.shape[0], K // QK, 34)
    d = _binary16_to_f64(blocks[:, :, 0], blocks[:, :, 1])          # [R, nb]
    q = blocks[:, :, 2:].astype(np.int64)
    q = np.where(q >= 128, q - 256, q).astype(np.float64)          # int8 two's complement
    return (d[:, :, None] * q).reshape(mat.shape[0], K)


def dequantize_q4_0(raw, M, K, rows=None):
    mat = _rows_view(raw, WTYPE_Q4_0, M, K, rows)
    blocks = mat.reshape(mat.shape[0], K // QK, 18)
    d = _binary16_to_f64(blocks[:, :, 0], blocks[:, :, 1])
    qs = blocks[:, :, 2:].astype(np.int64)                          # [R, nb, 16]
    codes = np.empty(qs.shape[:2] + (QK,), dtype=np.int64)
    codes[:, :, :16] = qs & 0x0F        # element j    <- low nibble of byte j
    codes[:, :, 16:] = qs >> 4          # element j+16 <- high nibble of byte j
    return (d[:, :, None] * (codes - 8).astype(np.float64)).reshape(mat.shape[0], K)


def dequantize(raw, wtype, M, K, rows=None):
    """Decoded weights as float64 [len(rows) or M, K]."""
    fn = {WTYPE_F32: dequantize_f32, WTYPE_F16: dequantize_f16,
          WTYPE_Q8_0: dequantize_q8_0, WTYPE_Q4_0: dequantize_q4_0}[wtype]
    return fn(raw, M, K, rows)
