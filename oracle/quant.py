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
* Q4_K (named in the same section and in its Measured table, also in "feat(cuda):
  fuse activations and residual add into mmv f/q epilogues", Measurements; the
  layout is a reading, the ggml K-quant super-block): each row is K/256 super-blocks
  of 144 bytes -- binary16 d, binary16 dmin, 12 bytes of packed 6-bit scales sc[j]
  and mins m[j] for eight sub-blocks of 32 elements, then 128 bytes of 4-bit codes.
  Scale bytes: byte j (j < 4) holds sc[j] in its low 6 bits and bits 4..5 of sc[j+4]
  in its top 2; byte j+4 (j < 4) holds m[j] and bits 4..5 of m[j+4] likewise; byte
  8+j (j < 4) holds bits 0..3 of sc[j+4] (low nibble) and of m[j+4] (high nibble).
  Codes: four groups of 32 bytes; group g holds sub-block 2g in its low nibbles and
  sub-block 2g+1 in its high nibbles, element t of a sub-block in byte t of the group.
  value = d * sc[j] * q - dmin * m[j]   (exact in float64).

Every decoded value is exact in float64 (and in float32: an 11-bit significand times
a code of at most 8 bits).  Decoding is written out by hand from the byte stream.
"""

import numpy as np

QK = 32  # elements per quant block
QK_K = 256  # elements per K-quant super-block
WTYPE_F32, WTYPE_F16, WTYPE_Q8_0, WTYPE_Q4_0, WTYPE_Q4_K = 0, 1, 2, 3, 4
BLOCK_BYTES = {WTYPE_Q8_0: 2 + QK, WTYPE_Q4_0: 2 + QK // 2}
Q4_K_BYTES = 2 + 2 + 12 + QK_K // 2  # 144


def row_bytes(wtype, K):
    """Bytes of one weight row of K elements."""
    if wtype == WTYPE_F32:
        return 4 * K
    if wtype == WTYPE_F16:
        return 2 * K
    if wtype == WTYPE_Q4_K:
        if K % QK_K:
            raise ValueError("Q4_K rows need K % 256 == 0")
        return (K // QK_K) * Q4_K_BYTES
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


def q4_k_scales_mins(sb):
    """The eight 6-bit scales and mins of super-blocks from their 12 packed bytes
    (uint8 [..., 12]) -> (sc, m), int64 [..., 8] each."""
    b = sb.astype(np.int64)
    sc = np.empty(b.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = b[..., j] & 63
        m[..., j] = b[..., j + 4] & 63
        sc[..., j + 4] = (b[..., 8 + j] & 15) | ((b[..., j] >> 6) << 4)
        m[..., j + 4] = (b[..., 8 + j] >> 4) | ((b[..., j + 4] >> 6) << 4)
    return sc, m


def q4_k_codes(qs):
    """The 256 codes of super-blocks from their 128 code bytes (uint8 [..., 128]) ->
    int64 [..., 256] in element order."""
    b = qs.astype(np.int64)
    out = np.empty(b.shape[:-1] + (QK_K,), dtype=np.int64)
    for g in range(4):
        grp = b[..., 32 * g:32 * g + 32]
        out[..., 64 * g:64 * g + 32] = grp & 15        # sub-block 2g: low nibbles
        out[..., 64 * g + 32:64 * g + 64] = grp >> 4   # sub-block 2g+1: high nibbles
    return out


def q4_k_parts(raw, M, K, rows=None):
    """Per element the two terms of a Q4_K weight, float64 [R, K] each:
    a = d * sc[j] * q (the scaled code) and b = dmin * m[j] (the sub-block min);
    the weight is a - b."""
    mat = _rows_view(raw, WTYPE_Q4_K, M, K, rows)
    R, nsb = mat.shape[0], K // QK_K
    blocks = mat.reshape(R, nsb, Q4_K_BYTES)
    d = _binary16_to_f64(blocks[:, :, 0], blocks[:, :, 1])        # [R, nsb]
    dmin = _binary16_to_f64(blocks[:, :, 2], blocks[:, :, 3])
    sc, m = q4_k_scales_mins(blocks[:, :, 4:16])                   # [R, nsb, 8]
    q = q4_k_codes(blocks[:, :, 16:]).astype(np.float64)           # [R, nsb, 256]
    scale = (d[:, :, None] * sc).repeat(QK, axis=2)                # per element
    mins = (dmin[:, :, None] * m).repeat(QK, axis=2)
    return (scale * q).reshape(R, K), mins.reshape(R, K)


def dequantize_q4_k(raw, M, K, rows=None):
    a, b = q4_k_parts(raw, M, K, rows)
    return a - b


def dequantize(raw, wtype, M, K, rows=None):
    """Decoded weights as float64 [len(rows) or M, K]."""
    fn = {WTYPE_F32: dequantize_f32, WTYPE_F16: dequantize_f16,
          WTYPE_Q8_0: dequantize_q8_0, WTYPE_Q4_0: dequantize_q4_0,
          WTYPE_Q4_K: dequantize_q4_k}[wtype]
    return fn(raw, M, K, rows)
