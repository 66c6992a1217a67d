"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module only draws random numbers and lays them out in the storage formats; it
holds none of the method's arithmetic (no decoding, no dot products, no tails, no
transform).  One ``numpy.random.Generator(PCG64(seed))`` per tensor.

Storage formats (the ggml block convention; the format names come from "ggml-cpu:
fuse element-wise epilogues (ADD, MUL, SILU) into ggml_compute_forward_mul_mat",
Correctness):
  F32 / F16: row-major [M][K] little-endian.
  Q8_0: per 32 elements, binary16 d then 32 int8 codes.
  Q4_0: per 32 elements, binary16 d then 16 bytes; byte j = code[j] | code[j+16] << 4.
  Q4_K: per 256 elements, binary16 d, binary16 dmin, 12 bytes of packed 6-bit scales
        and mins of the eight 32-element sub-blocks, then 128 code bytes (four groups
        of 32 bytes: sub-block 2g in the low nibbles, 2g+1 in the high nibbles).
"""

import numpy as np

F32, F16, Q8_0, Q4_0, Q4_K = 0, 1, 2, 3, 4
QK = 32
QK_K = 256


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(wtype, K):
    if wtype == F32:
        return 4 * K
    if wtype == F16:
        return 2 * K
    if wtype == Q4_K:
        return (K // QK_K) * 144
    return (K // QK) * (34 if wtype == Q8_0 else 18)


def pack_q8_0(codes, d16):
    """codes int8-valued [M, K], d16 float16 [M, K/32] -> uint8 [M, row_bytes]."""
    M, K = codes.shape
    nb = K // QK
    out = np.empty((M, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d16.astype("<f2")).view(np.uint8).reshape(M, nb, 2)
    out[:, :, 2:] = codes.astype(np.int8).view(np.uint8).reshape(M, nb, QK)
    return out.reshape(M, nb * 34)


def pack_q4_0(codes, d16):
    """codes in 0..15 [M, K], d16 float16 [M, K/32] -> uint8 [M, row_bytes]."""
    M, K = codes.shape
    nb = K // QK
    c = codes.astype(np.uint8).reshape(M, nb, QK)
    out = np.empty((M, nb, 18), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d16.astype("<f2")).view(np.uint8).reshape(M, nb, 2)
    out[:, :, 2:] = c[:, :, :16] | (c[:, :, 16:] << 4)
    return out.reshape(M, nb * 18)


def pack_q4_k(codes, sc, mn, d16, dmin16):
    """codes in 0..15 [M, K]; 6-bit sc, mn [M, K/256, 8]; d16, dmin16 float16 [M, K/256]
    -> uint8 [M, row_bytes]."""
    M, K = codes.shape
    nsb = K // QK_K
    sc = sc.astype(np.uint8)
    mn = mn.astype(np.uint8)
    out = np.empty((M, nsb, 144), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d16.astype("<f2")).view(np.uint8).reshape(M, nsb, 2)
    out[:, :, 2:4] = np.ascontiguousarray(dmin16.astype("<f2")).view(np.uint8).reshape(M, nsb, 2)
    for j in range(4):
        out[:, :, 4 + j] = (sc[:, :, j] & 63) | ((sc[:, :, j + 4] >> 4) << 6)
        out[:, :, 8 + j] = (mn[:, :, j] & 63) | ((mn[:, :, j + 4] >> 4) << 6)
        out[:, :, 12 + j] = (sc[:, :, j + 4] & 15) | ((mn[:, :, j + 4] & 15) << 4)
    c = codes.astype(np.uint8).reshape(M, nsb, 4, 2, 32)   # [.., group, half, t]
    out[:, :, 16:] = (c[:, :, :, 0, :] | (c[:, :, :, 1, :] << 4)).reshape(M, nsb, 128)
    return out.reshape(M, nsb * 144)


def weights(wtype, M, K, seed, dist=None):
    """Weight bytes (uint8 [M * row_bytes]) with the workload distributions:
    F32 ~ U(-1/sqrt(K), 1/sqrt(K)); F16 ~ N(0, 0.02);
    Q8_0 q ~ U{-127..127}, d ~ U(0.001, 0.01); Q4_0 q ~ U{0..15}, d ~ U(0.001, 0.02);
    Q4_K q ~ U{0..15}, sc ~ U{1..63}, d ~ U(1e-4, 4e-4), and per super-block dmin = the
    largest d * sc[j] * 7.5 / 63 of its sub-blocks times U(1, 1.25), with
    m[j] = round(d * sc[j] * 7.5 / dmin) in 0..63: each sub-block's min centres its scaled
    codes, so the weights have mean ~0 as the quantised weights of a trained layer do
    (drawing m and dmin independently gives weights whose mean is ~40% of their size,
    which a layer's residual stream turns into gates deep in silu's saturation).
    The fp16 scales are drawn in float64 and rounded to binary16 (nearest even)."""
    g = rng(seed)
    if wtype == F32:
        lim = 1.0 / np.sqrt(max(K, 1))
        w = g.uniform(-lim, lim, size=(M, K)).astype(np.float32)
        return w.view(np.uint8).reshape(-1)
    if wtype == F16:
        std = 0.02 if dist is None else dist
        w = (g.standard_normal(size=(M, K)) * std).astype(np.float16)
        return w.view(np.uint8).reshape(-1)
    if wtype == Q4_K:
        nsb = K // QK_K
        codes = g.integers(0, 16, size=(M, K), dtype=np.int16)
        sc = g.integers(1, 64, size=(M, nsb, 8), dtype=np.int16)
        d = g.uniform(1e-4, 4e-4, size=(M, nsb)).astype(np.float16)
        centre = d.astype(np.float64)[:, :, None] * sc * 7.5           # d * sc[j] * 7.5
        dmin = (centre.max(axis=2) / 63.0 * g.uniform(1.0, 1.25, size=(M, nsb))).astype(np.float16)
        mn = np.clip(np.rint(centre / dmin.astype(np.float64)[:, :, None]), 0, 63).astype(np.int16)
        return pack_q4_k(codes, sc, mn, d, dmin).reshape(-1)
    nb = K // QK
    if wtype == Q8_0:
        lo, hi = (0.001, 0.01) if dist is None else dist
        codes = g.integers(-127, 128, size=(M, K), dtype=np.int16)
        d = g.uniform(lo, hi, size=(M, nb)).astype(np.float16)
        return pack_q8_0(codes, d).reshape(-1)
    if wtype == Q4_0:
        lo, hi = (0.001, 0.02) if dist is None else dist
        codes = g.integers(0, 16, size=(M, K), dtype=np.int16)
        d = g.uniform(lo, hi, size=(M, nb)).astype(np.float16)
        return pack_q4_0(codes, d).reshape(-1)
    raise ValueError(wtype)


def normal(n, seed, dtype=np.float32):
    return rng(seed).standard_normal(size=n).astype(dtype)


def rademacher(n, seed):
    """+-1 signs as float32."""
    return np.where(rng(seed).integers(0, 2, size=n) == 0, -1.0, 1.0).astype(np.float32)
