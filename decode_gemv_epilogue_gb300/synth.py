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
"""

import numpy as np

F32, F16, Q8_0, Q4_0 = 0, 1, 2, 3
QK = 32


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(wtype, K):
    if wtype == F32:
        return 4 * K
    if wtype == F16:
        return 2 * K
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


def weights(wtype, M, K, seed, dist=None):
    """Weight bytes (uint8 [M * row_bytes]) with the workload distributions:
    F32 ~ U(-1/sqrt(K), 1/sqrt(K)); F16 ~ N(0, 0.02);
    Q8_0 q ~ U{-127..127}, d ~ U(0.001, 0.01); Q4_0 q ~ U{0..15}, d ~ U(0.001, 0.02).
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
