"""Oracle GEMV and element-wise tails (fp64).  Test infrastructure only.

Definition followed ("feat(cuda): fuse activations and residual add into mmv f/q
epilogues", Summary and What changed; "ggml-cpu: fuse element-wise epilogues (ADD,
MUL, SILU) into ggml_compute_forward_mul_mat", What):

    y[c, i]   = sum_k W[i, k] * x[c, k]            (decode case: one column, or a
                                                   small batch of independent columns)
    out[c, i] = tail(y[c, i])  with tail one of
        NONE      y
        SIGMOID   1 / (1 + exp(-y))
        SILU      y * sigmoid(y)
        SILU_MUL  silu(y) * m[c, i]    (activation, then the per-row multiplicand;
                                        never silu(y * m))
        ADD       y + r[c, i]          (residual add; the reshape view in between is an
                                        index identity on contiguous memory)

All arithmetic is float64; exp is libm's (numpy).  The dot product is numpy's own
(non-BLAS) einsum loop, one thread.
"""

import numpy as np

from . import quant

EPI_NONE, EPI_SIGMOID, EPI_SILU, EPI_SILU_MUL, EPI_ADD = 0, 1, 2, 3, 4
EPI_NAMES = {EPI_NONE: "none", EPI_SIGMOID: "sigmoid", EPI_SILU: "silu",
             EPI_SILU_MUL: "silu_mul", EPI_ADD: "add"}
NEEDS_AUX = (EPI_SILU_MUL, EPI_ADD)


def sigmoid(y):
    y = np.asarray(y, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-y))


def silu(y):
    y = np.asarray(y, dtype=np.float64)
    return y * sigmoid(y)


def apply_epilogue(y, epilogue, aux=None):
    """The fused tail applied to the fp64 GEMV result y (any shape; aux same shape)."""
    y = np.asarray(y, dtype=np.float64)
    if epilogue == EPI_NONE:
        return y.copy()
    if epilogue == EPI_SIGMOID:
        return sigmoid(y)
    if epilogue == EPI_SILU:
        return silu(y)
    if epilogue in NEEDS_AUX:
        a = np.asarray(aux, dtype=np.float64)
        if a.shape != y.shape:
            raise ValueError("aux must have the output's shape (no broadcast)")
        return silu(y) * a if epilogue == EPI_SILU_MUL else y + a
    raise ValueError("unknown epilogue %r" % (epilogue,))


def _as_cols(v, n):
    v = np.asarray(v, dtype=np.float64)
    return v.reshape(-1, n)


def gemv(raw, wtype, x, M, K, epilogue=EPI_NONE, aux=None, rows=None):
    """out[c, i] for columns c of x (shape [ncols, K] or [K]) and rows i (all, or the
    listed subset).  Returns float64 [ncols, len(rows)].  aux has shape [ncols, M]."""
    W = quant.dequantize(raw, wtype, M, K, rows)          # [R, K] float64
    X = _as_cols(x, K)                                    # [ncols, K]
    y = np.einsum("ik,ck->ci", W, X)                      # plain sum over k, per (c, i)
    a = None
    if epilogue in NEEDS_AUX:
        a = _as_cols(aux, M)
        if rows is not None:
            a = a[:, np.asarray(rows, dtype=np.int64)]
    return apply_epilogue(y, epilogue, a)


def gemv_glu(raw_gate, raw_up, wtype, x, M, K, rows=None):
    """The gated dual GEMV: out[c, i] = silu(g[c, i]) * u[c, i] with g = Wg x and
    u = Wu x, both weights in the same format and shape.  This is the SwiGLU gate and
    the gate x up product of one FFN ("ggml-cpu: fuse element-wise epilogues (ADD, MUL,
    SILU) into ggml_compute_forward_mul_mat", What) taken as one operation -- the
    gated branch that "feat(cuda): fuse activations and residual add into mmv f/q
    epilogues", Summary, leaves to its existing GLU path.  Returns float64
    [ncols, len(rows)]."""
    g = gemv(raw_gate, wtype, x, M, K, EPI_NONE, rows=rows)
    u = gemv(raw_up, wtype, x, M, K, EPI_NONE, rows=rows)
    return silu(g) * u


def _abs_weights(raw, wtype, M, K, rows):
    """|W| for the tolerance scale.  For Q4_K, whose weight is a difference a - b of a
    scaled code and a sub-block min, |a| + |b|: a kernel may add the two terms'
    products separately (the min term through a per-sub-block sum of x), and its
    rounding then scales with both terms, not with their difference."""
    if wtype == quant.WTYPE_Q4_K:
        a, b = quant.q4_k_parts(raw, M, K, rows)
        return np.abs(a) + np.abs(b)
    return np.abs(quant.dequantize(raw, wtype, M, K, rows))


def abs_dot(raw, wtype, x, M, K, rows=None):
    """sum_k |W[i,k] * x[c,k]| in fp64: the scale of the parity tolerance."""
    X = _as_cols(x, K)
    return np.einsum("ik,ck->ci", _abs_weights(raw, wtype, M, K, rows), np.abs(X))


def block_max_dot(raw, wtype, x, M, K, rows=None, block=32):
    """sum over blocks b of max_{k in b} |x[c,k]| * sum_{k in b} |W[i,k]|, blocks of
    `block` consecutive elements: the scale of the error of a product that rounds x
    relative to the largest |x| of each block (a parity-tolerance term)."""
    X = np.abs(_as_cols(x, K))
    if K % block:
        raise ValueError("K must be a multiple of the block")
    mx = X.reshape(X.shape[0], K // block, block).max(axis=2)                 # [C, nb]
    Wa = _abs_weights(raw, wtype, M, K, rows)
    wb = Wa.reshape(Wa.shape[0], K // block, block).sum(axis=2)              # [R, nb]
    return np.einsum("cb,ib->ci", mx, wb)


def abs_w_dot(raw, wtype, e, M, K, rows=None):
    """sum_k |W[i,k]| * e[c,k] for a non-negative per-element error e [ncols, K]."""
    return np.einsum("ik,ck->ci", _abs_weights(raw, wtype, M, K, rows), _as_cols(e, K))
