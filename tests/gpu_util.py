"""Helpers for the GPU parity tests: upload seeded inputs, call the C ABI through the
binding, and compute the oracle's value and the parity bound for the same inputs."""

import numpy as np

from oracle import fwht as ofwht
from oracle import gemv as ogemv

TOL_REL = 2e-5   # |gpu - oracle| <= 2e-5 * sum_k |W_ik x_k| + 1e-6 (fp32 accumulation)
TOL_ABS = 1e-6


def dev_tensor(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def gemv_bound(raw, wt, x, M, K, rows=None, x_err=None):
    """Per-element tolerance [ncols, rows]: the literal bound, for every weight format,
    plus the propagated error of an on-chip prologue (x_err: per-element bound on
    |x' - x'_exact|)."""
    b = TOL_REL * ogemv.abs_dot(raw, wt, x, M, K, rows) + TOL_ABS
    if x_err is not None:
        b = b + ogemv.abs_w_dot(raw, wt, x_err, M, K, rows)
    return b


def int_rounding_scale(raw, wt, x, M, K, rows=None):
    """sum over 32-element blocks of max_block |x| * sum_block |w|: the scale of the error
    the integer dot products would make if they rounded every x of a block relative to
    its largest |x| (2^-23 of this).  Reported next to the gate, never added to it."""
    return ogemv.block_max_dot(raw, wt, np.abs(np.asarray(x, dtype=np.float64)), M, K, rows)


def fwht_err_bound(x, block):
    """Bound on the fp32 error of the transform itself (same form with W = H / sqrt(B))."""
    return TOL_REL * ofwht.fwht_abs_scale(x, block) + TOL_ABS


def assert_within(got, want, bound, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = ~(err <= bound)
    if np.any(bad):
        i = np.flatnonzero(bad.reshape(-1))[0]
        raise AssertionError("%s: %d/%d elements out of tolerance; first flat index %d: got %r want %r "
                             "bound %r (max err/bound %.3g)"
                             % (what, int(bad.sum()), bad.size, i, got.reshape(-1)[i], want.reshape(-1)[i],
                                np.asarray(bound).reshape(-1)[i], float(np.max(err / bound))))
    return float(np.max(err / bound)) if err.size else 0.0


# RMS-normalisation prologue: the kernel scales the finished dot product by its own
# 1/rms (fp32 sum of squares in a fixed, mostly pairwise order, then 1/sqrt).  Its
# relative error (a few ulp from the square root and division, plus the sum's rounding,
# under 1e-6 for K <= 16384) adds at most this fraction of sum_k |W_ik x'_k|.
TOL_NORM_REL = 2e-6


def norm_bound(raw, wt, xn, M, K, rows=None):
    """Tolerance with the RMS prologue: the literal bound on x' = oracle-normalised x,
    plus the 1/rms term."""
    from oracle import gemv as _g
    return gemv_bound(raw, wt, xn, M, K, rows) + TOL_NORM_REL * _g.abs_dot(raw, wt, xn, M, K, rows)


def glu_bound(raw_g, raw_u, wt, x, M, K, rows=None, x_err=None, extra_rel=0.0):
    """Tolerance of silu(g) * u given the bounds Bg, Bu of the two GEMVs (each the
    literal bound, plus extra_rel * sum|W x| for a prologue): first-order propagation with
    |silu'| <= 1.1, the product of the two errors, and the rounding of the tail itself
    (expf, the division and two products: under 1e-6 relative)."""
    from oracle import gemv as _g
    gv = _g.gemv(raw_g, wt, x, M, K, rows=rows)
    uv = _g.gemv(raw_u, wt, x, M, K, rows=rows)
    bg = gemv_bound(raw_g, wt, x, M, K, rows, x_err) + extra_rel * _g.abs_dot(raw_g, wt, x, M, K, rows)
    bu = gemv_bound(raw_u, wt, x, M, K, rows, x_err) + extra_rel * _g.abs_dot(raw_u, wt, x, M, K, rows)
    sg = _g.silu(gv)
    return 1.1 * bg * (np.abs(uv) + bu) + np.abs(sg) * bu + 1e-6 * np.abs(sg * uv)
