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
    """Per-element tolerance [ncols, rows]: the literal bound, plus the propagated
    error of an on-chip prologue (x_err: per-element bound on |x' - x'_exact|)."""
    b = TOL_REL * ogemv.abs_dot(raw, wt, x, M, K, rows) + TOL_ABS
    if x_err is not None:
        b = b + ogemv.abs_w_dot(raw, wt, x_err, M, K, rows)
    return b


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
