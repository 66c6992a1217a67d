"""Oracle RMS normalisation prologue (fp64).  Test infrastructure only.

Source: "ggml-cpu: fuse element-wise epilogues (ADD, MUL, SILU) into
ggml_compute_forward_mul_mat", What: the executor already fuses RMS_NORM with the MUL
that follows it, i.e. the normalised activation times an element-wise weight gamma,
ahead of the matmul.  The pages name the pair but do not print the normalisation;
the reading taken is the usual root-mean-square normalisation with an additive eps
inside the square root, per column of the batch:

    rms[c]  = sqrt( (1/K) * sum_k x[c, k]^2  +  eps )
    x'[c,k] = (x[c, k] / rms[c]) * gamma[k]

Everything in float64 (numpy), column by column, in the order written.
"""

import numpy as np


def rms_norm(x, gamma, eps, K):
    """x: [ncols, K] or [K]; gamma: [K]; returns float64 [ncols, K]."""
    X = np.asarray(x, dtype=np.float64).reshape(-1, K)
    g = np.asarray(gamma, dtype=np.float64).reshape(K)
    out = np.empty_like(X)
    for c in range(X.shape[0]):
        mean_sq = float(np.sum(X[c] * X[c])) / K if K > 0 else 0.0
        rms = np.sqrt(mean_sq + float(eps))
        out[c] = (X[c] / rms) * g
    return out
