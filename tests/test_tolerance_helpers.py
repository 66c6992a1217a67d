"""The tolerance scales used by the parity bounds, checked by brute force on tiny inputs
(they are test infrastructure, not part of what the path computes)."""

import numpy as np

from decode_gemv_epilogue_gb300 import synth
from oracle import gemv as ogemv, quant


def test_block_max_dot_brute_force():
    M, K = 3, 64
    for wt in (synth.F32, synth.Q8_0, synth.Q4_0):
        raw = synth.weights(wt, M, K, seed=11)
        x = synth.normal(2 * K, seed=12).reshape(2, K)
        W = quant.dequantize(raw, wt, M, K)
        got = ogemv.block_max_dot(raw, wt, x, M, K)
        for c in range(2):
            for i in range(M):
                want = 0.0
                for b in range(K // 32):
                    mx = max(abs(float(x[c, k])) for k in range(32 * b, 32 * b + 32))
                    want += mx * sum(abs(float(W[i, k])) for k in range(32 * b, 32 * b + 32))
                assert abs(got[c, i] - want) <= 1e-12 * want


def test_block_max_dot_bounds_abs_dot():
    # max_b |x| * sum_b |w| >= sum_b |w x| for every block
    M, K = 5, 256
    raw = synth.weights(synth.Q4_0, M, K, seed=13)
    x = synth.normal(K, seed=14)
    assert np.all(ogemv.block_max_dot(raw, synth.Q4_0, x, M, K) >= ogemv.abs_dot(raw, synth.Q4_0, x, M, K))
