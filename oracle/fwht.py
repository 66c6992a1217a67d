"""Oracle signed Walsh-Hadamard transform (fp64).  Test infrastructure only.

Source: "vulkan: fuse the sign multiply into the Hadamard FWHT", Overview.  The graph
computes MUL(signs) -> RESHAPE -> MUL_MAT(hint=hadamard): the activation is multiplied
element-wise by a +-1 sign vector (broadcast over the sign vector's length), the
result is viewed as consecutive blocks of B elements, and each block is multiplied by
the B x B Hadamard matrix.  The sign multiply happens before the transform.

Readings taken where the page is silent (the page gives neither the matrix order nor
the normalisation): the Hadamard matrix is Sylvester's, H[i, j] = (-1)^popcount(i & j),
and the product is normalised by 1/sqrt(B) so the transform is orthonormal.  Sign
index of element k is k mod nsigns.

``fwht_signed`` is the plain definition (dense H times each block).  ``fwht_butterfly``
is the fast butterfly, kept only so the tests can pin one against the other.
"""

import numpy as np


def _popcount(a):
    a = np.asarray(a, dtype=np.int64)
    c = np.zeros_like(a)
    while np.any(a):
        c += a & 1
        a = a >> 1
    return c


_H_CACHE = {}


def hadamard(n):
    """Sylvester-ordered Hadamard matrix, closed form (-1)^popcount(i & j), float64."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    if n not in _H_CACHE:
        i = np.arange(n, dtype=np.int64)
        H = np.where(_popcount(i[:, None] & i[None, :]) % 2 == 0, 1.0, -1.0)
        H.setflags(write=False)
        _H_CACHE[n] = H
    return _H_CACHE[n].copy()


def signed_input(x, signs):
    """x * s with s broadcast: element k uses s[k mod len(s)]."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    if x.size % s.size:
        raise ValueError("len(x) must be a multiple of len(signs)")
    return x * np.tile(s, x.size // s.size)


def fwht_signed(x, signs, block):
    """x'_b = H_B (x_b * s) / sqrt(B) for every consecutive block b of B elements.
    ``signs=None`` means all +1 (the plain transform)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    if x.size % block:
        raise ValueError("len(x) must be a multiple of the block")
    v = x if signs is None else signed_input(x, signs)
    H = hadamard(block)
    blocks = v.reshape(-1, block)
    # plain sum over t of H[j, t] * v[b, t] (numpy's own loop: one thread, no BLAS)
    return (np.einsum("jt,bt->bj", H, blocks) / np.sqrt(block)).reshape(-1)


def fwht_butterfly(x, signs, block):
    """Same transform by log2(B) butterfly stages (a, b) -> (a + b, a - b)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    v = (x if signs is None else signed_input(x, signs)).reshape(-1, block).copy()
    h = 1
    while h < block:
        v = v.reshape(v.shape[0], -1, 2, h)
        a = v[:, :, 0, :].copy()
        b = v[:, :, 1, :].copy()
        v[:, :, 0, :] = a + b
        v[:, :, 1, :] = a - b
        v = v.reshape(-1, block)
        h *= 2
    return (v / np.sqrt(block)).reshape(-1)


def fwht_abs_scale(x, block):
    """sum over the block of |x_t| / sqrt(B), per element: the scale of the FWHT
    output tolerance (each output is a +-1 combination of its block, over sqrt(B))."""
    x = np.abs(np.asarray(x, dtype=np.float64).reshape(-1, block))
    return np.repeat(x.sum(axis=1) / np.sqrt(block), block)
