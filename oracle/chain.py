"""Oracle decode-layer chain (fp64).  Test infrastructure only.

Sources: "feat(cuda): fuse activations and residual add into mmv f/q epilogues",
Measurements (the folded ops per layer: beta sigmoid, silu(z) * m, attention residual
add) and "ggml-cpu: fuse element-wise epilogues (ADD, MUL, SILU) into
ggml_compute_forward_mul_mat", What (one layer fuses MUL_MAT+ADD twice for the
attention and FFN residuals, MUL_MAT+SILU for the SwiGLU gate and MUL_MAT+MUL for
gate x up).

One layer, in launch order (attention and norms are not on the path; ``a`` stands in
for the attention output, and the FFN reads the residual stream directly):

    q = Wq x ; k = Wk x ; v = Wv x          (no tail)
    r1 = r + Wo a                           (ADD, in place on r)
    u = Wup r1                              (no tail)
    g = silu(Wgate r1) * u                  (SILU_MUL, multiplicand = up output)
    r2 = r1 + Wdown g                       (ADD, in place on r)
    beta = sigmoid(Wbeta x)                 (SIGMOID)

``weights`` maps each name to (raw bytes, wtype, M, K).
"""

from . import gemv as G

LAYER_ORDER = ("q", "k", "v", "o", "up", "gate", "down", "beta")


def decode_layer(weights, x, a, r):
    def mv(name, vec, epi=G.EPI_NONE, aux=None):
        raw, wt, M, K = weights[name]
        return G.gemv(raw, wt, vec, M, K, epi, aux)[0]

    out = {}
    out["q"] = mv("q", x)
    out["k"] = mv("k", x)
    out["v"] = mv("v", x)
    out["r1"] = mv("o", a, G.EPI_ADD, r)
    out["u"] = mv("up", out["r1"])
    out["g"] = mv("gate", out["r1"], G.EPI_SILU_MUL, out["u"])
    out["r2"] = mv("down", out["g"], G.EPI_ADD, out["r1"])
    out["beta"] = mv("beta", x, G.EPI_SIGMOID)
    return out
