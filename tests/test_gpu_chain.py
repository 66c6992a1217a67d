"""Persistent chains (gf_prepare_chain): the calls of a decode layer run by one launch.
The results must equal those of the same prepared calls launched one after another, bit
for bit (every stage does the same per-row arithmetic), the grid barriers must sit exactly
before the stages that depend on an earlier one, and repeated launches (serial, PDL
back to back, graph replays) must keep giving those results."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, gemv_bound
from oracle import gemv as ogemv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

NONE, SIG, SILU_MUL, ADD = ogemv.EPI_NONE, ogemv.EPI_SIGMOID, ogemv.EPI_SILU_MUL, ogemv.EPI_ADD


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


class Layer:
    """Weights and buffers of one decode layer: q, k, v (d x d), o + residual add,
    up and gate silu*m (f x d), down + residual add (d x f), a sigmoid head (nb x d)."""

    def __init__(self, wt, d, f, nb, seed):
        self.wt, self.d, self.f, self.nb = wt, d, f, nb
        self.shapes = {"q": (d, d), "k": (d, d), "v": (d, d), "o": (d, d), "up": (f, d), "gate": (f, d),
                       "down": (d, f), "beta": (nb, d)}
        self.raw = {n: synth.weights(wt, M, K, seed=seed + i) for i, (n, (M, K)) in enumerate(self.shapes.items())}
        self.W = {n: dev_tensor(r) for n, r in self.raw.items()}
        self.x0 = synth.normal(d, seed=seed + 20)
        self.a0 = synth.normal(d, seed=seed + 21)
        self.r0 = synth.normal(d, seed=seed + 22)
        self.x, self.a, self.r = dev_tensor(self.x0), dev_tensor(self.a0), dev_tensor(self.r0)
        self.out = {n: torch.empty(self.shapes[n][0], device="cuda") for n in ("q", "k", "v", "up", "gate", "beta")}

    def reset(self):
        self.r.copy_(torch.from_numpy(self.r0))
        for t in self.out.values():
            t.fill_(float("nan"))
        torch.cuda.synchronize()

    def calls(self, G, pdl=True):
        """The eight calls in layer order."""
        s, o, wt = self.shapes, self.out, self.wt

        def p(n, vec, epi, aux, dst):
            M, K = s[n]
            return G.prepare(self.W[n], wt, vec, M, K, epi, aux, dst, pdl=pdl, split_k=False)

        return [p("q", self.x, NONE, None, o["q"]), p("k", self.x, NONE, None, o["k"]),
                p("v", self.x, NONE, None, o["v"]), p("o", self.a, ADD, self.r, self.r),
                p("up", self.r, NONE, None, o["up"]), p("gate", self.r, SILU_MUL, o["up"], o["gate"]),
                p("down", o["gate"], ADD, self.r, self.r), p("beta", self.x, SIG, None, o["beta"])]

    def calls_fused(self, G, pdl=True):
        """The same layer as four calls: q, k, v and the head sharing x; o + add; the gated
        dual GEMV (gate and up in one pass); down + add."""
        s, o, wt, d = self.shapes, self.out, self.wt, self.d
        multi = G.prepare_multi([(self.W["q"], d, NONE, None, o["q"]), (self.W["k"], d, NONE, None, o["k"]),
                                 (self.W["v"], d, NONE, None, o["v"]), (self.W["beta"], self.nb, SIG, None, o["beta"])],
                                wt, self.x, d, pdl=pdl)
        oc = G.prepare(self.W["o"], wt, self.a, d, d, ADD, self.r, self.r, pdl=pdl, split_k=False)
        glu = G.prepare_glu(self.W["gate"], self.W["up"], wt, self.r, self.f, d, o["gate"], pdl=pdl, split_k=False)
        down = G.prepare(self.W["down"], wt, o["gate"], d, self.f, ADD, self.r, self.r, pdl=pdl, split_k=False)
        return [multi, oc, glu, down]

    def snapshot(self, names=("q", "k", "v", "up", "gate", "beta")):
        torch.cuda.synchronize()
        snap = {n: self.out[n].cpu().numpy().view(np.uint32).copy() for n in names}
        snap["r"] = self.r.cpu().numpy().view(np.uint32).copy()
        return snap


def _equal(a, b, what):
    for n in a:
        assert np.array_equal(a[n], b[n]), "%s: output %s differs" % (what, n)


@pytest.fixture(scope="module")
def q4_layer():
    return Layer(synth.Q4_0, 4096, 14336, 32, seed=300)


def test_q4_0_layer_chain_equals_serial_calls(G, q4_layer):
    L = q4_layer
    calls = L.calls(G)
    L.reset()
    G.launch_prepared(calls)
    want = L.snapshot()
    chain = G.prepare_chain(calls)
    info = G.chain_info(chain)
    # barriers before up (reads r, written by o), gate (reads up's output) and down (reads
    # gate's); k and v reuse q's staged x, gate reuses up's
    assert (info["stages"], info["barriers"], info["barrier_mask"]) == (8, 3, 0b01110000)
    assert info["reuse_mask"] == 0b00100110
    assert info["grid"] == torch.cuda.get_device_properties(0).multi_processor_count
    L.reset()
    chain.launch()
    got = L.snapshot()
    _equal(want, got, "chain")
    assert G.device_status() == 0


def test_q4_0_layer_chain_against_the_oracle(G, q4_layer):
    """Stage by stage on sampled rows: the chain's outputs against the oracle, with the
    inputs each stage saw (taken from a serial run that the chain matches bit for bit)."""
    L = q4_layer
    calls = L.calls(G)
    L.reset()
    for c in calls[:4]:
        c.launch()
    torch.cuda.synchronize()
    r1 = L.r.cpu().numpy().astype(np.float64)
    L.reset()
    G.prepare_chain(calls).launch()
    torch.cuda.synchronize()
    h = {n: t.cpu().numpy().astype(np.float64) for n, t in L.out.items()}
    r2 = L.r.cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(5)

    def check(name, vec, epi, aux, got):
        M, K = L.shapes[name]
        rows = np.sort(rng.choice(M, size=min(M, 256), replace=False))
        want = ogemv.gemv(L.raw[name], L.wt, vec, M, K, epi, aux, rows=rows)
        assert_within(got[rows], want[0], gemv_bound(L.raw[name], L.wt, vec, M, K, rows)[0], name)

    check("q", L.x0, NONE, None, h["q"])
    check("v", L.x0, NONE, None, h["v"])
    check("up", r1.astype(np.float32), NONE, None, h["up"])
    check("gate", r1.astype(np.float32), SILU_MUL, h["up"], h["gate"])
    check("down", h["gate"].astype(np.float32), ADD, r1, r2)
    check("beta", L.x0, SIG, None, h["beta"])


def test_q4_0_fused_layer_chain(G, q4_layer):
    """Multi-matrix, gated dual and plain calls in one chain."""
    L = q4_layer
    calls = L.calls_fused(G)
    L.reset()
    G.launch_prepared(calls)
    want = L.snapshot(("q", "k", "v", "gate", "beta"))
    chain = G.prepare_chain(calls)
    info = G.chain_info(chain)
    assert (info["stages"], info["barriers"], info["barrier_mask"], info["reuse_mask"]) == (4, 2, 0b1100, 0)
    L.reset()
    chain.launch()
    _equal(want, L.snapshot(("q", "k", "v", "gate", "beta")), "fused chain")


def test_repeated_chain_launches(G, q4_layer):
    """The barrier counter carries over between launches: three launches serially, three
    PDL-chained back to back, and three graph replays all match three serial rounds of
    the separate calls (r accumulates in place)."""
    L = q4_layer
    calls = L.calls(G)
    L.reset()
    for _ in range(3):
        G.launch_prepared(calls)
    want = L.snapshot()
    chain = G.prepare_chain(calls)
    L.reset()
    for _ in range(3):
        chain.launch()
        torch.cuda.synchronize()
    _equal(want, L.snapshot(), "serial launches")
    L.reset()
    G.launch_prepared([chain, chain, chain])
    _equal(want, L.snapshot(), "back-to-back launches")
    graph = G.Graph([chain])
    L.reset()
    for _ in range(3):
        graph.launch()
    _equal(want, L.snapshot(), "graph replays")
    graph.close()
    assert G.device_status() == 0


@pytest.mark.parametrize("wt,d,f,nb", [
    (synth.F16, 1024, 2816, 8),
    (synth.Q8_0, 2048, 5632, 32),
    (synth.Q4_K, 1024, 2816, 16),
    (synth.F32, 512, 1536, 5),
    (synth.Q4_0, 1024, 2816, 3),
])
def test_layer_chain_every_format(G, wt, d, f, nb):
    L = Layer(wt, d, f, nb, seed=400 + wt)
    calls = L.calls(G)
    L.reset()
    G.launch_prepared(calls)
    want = L.snapshot()
    chain = G.prepare_chain(calls)
    info = G.chain_info(chain)
    assert (info["stages"], info["barrier_mask"]) == (8, 0b01110000)
    L.reset()
    chain.launch()
    _equal(want, L.snapshot(), "chain of format %d" % wt)
    M, K = L.shapes["q"]
    got = L.out["q"].cpu().numpy()
    want_q = ogemv.gemv(L.raw["q"], wt, L.x0, M, K, NONE, None)
    assert_within(got, want_q[0], gemv_bound(L.raw["q"], wt, L.x0, M, K)[0], "q of format %d" % wt)


def test_reuse_across_a_short_stage(G, q4_layer):
    """q, then a 32-row head and k on the same x: the head reuses q's staged x (its CTAs
    all had q rows); k does not (most CTAs had no head rows) and copies x again."""
    L = q4_layer
    d = L.d
    s = {n: torch.empty(L.shapes[n][0], device="cuda") for n in ("q", "beta", "k")}
    calls = [G.prepare(L.W["q"], L.wt, L.x, d, d, NONE, None, s["q"], pdl=True),
             G.prepare(L.W["beta"], L.wt, L.x, L.nb, d, SIG, None, s["beta"], pdl=True, split_k=False),
             G.prepare(L.W["k"], L.wt, L.x, d, d, NONE, None, s["k"], pdl=True)]
    G.launch_prepared(calls)
    torch.cuda.synchronize()
    want = {n: t.cpu().numpy().view(np.uint32).copy() for n, t in s.items()}
    chain = G.prepare_chain(calls)
    info = G.chain_info(chain)
    assert (info["barriers"], info["reuse_mask"]) == (0, 0b010)
    for t in s.values():
        t.fill_(float("nan"))
    chain.launch()
    torch.cuda.synchronize()
    _equal(want, {n: t.cpu().numpy().view(np.uint32).copy() for n, t in s.items()}, "reuse")


def test_chain_refusals(G, q4_layer):
    L = q4_layer
    d = L.d
    y = torch.empty(2 * d, device="cuda")
    one = G.prepare(L.W["q"], L.wt, L.x, d, d, NONE, None, y[:d])
    x2 = torch.zeros(2 * d, device="cuda")
    two_cols = G.prepare(L.W["k"], L.wt, x2, d, d, NONE, None, y, ncols=2)
    assert G.prepare_chain([one, two_cols], check=False) == G.ERR_UNSUPPORTED
    Wf = dev_tensor(synth.weights(synth.F16, 256, d, seed=9))
    f16 = G.prepare(Wf, synth.F16, L.x, 256, d, NONE, None, y[d:d + 256])
    assert G.prepare_chain([one, f16], check=False) == G.ERR_UNSUPPORTED  # two formats
    signs = dev_tensor(synth.rademacher(1024, seed=3))
    ws = torch.empty(d, device="cuda")
    fw = G.prepare(L.W["k"], L.wt, L.x, d, d, NONE, None, y[d:], fwht_signs=signs, fwht_block=1024, fwht_workspace=ws)
    assert G.prepare_chain([one, fw], check=False) == G.ERR_UNSUPPORTED  # a stand-alone transform first
    ch = G.prepare_chain([one])
    assert G.prepare_chain([ch, one], check=False) == G.ERR_UNSUPPORTED  # no chain in a chain
    # a stage whose output lands in another stage's weights
    Wk = L.W["k"].clone()
    into_w = Wk.view(torch.float32)[:d]
    bad = G.prepare(L.W["q"], L.wt, L.x, d, d, NONE, None, into_w)
    k = G.prepare(Wk, L.wt, L.x, d, d, NONE, None, y[d:])
    assert G.prepare_chain([bad, k], check=False) == G.ERR_ALIAS
    # calls without rows are skipped; a chain of only those launches nothing
    empty = G.prepare(L.W["q"], L.wt, L.x, 0, d, NONE, None, y)
    assert G.chain_info(G.prepare_chain([empty, one]))["stages"] == 1
    nothing = G.prepare_chain([empty])
    assert G.chain_info(nothing)["stages"] == 0
    nothing.launch()
    torch.cuda.synchronize()
    assert G.device_status() == 0


def test_chain_hazards_and_prologues(G):
    """Barriers for every kind of hazard between stages, and stages with the RMS prologue:
    stage 1 writes what stage 0 reads (write after read), stage 2 writes what stage 1
    writes (write after write), stage 3 reads nothing earlier stages write but shares their
    x with the RMS prologue, stage 4 reads stage 3's output as its aux."""
    wt, K, M = synth.Q4_0, 2048, 1024
    raw = [synth.weights(wt, M, K, seed=900 + i) for i in range(5)]
    W = [dev_tensor(r) for r in raw]
    xa = dev_tensor(synth.normal(K, seed=910))
    b = dev_tensor(synth.normal(K, seed=911))  # stage 0's x; its first M elements are stage 1's and 2's output
    gamma = dev_tensor(synth.normal(K, seed=912))
    y0, y3, y4 = (torch.empty(M, device="cuda") for _ in range(3))
    y1 = b[:M]
    def calls():
        return [G.prepare(W[0], wt, b, M, K, NONE, None, y0, pdl=True),                 # reads b
                G.prepare(W[1], wt, xa, M, K, NONE, None, y1, pdl=True),                # writes b: WAR
                G.prepare(W[2], wt, xa, M, K, SIG, None, y1, pdl=True),                 # writes b again: WAW
                G.prepare(W[3], wt, xa, M, K, NONE, None, y3, pdl=True, rms_norm_weight=gamma, rms_norm_eps=1e-5),
                G.prepare(W[4], wt, xa, M, K, ADD, y3, y4, pdl=True)]                   # reads y3: RAW
    b0 = b.clone()

    def run(fn):
        b.copy_(b0)
        for t in (y0, y3, y4):
            t.fill_(float("nan"))
        fn()
        torch.cuda.synchronize()
        return {n: t.cpu().numpy().view(np.uint32).copy() for n, t in (("y0", y0), ("b", b), ("y3", y3), ("y4", y4))}

    cs = calls()
    want = run(lambda: G.launch_prepared(cs))
    chain = G.prepare_chain(cs)
    info = G.chain_info(chain)
    # barriers before stages 1 (WAR on b), 2 (WAW on b) and 4 (RAW on y3), none before 3;
    # stage 2 reuses stage 1's staged x
    assert (info["barrier_mask"], info["reuse_mask"]) == (0b10110, 0b00100), info
    got = run(lambda: chain.launch())
    _equal(want, got, "hazards")
    # stage 0 against the oracle on the original b
    want0 = ogemv.gemv(raw[0], wt, b0.cpu().numpy(), M, K, NONE, None)
    assert_within(got["y0"].view(np.float32), want0[0], gemv_bound(raw[0], wt, b0.cpu().numpy(), M, K)[0], "y0")
