"""Several matrices sharing x in one pass (gemv_multi): the same bits as the separate
calls, within the parity bound of the fp64 oracle, for shapes that cut a tile at a
matrix boundary, every format, batches, both prologues and the per-matrix fallback."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, gemv_bound, norm_bound
from oracle import gemv as ogemv
from oracle import norm as onorm

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module")
def G(lib):
    assert lib.device_status(reset=True) == 0
    yield lib
    assert lib.device_status() == 0, "a kernel reported a bounded-wait timeout"


def _bits(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32).copy()


def _setup(wt, K, specs, ncols, seed):
    """specs: [(M, epilogue)] -> raw weights, device tensors, aux values per item."""
    out = []
    for i, (M, epi) in enumerate(specs):
        raw = synth.weights(wt, M, K, seed=seed + 3 * i)
        aux = synth.normal(ncols * M, seed=seed + 3 * i + 1).astype(np.float32) if epi in (3, 4) else None
        out.append((raw, M, epi, aux))
    return out


def _run(G, wt, K, items, x, ncols, multi, **kw):
    dsts, call = [], []
    for raw, M, epi, aux in items:
        Wd = dev_tensor(raw)
        a = dev_tensor(aux) if aux is not None else None
        d = a if epi == 4 else torch.full((ncols * M,), float("nan"), device="cuda")
        dsts.append(d)
        call.append((Wd, M, epi, a, d))
    if multi:
        G.gemv_multi(call, wt, x, K, ncols=ncols, pdl=True, **kw)
    else:
        for (Wd, M, epi, a, d) in call:
            G.gemv_fused_ex(Wd, wt, x, M, K, epi, a, d, ncols=ncols, pdl=True, tensor_cores=False, **kw)
    return [_bits(d) for d in dsts]


CASES = [
    # (wtype, K, [(M, epilogue)], ncols)
    (synth.Q4_0, 4096, [(4096, 0), (1024, 0), (1024, 0), (32, 1)], 1),   # q, k, v and a sigmoid head
    (synth.Q4_0, 2048, [(37, 4), (5, 3), (203, 2)], 1),                    # tiles cut at every boundary
    (synth.Q8_0, 4096, [(3000, 3), (300, 0)], 1),
    (synth.Q4_K, 4096, [(700, 0), (900, 4)], 1),
    (synth.F16, 4096, [(1000, 4), (1000, 1)], 1),
    (synth.F32, 1024, [(300, 2), (77, 0)], 1),
    (synth.Q4_0, 4096, [(1024, 4), (512, 0), (64, 3)], 3),                 # a batch of three columns
    (synth.F16, 4096, [(512, 0), (512, 4)], 12),                           # two column blocks
    (synth.F32, 1000, [(64, 0), (64, 4)], 1),                              # K % 16: one launch per matrix
]


@pytest.mark.parametrize("case", CASES, ids=["case%d" % i for i in range(len(CASES))])
def test_multi_equals_separate_and_oracle(G, case):
    wt, K, specs, ncols = case
    items = _setup(wt, K, specs, ncols, seed=700)
    X = synth.normal(ncols * K, seed=799).astype(np.float32).reshape(ncols, K)
    x = dev_tensor(X.reshape(-1))
    sep = _run(G, wt, K, items, x, ncols, multi=False)
    got = _run(G, wt, K, items, x, ncols, multi=True)
    for (raw, M, epi, aux), a, b in zip(items, sep, got):
        assert np.array_equal(a, b), "multi differs from the separate call (M=%d epi=%d)" % (M, epi)
        want = ogemv.gemv(raw, wt, X, M, K, epi, aux.reshape(ncols, M) if aux is not None else None)
        assert_within(b.view(np.float32).astype(np.float64).reshape(ncols, M), want,
                      gemv_bound(raw, wt, X, M, K), "multi M=%d epi=%d" % (M, epi))


def test_multi_with_rms_norm_prologue(G):
    wt, K, eps = synth.Q4_0, 4096, 1e-5
    items = _setup(wt, K, [(512, 0), (256, 4)], 1, seed=810)
    X = synth.normal(K, seed=811).astype(np.float32).reshape(1, K)
    gamma = (1.0 + 0.1 * synth.normal(K, seed=812)).astype(np.float32)
    x, gd = dev_tensor(X.reshape(-1)), dev_tensor(gamma)
    sep = _run(G, wt, K, items, x, 1, multi=False, rms_norm_weight=gd, rms_norm_eps=eps)
    got = _run(G, wt, K, items, x, 1, multi=True, rms_norm_weight=gd, rms_norm_eps=eps)
    Xn = onorm.rms_norm(X, gamma, eps, K)
    for (raw, M, epi, aux), a, b in zip(items, sep, got):
        assert np.array_equal(a, b)
        want = ogemv.gemv(raw, wt, Xn, M, K, epi, aux.reshape(1, M) if aux is not None else None)
        assert_within(b.view(np.float32).astype(np.float64).reshape(1, M), want, norm_bound(raw, wt, Xn, M, K),
                      "multi rms")


def test_multi_prepared_and_fwht_workspace(G):
    wt, K, B = synth.F16, 5120, 1024
    items = _setup(wt, K, [(640, 0), (128, 4)], 1, seed=820)
    X = synth.normal(K, seed=821).astype(np.float32)
    x = dev_tensor(X)
    s = dev_tensor(synth.rademacher(B, seed=822))
    ws = torch.empty(K, device="cuda")
    sep = _run(G, wt, K, items, x, 1, multi=False, fwht_signs=s, fwht_block=B, fwht_workspace=ws)
    call, dsts = [], []
    for raw, M, epi, aux in items:
        a = dev_tensor(aux) if aux is not None else None
        d = a if epi == 4 else torch.empty(M, device="cuda")
        dsts.append(d)
        call.append((dev_tensor(raw), M, epi, a, d))
    p = G.prepare_multi(call, wt, x, K, fwht_signs=s, fwht_block=B, fwht_workspace=ws, pdl=True)
    p.launch()
    for a, d in zip(sep, dsts):
        assert np.array_equal(a, _bits(d))
    p.close()
