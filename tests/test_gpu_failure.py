"""Failure handling on the GPU without a fault: a bounded wait that runs out.

The self-test kernel waits, through the same bounded-wait routine every GEMV kernel
uses, on a barrier phase that nothing completes.  The wait must give up after its limit,
set the abort flag (a second wait returns at once) and the device error word, which
gf_device_status reports as GF_ERR_TIMEOUT; the context stays usable and a GEMV after
the reset is correct."""

import numpy as np
import pytest

from decode_gemv_epilogue_gb300 import synth
from gpu_util import assert_within, dev_tensor, gemv_bound
from oracle import gemv as ogemv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_bounded_wait_gives_up_and_reports(lib):
    G = lib
    assert G.device_status(reset=True) == G.OK
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    G.selftest_wait_timeout(20000, out)  # 20 ms
    torch.cuda.synchronize()
    first, second, us1, us2 = out.cpu().tolist()
    assert first == 0 and second == 0
    assert 20000 <= us1 < 1000000          # gave up after its limit, not much later
    assert us2 < 1000                      # the abort flag stops the next wait at once
    assert G.device_status() == G.ERR_TIMEOUT
    assert G.device_status(reset=True) == G.ERR_TIMEOUT
    assert G.device_status() == G.OK
    # the context is still usable
    M, K = 256, 1024
    raw = synth.weights(synth.Q4_0, M, K, seed=900)
    x = synth.normal(K, seed=901)
    d = torch.full((M,), float("nan"), device="cuda")
    G.gemv_fused(dev_tensor(raw), synth.Q4_0, dev_tensor(x), M, K, ogemv.EPI_NONE, None, d)
    torch.cuda.synchronize()
    assert_within(d.cpu().numpy().astype(np.float64), ogemv.gemv(raw, synth.Q4_0, x, M, K)[0],
                  gemv_bound(raw, synth.Q4_0, x, M, K)[0], "gemv after the timeout")
    assert G.device_status() == G.OK
