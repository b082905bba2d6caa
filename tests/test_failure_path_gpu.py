"""The device-side failure path, exercised without a fault: a bounded wait that runs out
must set the status word, the host must read it as QL_ERR_TIMEOUT (once: reading clears
it), and the context must stay usable for the next call."""
import numpy as np
import pytest

import oracle
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_weight_only_gb300 import build
    build.build()
    import gguf_weight_only_gb300 as q
    q.lib()
    return q


def test_expired_wait_is_reported_once_and_the_context_survives(ql):
    assert ql.device_status() == 0
    ql.selftest_wait_timeout()
    assert ql.device_status() == -6          # QL_ERR_TIMEOUT
    assert ql.device_status() == 0           # reading cleared it

    # the next call runs normally and is correct
    t, N, K, M = 12, 48, 1024, 3
    W = synth.weights(t, N, K, [300, t])
    x = synth.activations(M, K, [301, t])
    y = ql.qlinear(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(x).cuda())
    assert ql.device_status() == 0
    ref = oracle.qlinear(t, W, N, K, x)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= oracle.tolerance(t, W, N, K, x))
