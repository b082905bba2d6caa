"""GPU checks of non-finite inputs against the readings of the pages: a NaN propagates per
IEEE (a NaN in token m's activations makes every y[m, :] NaN and leaves the other tokens
exact), and the greedy head ranks a NaN logit above every number (numpy's argmax)."""
import numpy as np
import pytest

import oracle
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TYPES = (12, 13, 14, 23)
D_OFFSET = {12: 0, 13: 0, 14: 208, 23: 0}   # byte offset of the fp16 superblock scale d


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_weight_only_gb300 import build
    build.build()
    import gguf_weight_only_gb300 as q
    q.lib()
    return q


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", [(40, 512, 2), (300, 1024, 40), (8000, 4096, 1)])
def test_nan_in_x_poisons_only_its_token(ql, t, N, K, M):
    W = synth.weights(t, N, K, [950, t, N])
    x = synth.activations(M, K, [951, t, M])
    x[0, 5] = np.nan
    y = ql.qlinear(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    y = y.cpu().numpy().astype(np.float64)
    assert np.isnan(y[0]).all()
    if M > 1:
        ref = oracle.qlinear(t, W, N, K, x[1:])
        tol = oracle.tolerance(t, W, N, K, x[1:])
        assert np.all(np.abs(y[1:] - ref) <= tol)


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K", [(37, 1024), (4100, 8192)])
def test_argmax_takes_a_nan_row(ql, t, N, K):
    bb = ql.block_bytes(t)
    W = synth.weights(t, N, K, [960, t, N]).reshape(N, K // 256, bb).copy()
    W[N // 3, :, D_OFFSET[t]:D_OFFSET[t] + 2] = np.array([np.nan], np.float16).view(np.uint8)
    W = W.reshape(-1)
    x = synth.activations(1, K, [961, t])
    Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
    y = ql.qlinear(Wd, t, N, K, xd)
    idx, val = ql.qlinear_argmax(Wd, t, N, K, xd)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    y = y.cpu().numpy()
    assert np.isnan(y[0, N // 3]) and np.isfinite(np.delete(y[0], N // 3)).all()
    assert int(idx[0]) == N // 3 and np.isnan(float(val[0]))
