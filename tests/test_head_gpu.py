"""GPU parity of the embedding gather and the greedy output head against the fp64 oracle
(oracle/head.py).

Embedding: exact, the exact weight rounded once to fp32 or fp16 (compared as numbers: +0 == -0).
Greedy head: several answers can be right when two logits lie within the layer's tolerance, so
the chosen row is checked for validity against the oracle (its oracle value is within the two
rows' tolerances of the oracle maximum, and the returned value within its own tolerance), and
for exact agreement with the first maximum of qlinear()'s own output, bit for bit."""
import numpy as np
import pytest

import oracle
from oracle import head
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TYPES = (12, 13, 14, 23)


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_weight_only_gb300 import build
    build.build()
    import gguf_weight_only_gb300 as q
    q.lib()
    return q


# ------------------------------------------------------------------ embedding gather

@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K", [(16, 256), (300, 512), (37, 5120), (1000, 4096)])
@pytest.mark.parametrize("fp16", [False, True])
def test_embed_exact(ql, t, N, K, fp16):
    W = synth.weights(t, N, K, [900, t, N, K])
    ids = np.random.default_rng([901, t, N]).integers(0, N, size=11).astype(np.int32)
    ids[:3] = [0, N - 1, ids[3]]   # both ends and a repeat
    out = ql.qlinear_embed(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(ids).cuda(), fp16=fp16)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    ref = head.embed_rows(t, W, N, K, ids).astype(np.float16 if fp16 else np.float32)
    got = out.cpu().numpy()
    assert got.dtype == ref.dtype
    # equal as numbers (a zero weight may come out as -0 from the oracle's order of products)
    assert np.array_equal(got, ref)


def test_embed_bad_id_gives_zero_row_and_status(ql):
    t, N, K = 12, 64, 512
    W = synth.weights(t, N, K, [910])
    ids = np.array([3, N, 7, -1], np.int32)
    out = ql.qlinear_embed(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == -9    # QL_ERR_INDEX, once
    assert ql.device_status() == 0
    got = out.cpu().numpy()
    assert np.all(got[1] == 0) and np.all(got[3] == 0)
    ref = head.embed_rows(t, W, N, K, [3, 7]).astype(np.float32)
    assert np.array_equal(got[[0, 2]], ref)


# ------------------------------------------------------------------ greedy head

def check_choice(ql, t, W, N, K, x, idx, val):
    """idx/val against qlinear()'s own y (exact) and the oracle (validity within tolerance)."""
    Wd = torch.from_numpy(W).cuda()
    y = ql.qlinear(Wd, t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    first = np.argmax(y, axis=1)
    assert np.array_equal(idx, first), (idx, first)
    assert np.array_equal(val.view(np.uint32), y[np.arange(len(idx)), idx].view(np.uint32))
    ref = oracle.qlinear(t, W, N, K, x)
    tol = oracle.tolerance(t, W, N, K, x)
    m = np.arange(len(idx))
    best = np.argmax(ref, axis=1)
    assert np.all(ref[m, idx] >= ref[m, best] - tol[m, idx] - tol[m, best])
    assert np.all(np.abs(val.astype(np.float64) - ref[m, idx]) <= tol[m, idx])


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", [(37, 1024, 1), (1000, 2560, 3), (300, 768, 8), (16, 256, 1), (4099, 512, 2),
                                   (4100, 8192, 1)])   # the last: the single-token K-quant kernel
def test_argmax_matches_materialised_logits(ql, t, N, K, M):
    W = synth.weights(t, N, K, [920, t, N, K])
    x = synth.activations(M, K, [921, t, M])
    idx, val = ql.qlinear_argmax(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    check_choice(ql, t, W, N, K, x, idx.cpu().numpy(), val.cpu().numpy())


@pytest.mark.parametrize("t", TYPES)
def test_argmax_ties_pick_the_first_row(ql, t):
    N, K = 200, 1024
    W = synth.weights(t, N, K, [930, t]).reshape(N, -1).copy()
    x = synth.activations(1, K, [931, t])
    y = oracle.qlinear(t, W.reshape(-1), N, K, x)[0]
    top = int(np.argmax(y))
    for r in (150, 180, 199):          # copies of the best row after it ...
        W[r] = W[top]
    if top > 10:
        W[3] = W[top]                  # ... and one before it, which must win
    W = W.reshape(-1)
    idx, val = ql.qlinear_argmax(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert int(idx[0]) == (3 if top > 10 else top)


# full-size greedy heads, all rows checked: a Q6_K 32K-vocabulary head at the 8B width, and
# its Q4_K counterpart with four tokens
@pytest.mark.parametrize("t,K,N,M", [(14, 4096, 32000, 1), (12, 4096, 32000, 4)])
def test_argmax_full_head(ql, t, K, N, M):
    W = synth.weights(t, N, K, [940, t, N])
    x = synth.activations(M, K, [941, t, M])
    idx, val = ql.qlinear_argmax(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    check_choice(ql, t, W, N, K, x, idx.cpu().numpy(), val.cpu().numpy())
