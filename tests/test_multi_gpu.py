"""GPU parity of qlinear_multi: several projections sharing x and K in one call, each output
against the fp64 oracle element by element (tolerance 2e-3 * sum_k |x_k * w_k|). The pages
check that a fused pair of linears equals the separate layers
(test/unit/test_llm_quant_cpu.py, test_q8_linear_pair_matches_separate); here both are held
to the oracle, and a single projection must reproduce qlinear() bit for bit."""
import numpy as np
import pytest

import oracle
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


def check(y, ref, tol, what):
    assert y.shape == ref.shape, what
    assert np.all(np.isfinite(y)), what
    bad = np.abs(y - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


def run_multi(ql, t, Ws, Ns, K, x):
    outs = ql.qlinear_multi([torch.from_numpy(W).cuda() for W in Ws], t, Ns, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    return [o.cpu().numpy().astype(np.float64) for o in outs]


# ragged projections: tails inside a tile, a single-tile projection, tiles of several
# projections inside one CTA's run
@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("Ns,K,M", [((37, 300, 16, 129), 1024, 1), ((7, 13), 512, 3), ((64, 1, 200), 2560, 8),
                                    ((300, 301), 768, 2), ((129, 37, 16), 1024, 9), ((40, 24), 512, 20),
                                    ((200, 77), 12288, 8)])   # the last: x sent with every weight stage
def test_multi_matches_oracle(ql, t, Ns, K, M):
    Ws = [synth.weights(t, N, K, [600, t, j, N]) for j, N in enumerate(Ns)]
    x = synth.activations(M, K, [601, t, M])
    ys = run_multi(ql, t, Ws, Ns, K, x)
    for j, (W, N, y) in enumerate(zip(Ws, Ns, ys)):
        check(y, oracle.qlinear(t, W, N, K, x), oracle.tolerance(t, W, N, K, x), f"t={t} proj {j} N={N}")


@pytest.mark.parametrize("t", TYPES)
def test_single_projection_is_qlinear(ql, t):
    N, K, M = 300, 1024, 4
    W = torch.from_numpy(synth.weights(t, N, K, [610, t])).cuda()
    x = torch.from_numpy(synth.activations(M, K, [611, t])).cuda()
    (y1,) = ql.qlinear_multi([W], t, [N], K, x)
    y2 = ql.qlinear(W, t, N, K, x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("t", TYPES)
def test_multi_deterministic(ql, t):
    Ns, K = (200, 77, 16), 1024
    Ws = [torch.from_numpy(synth.weights(t, N, K, [620, t, j])).cuda() for j, N in enumerate(Ns)]
    x = torch.from_numpy(synth.activations(2, K, [621, t])).cuda()
    a = ql.qlinear_multi(Ws, t, Ns, K, x)
    b = ql.qlinear_multi(Ws, t, Ns, K, x)
    torch.cuda.synchronize()
    assert all(torch.equal(u, v) for u, v in zip(a, b))


# full-size projection sets, sampled rows: the 8B layer's Q/K/V and gate/up, and a Q6_K pair
# whose rows are not 16-byte multiples (per-row copies)
FULL = [(12, 4096, (4096, 1024, 1024), 1), (12, 4096, (12288, 12288), 4),
        (23, 5120, (5120, 1024, 1024), 1), (14, 5120, (17408, 5120), 1)]


@pytest.mark.parametrize("t,K,Ns,M", FULL)
def test_multi_full_size_sampled_rows(ql, t, K, Ns, M):
    Ws = [synth.weights(t, N, K, [630, t, j, N]) for j, N in enumerate(Ns)]
    x = synth.activations(M, K, [631, t, M])
    ys = run_multi(ql, t, Ws, Ns, K, x)
    rng = np.random.default_rng(632)
    for j, (W, N, y) in enumerate(zip(Ws, Ns, ys)):
        rows = np.unique(np.concatenate([[0, N - 1, N // 2], rng.choice(N, 40, replace=False)]))
        ref = oracle.qlinear_rows(t, W, N, K, x, rows)
        tol = oracle.tolerance_rows(t, W, N, K, x, rows)
        check(y[:, rows], ref, tol, f"full t={t} K={K} proj {j} N={N} M={M}")
