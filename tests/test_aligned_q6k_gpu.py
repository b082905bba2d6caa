"""GPU tests of the aligned Q6_K layout (QL_Q6_K_A16, 224-byte blocks made by qlinear_repack):
the repacked bytes are the source blocks each followed by 14 zero bytes, and every entry point
given the repacked weights matches the fp64 oracle on the original Q6_K weights."""
import numpy as np
import pytest

import oracle
from oracle import fused, head
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

A16 = 270


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


def repacked(ql, W, N, K):
    Wp = ql.repack(torch.from_numpy(W).cuda(), 14, N, K)
    torch.cuda.synchronize()
    return Wp


@pytest.mark.parametrize("N,K", [(7, 256), (37, 1280), (300, 5120)])
def test_repack_layout(ql, N, K):
    W = synth.weights(14, N, K, [960, N, K])
    got = repacked(ql, W, N, K).cpu().numpy().reshape(-1, 224)
    blocks = W.reshape(-1, 210)
    assert np.array_equal(got[:, :210], blocks)
    assert not got[:, 210:].any()


@pytest.mark.parametrize("N,K,M", [(1, 256, 1), (37, 1280, 3), (300, 5120, 1), (129, 768, 8), (64, 4096, 9),
                                   (300, 2560, 64), (200, 1024, 257)])
def test_aligned_layout_matches_oracle(ql, N, K, M):
    W = synth.weights(14, N, K, [961, N, K])
    x = synth.activations(M, K, [962, M, K])
    y = ql.qlinear(repacked(ql, W, N, K), A16, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    check(y.cpu().numpy().astype(np.float64), oracle.qlinear(14, W, N, K, x), oracle.tolerance(14, W, N, K, x),
          f"aligned Q6_K N={N} K={K} M={M}")


def test_aligned_layout_other_entry_points(ql):
    N, K = 300, 2560
    W = synth.weights(14, N, K, [963])
    Wp = repacked(ql, W, N, K)
    # several projections
    W2 = synth.weights(14, 77, K, [964])
    x = synth.activations(2, K, [965])
    ys = ql.qlinear_multi([Wp, repacked(ql, W2, 77, K)], A16, [N, 77], K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    for Wj, Nj, yj in ((W, N, ys[0]), (W2, 77, ys[1])):
        check(yj.cpu().numpy().astype(np.float64), oracle.qlinear(14, Wj, Nj, K, x),
              oracle.tolerance(14, Wj, Nj, K, x), "aligned multi")
    # fused SiLU-gated prologue
    rng = np.random.default_rng(966)
    gate = (3 * rng.standard_normal((1, K))).astype(np.float16)
    up = rng.standard_normal((1, K)).astype(np.float32)
    y = ql.qlinear_silu_mul(Wp, A16, N, K, torch.from_numpy(gate).cuda(), torch.from_numpy(up).cuda())
    torch.cuda.synchronize()
    xs = fused.silu_mul_x(gate, up)
    check(y.cpu().numpy().astype(np.float64), oracle.qlinear(14, W, N, K, xs), fused.tolerance_fused(14, W, N, K, xs),
          "aligned silu")
    # greedy head: the same choice as the original layout's call
    x1 = synth.activations(1, K, [967])
    i1, v1 = ql.qlinear_argmax(Wp, A16, N, K, torch.from_numpy(x1).cuda())
    y1 = ql.qlinear(Wp, A16, N, K, torch.from_numpy(x1).cuda())
    torch.cuda.synchronize()
    assert int(i1[0]) == int(torch.argmax(y1[0]))
    # embedding gather: exact
    ids = np.array([0, 5, N - 1], np.int32)
    e = ql.qlinear_embed(Wp, A16, N, K, torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(e.cpu().numpy(), head.embed_rows(14, W, N, K, ids).astype(np.float32))
    assert ql.device_status() == 0


@pytest.mark.parametrize("M", [1, 256])
def test_aligned_layout_full_size_sampled_rows(ql, M):
    N, K = 17408, 5120
    W = synth.weights(14, N, K, [968, M])
    x = synth.activations(M, K, [969, M])
    y = ql.qlinear(repacked(ql, W, N, K), A16, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(970).choice(N, 50, replace=False)]))
    check(y.cpu().numpy().astype(np.float64)[:, rows], oracle.qlinear_rows(14, W, N, K, x, rows),
          oracle.tolerance_rows(14, W, N, K, x, rows), f"aligned full M={M}")
