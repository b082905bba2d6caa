"""GPU parity of the fused decode prologues and the residual epilogue against the fp64 oracle
(oracle/fused.py), element by element. The bound is the layer's 2e-3 * sum_k |x_k w_k|
widened by one fp16 rounding step per activation: the kernel evaluates silu / RMSNorm in
fp32 and rounds once to fp16, and may round across a boundary the fp64 value does not."""
import numpy as np
import pytest

import oracle
from oracle import fused
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TYPES = (12, 13, 14, 23)
SHAPES = [(37, 1024, 1), (300, 2560, 3), (129, 768, 8), (64, 4096, 2), (16, 256, 1),
          (4100, 8192, 1)]   # the last: one token on the single-token K-quant kernel


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


def silu_inputs(M, K, seed):
    rng = np.random.default_rng(seed)
    gate = (3 * rng.standard_normal((M, K))).astype(np.float16)
    up = rng.standard_normal((M, K)).astype(np.float32)
    return gate, up


def rms_inputs(M, K, seed):
    rng = np.random.default_rng(seed)
    h = (5 * rng.standard_normal((M, K))).astype(np.float32)
    w = rng.standard_normal(K).astype(np.float32)
    return h, w


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", SHAPES)
def test_silu_mul_prologue(ql, t, N, K, M):
    W = synth.weights(t, N, K, [700, t, N, K])
    gate, up = silu_inputs(M, K, [701, t, M, K])
    y = ql.qlinear_silu_mul(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(gate).cuda(),
                            torch.from_numpy(up).cuda())
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    x = fused.silu_mul_x(gate, up)
    check(y.cpu().numpy().astype(np.float64), fused.qlinear_fused(t, W, N, K, x),
          fused.tolerance_fused(t, W, N, K, x), f"silu t={t} N={N} K={K} M={M}")


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", SHAPES)
def test_rmsnorm_prologue_and_normalised_output(ql, t, N, K, M):
    W = synth.weights(t, N, K, [710, t, N, K])
    h, w = rms_inputs(M, K, [711, t, M, K])
    eps = 1e-6
    Wd = torch.from_numpy(W).cuda()
    xn = torch.empty((M, K), dtype=torch.float16, device="cuda")
    y = ql.qlinear_rmsnorm(Wd, t, N, K, torch.from_numpy(h).cuda(), torch.from_numpy(w).cuda(), eps, xnorm=xn)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    x = fused.rmsnorm_x(h, w, eps)
    check(y.cpu().numpy().astype(np.float64), fused.qlinear_fused(t, W, N, K, x),
          fused.tolerance_fused(t, W, N, K, x), f"rmsnorm t={t} N={N} K={K} M={M}")
    # the normalised activations: within one fp16 step of the once-rounded fp64 value
    g = xn.cpu().numpy()
    assert np.all(np.abs(g.astype(np.float64) - x.astype(np.float64)) <= np.spacing(np.abs(x)).astype(np.float64))
    # and the fused launch equals the separate layer applied to them, bit for bit
    y2 = ql.qlinear(Wd, t, N, K, xn)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("in_place", [False, True])
def test_residual_epilogue(ql, t, in_place):
    N, K, M = 200, 1024, 4
    W = synth.weights(t, N, K, [720, t])
    gate, up = silu_inputs(M, K, [721, t])
    r = np.random.default_rng([722, t]).standard_normal((M, N)).astype(np.float32) * 50
    rd = torch.from_numpy(r).cuda()
    y = ql.qlinear_silu_mul(torch.from_numpy(W).cuda(), t, N, K, torch.from_numpy(gate).cuda(),
                            torch.from_numpy(up).cuda(), residual=rd, out=rd if in_place else None)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    x = fused.silu_mul_x(gate, up)
    check(y.cpu().numpy().astype(np.float64), fused.qlinear_fused(t, W, N, K, x, r),
          fused.tolerance_fused(t, W, N, K, x, r), f"residual t={t} in_place={in_place}")


def test_rmsnorm_of_zero_rows_is_zero(ql):
    t, N, K, M = 12, 48, 512, 2
    W = torch.from_numpy(synth.weights(t, N, K, [730])).cuda()
    h = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    w = torch.ones(K, dtype=torch.float32, device="cuda")
    y = ql.qlinear_rmsnorm(W, t, N, K, h, w, 1e-6)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0


# full-size decode layers, sampled rows: the 8B down projection fed by the SiLU gate, and the
# 8B gate projection fed by RMSNorm; a Q6_K layer whose rows take per-row copies
FULL = [("silu", 12, 12288, 4096, 1), ("rms", 12, 4096, 12288, 1), ("rms", 14, 5120, 17408, 1),
        ("silu", 23, 17408, 5120, 1)]


@pytest.mark.parametrize("kind,t,K,N,M", FULL)
def test_fused_full_size_sampled_rows(ql, kind, t, K, N, M):
    W = synth.weights(t, N, K, [740, t, K, N])
    Wd = torch.from_numpy(W).cuda()
    if kind == "silu":
        gate, up = silu_inputs(M, K, [741, t])
        y = ql.qlinear_silu_mul(Wd, t, N, K, torch.from_numpy(gate).cuda(), torch.from_numpy(up).cuda())
        x = fused.silu_mul_x(gate, up)
    else:
        h, w = rms_inputs(M, K, [742, t])
        y = ql.qlinear_rmsnorm(Wd, t, N, K, torch.from_numpy(h).cuda(), torch.from_numpy(w).cuda(), 1e-5)
        x = fused.rmsnorm_x(h, w, 1e-5)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    rng = np.random.default_rng(743)
    rows = np.unique(np.concatenate([[0, N - 1, N // 2], rng.choice(N, 50, replace=False)]))
    ref = oracle.qlinear_rows(t, W, N, K, x, rows)
    tol = oracle.tolerance_rows(t, W, N, K, x, rows)
    aw = np.abs(oracle.dequant(t, np.concatenate([W.reshape(N, -1)[r] for r in rows]), len(rows), K))
    tol = tol + 2.0 ** -10 * (np.abs(x.astype(np.float64)) @ aw.T) + 2.0 ** -24 * aw.sum(1)[None, :]
    check(y.cpu().numpy().astype(np.float64)[:, rows], ref, tol, f"full {kind} t={t} K={K} N={N}")
