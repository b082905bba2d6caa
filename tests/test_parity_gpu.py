"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle, element by
element, with the stated tolerance |y - y_oracle| <= 2e-3 * sum_k |x_k * w_k|."""
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


def run(ql, path, t, W, N, K, x):
    Wd = torch.from_numpy(W).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = ql.qlinear(Wd, t, N, K, xd, path=path)
    torch.cuda.synchronize()
    assert ql.device_status() == 0
    return y.cpu().numpy().astype(np.float64)


def check(y, ref, tol, what):
    assert y.shape == ref.shape, what
    assert np.all(np.isfinite(y)), what
    err = np.abs(y - ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {tuple(i)} "
                             f"y={y[tuple(i)]} ref={ref[tuple(i)]} tol={tol[tuple(i)]} max_ratio={np.max(err / np.maximum(tol, 1e-300))}")


# ------------------------------------------------------------------ small / ragged shapes, both kernels

GEMV_SHAPES = [(1, 256, 1), (7, 512, 3), (13, 1024, 8), (37, 768, 2), (129, 2560, 5), (300, 5120, 1), (64, 4096, 4),
               (45, 1280, 7)]


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", GEMV_SHAPES)
def test_gemv_matches_oracle(ql, t, N, K, M):
    W = synth.weights(t, N, K, [100, t, N, K])
    x = synth.activations(M, K, [101, t, M, K])
    ref = oracle.qlinear(t, W, N, K, x)
    check(run(ql, "gemv", t, W, N, K, x), ref, oracle.tolerance(t, W, N, K, x), f"gemv t={t} N={N} K={K} M={M}")


GEMM_SHAPES = [(128, 256, 32), (129, 512, 9), (300, 1024, 33), (1, 256, 1), (256, 2048, 100), (200, 768, 256),
               (130, 1280, 300), (128, 512, 512),
               # one token tile over few row tiles: the superblocks of each row tile are split
               # between a head CTA and a tail CTA of a cluster (ragged rows and tokens), also
               # where the split plan replaces several token tiles (M = 64, 100, 128); 80 row
               # tiles take two heads per tail on 152 SMs
               (300, 5120, 9), (640, 4096, 32), (10240, 2048, 16), (1000, 4096, 128), (512, 2048, 64),
               (1, 4096, 3)]


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", GEMM_SHAPES)
def test_gemm_matches_oracle(ql, t, N, K, M):
    W = synth.weights(t, N, K, [200, t, N, K])
    x = synth.activations(M, K, [201, t, M, K])
    ref = oracle.qlinear(t, W, N, K, x)
    check(run(ql, "gemm", t, W, N, K, x), ref, oracle.tolerance(t, W, N, K, x), f"gemm t={t} N={N} K={K} M={M}")


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("M", [1, 8, 9, 64])
def test_auto_dispatch_matches_oracle(ql, t, M):
    N, K = 160, 1024
    W = synth.weights(t, N, K, [300, t])
    x = synth.activations(M, K, [301, t, M])
    ref = oracle.qlinear(t, W, N, K, x)
    check(run(ql, "auto", t, W, N, K, x), ref, oracle.tolerance(t, W, N, K, x), f"auto t={t} M={M}")


@pytest.mark.parametrize("t", TYPES)
def test_gemv_many_tokens_in_groups(ql, t):
    """The forced decode kernel handles M > 8 as groups of 8 tokens."""
    N, K, M = 40, 512, 19
    W = synth.weights(t, N, K, [310, t])
    x = synth.activations(M, K, [311, t])
    ref = oracle.qlinear(t, W, N, K, x)
    check(run(ql, "gemv", t, W, N, K, x), ref, oracle.tolerance(t, W, N, K, x), f"gemv groups t={t}")


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("t", TYPES)
def test_zero_weights_and_zero_activations(ql, path, t):
    N, K, M = 33, 512, 3
    W = synth.weights(t, N, K, [400, t])
    x = np.zeros((M, K), np.float16)
    y = run(ql, path, t, W, N, K, x)
    assert np.all(y == 0.0)
    Wz = np.zeros_like(W)                     # d = dmin = 0: every weight 0
    x = synth.activations(M, K, [401, t])
    assert np.all(run(ql, path, t, Wz, N, K, x) == 0.0)


@pytest.mark.parametrize("t", TYPES)
def test_unit_activation_picks_a_column(ql, t):
    """x = e_k: the decode kernel returns column k of dequant(W). Its fp16 MMA operand is the
    integer sc*q (K-quants, |.| <= 1953: exact), sc*(q-32) (Q6_K) or (ls-32)*codebook[q]
    (IQ4_XS, |.| <= 4064: rounded to 11 significant bits when above 2048), scaled in fp32."""
    N, K = 70, 768
    W = synth.weights(t, N, K, [410, t])
    w = oracle.dequant(t, W, N, K)
    ks = [0, 1, 255, 256, 511, 767]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = run(ql, "gemv", t, W, N, K, x)
    ref = w[:, ks].T
    rtol = 2 ** -11 if t in (14, 23) else 2 ** -20   # one fp16 rounding of the integer operand
    np.testing.assert_allclose(y, ref, rtol=rtol, atol=2 ** -40)


@pytest.mark.parametrize("t", (12, 13))
def test_unit_activation_single_token(ql, t):
    """M = 1, x = e_k, on the single-token K-quant path: the MMA's D column of sub-block j is
    q 2^-24 (q 2^-20 for high nibbles) exactly, the x sums are 1 or 0, and y = d sc q - dmin m
    is formed by a few fp32 products and sums: within 2^-20 of column k of dequant(W)."""
    N, K = 70, 768
    W = synth.weights(t, N, K, [411, t])
    w = oracle.dequant(t, W, N, K)
    for k in (0, 1, 31, 32, 63, 64, 255, 256, 511, 767):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1.0
        y = run(ql, "gemv", t, W, N, K, x)
        np.testing.assert_allclose(y[0], w[:, k], rtol=2 ** -20, atol=2 ** -40, err_msg=f"t={t} k={k}")


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("M", [40, 300])
def test_unit_activation_prefill(ql, t, M):
    """x = e_k through the tcgen05 prefill kernels (token m picks column k_m; M = 40 takes the
    split form, each row tile's superblocks shared by a CTA pair, M = 300 one CTA per tile): the
    dequantisers form each weight in fp32 and round it once to fp16 for tensor memory, so y is
    the weight to 11 significant bits (2^-24 absolute below fp16's normal range, where a weight
    that nearly cancels to zero lands on the subnormal grid)."""
    N, K = 200, 1024
    W = synth.weights(t, N, K, [412, t])
    w = oracle.dequant(t, W, N, K)
    ks = [(37 * m) % K for m in range(M)]
    x = np.zeros((len(ks), K), np.float16)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y = run(ql, "gemm", t, W, N, K, x)
    np.testing.assert_allclose(y, w[:, ks].T, rtol=2 ** -11, atol=2 ** -24)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("t", TYPES)
def test_deterministic(ql, path, t):
    # gemm: M=48 takes the split form (each row tile's sums from a CTA pair, added in a fixed
    # order), M=300 one CTA per row tile and token tile
    for M in ((6,) if path == "gemv" else (48, 300)):
        N, K = 257, 2048
        W = synth.weights(t, N, K, [420, t])
        x = synth.activations(M, K, [421, t])
        a = run(ql, path, t, W, N, K, x)
        b = run(ql, path, t, W, N, K, x)
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64)), M


@pytest.mark.parametrize("t", TYPES)
def test_unaligned_source_is_refused_and_a_copy_matches(ql, t):
    """The pages store W at a 68-byte offset (test_llm_quant_cpu.py); the ABI rejects an
    unaligned pointer and an aligned copy gives the oracle's result."""
    N, K, M = 64, 256, 1
    W = synth.weights(t, N, K, [430, t])
    x = synth.activations(M, K, [431, t])
    store = torch.from_numpy(np.concatenate([np.zeros(68, np.uint8), W])).cuda()
    view = store[68:]
    with pytest.raises(ql.QLinearError) as e:
        ql.qlinear(view, t, N, K, torch.from_numpy(x).cuda())
    assert e.value.status == -4
    y = ql.qlinear(view.clone(), t, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    check(y.cpu().numpy().astype(np.float64), oracle.qlinear(t, W, N, K, x), oracle.tolerance(t, W, N, K, x), "offset")


# ------------------------------------------------------------------ full-size workloads, sampled rows

FULL = [
    (12, 4096, 4096, 1), (12, 4096, 1024, 4), (12, 4096, 12288, 1), (12, 12288, 4096, 4),
    (23, 5120, 5120, 1), (23, 5120, 17408, 1), (23, 17408, 5120, 1),
    (12, 4096, 12288, 32), (12, 4096, 12288, 128), (12, 4096, 12288, 512),
    (13, 5120, 17408, 1), (13, 5120, 17408, 256), (14, 5120, 17408, 1), (14, 5120, 17408, 256),
    # the split prefill form at full size: CTA pairs (K=12288 N=4096, K=17408 N=5120) and two
    # heads per tail (N=10240, 80 row tiles)
    (12, 12288, 4096, 32), (12, 12288, 4096, 128), (23, 17408, 5120, 32), (14, 17408, 5120, 32), (13, 4096, 10240, 32),
]


@pytest.mark.parametrize("t,K,N,M", FULL)
def test_full_size_sampled_rows(ql, t, K, N, M):
    W = synth.weights(t, N, K, [500, t, K, N])
    x = synth.activations(M, K, [501, t, M])
    y = run(ql, "auto", t, W, N, K, x)
    rng = np.random.default_rng(502)
    rows = np.unique(np.concatenate([[0, 1, N - 1, N // 2], rng.choice(N, 60, replace=False)]))
    ref = oracle.qlinear_rows(t, W, N, K, x, rows)
    tol = oracle.tolerance_rows(t, W, N, K, x, rows)
    check(y[:, rows], ref, tol, f"full t={t} K={K} N={N} M={M}")


# ------------------------------------------------------------------ several reduction rounds (decode)

# Four tokens over N=20000 rows: on 152 SMs each CTA owns up to 9 row tiles, and its partial
# sums for 8 tiles at a time fill the 16 KB reduction area, so it reduces in two rounds.
@pytest.mark.parametrize("t", TYPES)
def test_gemv_two_reduction_rounds(ql, t):
    N, K, M = 20000, 4096, 4
    W = synth.weights(t, N, K, [545, t])
    x = synth.activations(M, K, [546, t])
    y = run(ql, "gemv", t, W, N, K, x)
    rng = np.random.default_rng(547)
    rows = np.unique(np.concatenate([[0, 127, 128, 143, 144, N - 1], rng.choice(N, 80, replace=False)]))
    check(y[:, rows], oracle.qlinear_rows(t, W, N, K, x, rows), oracle.tolerance_rows(t, W, N, K, x, rows),
          f"gemv two rounds t={t}")


# ------------------------------------------------------------------ x per stage (decode)

# Eight tokens at large K: each warp's slice of x for all tokens no longer fits in shared memory
# beside its ring, so on 152 SMs the plan sends x with every weight stage instead (the 8B and 27B
# down projections batched over 8 tokens, and four tokens at K=32768); every element checked.
@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K,M", [(300, 12288, 8), (300, 17408, 8), (37, 32768, 4)])
def test_gemv_x_per_stage_matches_oracle(ql, t, N, K, M):
    W = synth.weights(t, N, K, [540, t, N, K])
    x = synth.activations(M, K, [541, t, M, K])
    check(run(ql, "gemv", t, W, N, K, x), oracle.qlinear(t, W, N, K, x), oracle.tolerance(t, W, N, K, x),
          f"gemv x per stage t={t} N={N} K={K} M={M}")


# ------------------------------------------------------------------ single-token K-quant kernel

# Shapes where every warp has at least 8 superblocks, so one token takes the single-token
# kernel (sub-blocks on the MMA's n side); every output element checked, ragged N included.
# On 152 SMs the last four keep each warp's K slice (1 or 2 superblocks) in one stage and its
# B operand in registers: slices of 2 (K=4096), of 1 (K=256), and of 2 with a last slice of 1
# (K=1792: 2+2+2+1, K=768: 2+1).
@pytest.mark.parametrize("t", (12, 13, 23))
@pytest.mark.parametrize("N,K", [(4100, 8192), (2432, 16384), (8000, 4096), (20000, 256), (24000, 1792),
                                 (29184, 768), (9728, 5120)])
def test_single_token_kernel_matches_oracle(ql, t, N, K):
    W = synth.weights(t, N, K, [520, t, N, K])
    x = synth.activations(1, K, [521, t, K])
    y = run(ql, "auto", t, W, N, K, x)
    check(y, oracle.qlinear(t, W, N, K, x), oracle.tolerance(t, W, N, K, x), f"single token t={t} N={N} K={K}")
