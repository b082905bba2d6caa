"""Pins of the fused-prologue oracle (oracle/fused.py) against closed forms and invariants,
independent of its own formulas: hand-computed values of silu and RMSNorm, the fp16 rounding
of a known value, sign and scaling invariants, and row independence."""
import numpy as np

import oracle
from oracle import fused
from gguf_weight_only_gb300 import synth


def test_silu_closed_forms():
    # silu(g) = g / (1 + e^-g): e^-1 = 0.36787944117144233, e^-2 = 0.1353352832366127,
    # e^2 = 7.38905609893065
    got = fused.silu(np.array([0.0, 1.0, -1.0, 2.0, -2.0]))
    want = [0.0, 0.7310585786300049, -0.2689414213699951, 1.7615941559557649, -0.23840584404423515]
    assert np.allclose(got, want, rtol=1e-15, atol=0)
    # far tails: silu(g) -> g for g >> 0 and -> 0 (from below) for g << 0
    assert abs(fused.silu(np.array([30.0]))[0] - 30.0) < 1e-10
    t = fused.silu(np.array([-30.0]))[0]
    assert -1e-11 < t < 0


def test_silu_mul_rounds_once_to_fp16():
    # silu(1) * 1 = 0.73105857...; fp16 steps are 2^-11 on [0.5, 1): 1497.2 steps -> 1497 / 2048
    x = fused.silu_mul_x(np.array([1.0], np.float16), np.array([1.0], np.float32))
    assert x.dtype == np.float16 and float(x[0]) == 1497 / 2048
    # gate 0 gives 0 whatever up is; up 0 gives 0
    assert np.all(fused.silu_mul_x(np.zeros(4, np.float16), np.array([1, -5, 7, 1e3], np.float32)) == 0)
    assert np.all(fused.silu_mul_x(np.array([1, -2, 3, -4], np.float16), np.zeros(4, np.float32)) == 0)


def test_silu_mul_signs_and_power_of_two_scaling():
    rng = np.random.default_rng(70)
    g = rng.standard_normal(512).astype(np.float16)
    u = rng.standard_normal(512).astype(np.float32)
    x1 = fused.silu_mul_x(g, u).astype(np.float64)
    x2 = fused.silu_mul_x(g, 2 * u).astype(np.float64)
    nz = (x1 != 0) & (np.abs(x1) > 2 ** -13)
    assert np.all(np.sign(x1[nz]) == np.sign(g[nz].astype(np.float64) * u[nz]))
    assert np.array_equal(x2[nz], 2 * x1[nz])     # scaling by 2 commutes with rounding


def test_rmsnorm_closed_forms():
    h = np.array([[3.0, 4.0]], np.float32)        # mean(h^2) = 12.5
    assert np.allclose(fused.rmsnorm(h, np.ones(2, np.float32), 0.0), [[0.848528137423857, 1.131370849898476]],
                       rtol=1e-15, atol=0)
    assert np.allclose(fused.rmsnorm(h, np.array([2.0, -1.0], np.float32), 0.0),
                       [[1.697056274847714, -1.131370849898476]], rtol=1e-15, atol=0)
    # mean(1) = 1, eps = 3 -> 1 / sqrt(4)
    assert np.array_equal(fused.rmsnorm(np.ones((1, 4), np.float32), np.ones(4, np.float32), 3.0), np.full((1, 4), 0.5))
    # an all-zero row stays zero
    assert np.array_equal(fused.rmsnorm(np.zeros((1, 8), np.float32), np.ones(8, np.float32), 1e-6), np.zeros((1, 8)))


def test_rmsnorm_scale_invariance_and_row_independence():
    rng = np.random.default_rng(71)
    h = rng.standard_normal((1, 256)).astype(np.float32)
    w = rng.standard_normal(256).astype(np.float32)
    a = fused.rmsnorm(h, w, 0.0)
    b = fused.rmsnorm(4 * h, w, 0.0)
    assert np.allclose(a, b, rtol=1e-14, atol=0)
    both = fused.rmsnorm(np.concatenate([h, 8 * h]), w, 0.0)
    assert np.allclose(both[0], a[0], rtol=1e-14, atol=0) and np.allclose(both[1], a[0], rtol=1e-14, atol=0)
    # root mean square of the normalised row (w = 1, eps = 0) is one
    r = fused.rmsnorm(h, np.ones(256, np.float32), 0.0)
    assert abs(np.sqrt(np.mean(r * r)) - 1.0) < 1e-14


def test_residual_epilogue_on_zero_weights_is_the_residual():
    t, N, K, M = 12, 16, 256, 2
    W = np.zeros(N * (K // 256) * 144, np.uint8)  # d = dmin = 0: every weight is zero
    x = synth.activations(M, K, [72])
    r = np.random.default_rng(73).standard_normal((M, N)).astype(np.float32)
    assert np.array_equal(fused.qlinear_fused(t, W, N, K, x, r), r.astype(np.float64))


def test_fused_tolerance_widens_the_layer_bound():
    t, N, K, M = 12, 8, 512, 2
    W = synth.weights(t, N, K, [74])
    x = synth.activations(M, K, [75])
    base = oracle.tolerance(t, W, N, K, x)
    wide = fused.tolerance_fused(t, W, N, K, x)
    assert np.all(wide > base)
    # the extra term is 2^-10 sum|x w| + 2^-24 sum|w|: at most ~0.49 of the 2e-3 bound plus a tiny floor
    assert np.all(wide - base <= base * (2 ** -10 / 2e-3) + 2 ** -24 * np.abs(oracle.dequant(t, W, N, K)).sum(1)[None, :] + 1e-12)


def test_fused_tolerance_hand_computed():
    """Two Q4_K rows over K = 256: row 0 every weight 1 (d = 1, dmin = 0, sc = 1, m = 0, every
    nibble 1), row 1 every weight 0 (d = 0); x alternating +1, -1; residual (4, -8).
    Row 0: 2e-3 * 256 + 2^-10 * 256 + 2^-24 * 256 + 2^-23 * 4. Row 1: 2^-23 * 8 only."""
    def block(d):
        b = np.zeros(144, np.uint8)
        b[0:2] = np.array([d], np.float16).view(np.uint8)
        b[2:4] = np.array([0.0], np.float16).view(np.uint8)
        b[4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]   # sc = 1, m = 0 in all eight sub-blocks
        b[16:144] = 0x11                                  # both nibbles 1
        return b
    W = np.concatenate([block(1.0), block(0.0)])
    x = np.tile(np.array([1.0, -1.0], np.float16), 128).reshape(1, 256)
    r = np.array([[4.0, -8.0]], np.float32)
    got = fused.tolerance_fused(12, W, 2, 256, x, r)
    expect = [[2e-3 * 256 + 2.0 ** -10 * 256 + 2.0 ** -24 * 256 + 2.0 ** -23 * 4, 2.0 ** -23 * 8]]
    np.testing.assert_allclose(got, expect, rtol=1e-15, atol=0)
