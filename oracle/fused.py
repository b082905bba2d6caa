"""fp64 oracle of the fused decode prologues and epilogue.

TEST INFRASTRUCTURE (as the rest of oracle/): only tests/ and the CPU-baseline leg of
bench.py use it; it shares no code with the CUDA path.

The pages fuse two element-wise producers into the linear layer that consumes them and check
that the fused result equals the separate steps (test/unit/test_llm_quant_cpu.py):
  - test_q8_silu_linear_matches_separate: layer(silu_mul(gate, up).half()), gate fp16 and
    up fp32; silu(g) = g * sigmoid(g) = g / (1 + exp(-g)).
  - test_f16_linear_matches_standard: rmsnorm_f16_linear(norm, layer, x) returns the
    normalised activations and layer(normalised); RMSNorm(x) = x * rsqrt(mean(x^2) + eps) * w
    (tinygrad nn.RMSNorm), the mean taken over the feature axis.
The activations the layer consumes are fp16 (".half()"): each prologue value is computed in
fp64 and rounded once to fp16. The epilogue adds an fp32 residual [M, N] to y.
"""
from __future__ import annotations

import numpy as np

from . import qlinear as _qlinear
from . import tolerance as _tolerance


def silu(g: np.ndarray) -> np.ndarray:
    """g / (1 + e^-g) in fp64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def silu_mul_x(gate_f16: np.ndarray, up_f32: np.ndarray) -> np.ndarray:
    """The layer input of the SiLU-gated prologue: fp16(silu(gate) * up), gate read as fp16,
    up as fp32, the product formed in fp64 and rounded once."""
    g = np.asarray(gate_f16, dtype=np.float16).astype(np.float64)
    u = np.asarray(up_f32, dtype=np.float32).astype(np.float64)
    return (silu(g) * u).astype(np.float16)


def rmsnorm(h_f32: np.ndarray, w_f32: np.ndarray, eps: float) -> np.ndarray:
    """h * rsqrt(mean(h^2) + eps) * w over the last axis, in fp64 (h fp32 [M, K], w fp32 [K])."""
    h = np.asarray(h_f32, dtype=np.float32).astype(np.float64)
    w = np.asarray(w_f32, dtype=np.float32).astype(np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + float(np.float32(eps))) * w


def rmsnorm_x(h_f32: np.ndarray, w_f32: np.ndarray, eps: float) -> np.ndarray:
    """The layer input of the RMSNorm prologue: rmsnorm rounded once to fp16."""
    return rmsnorm(h_f32, w_f32, eps).astype(np.float16)


def qlinear_fused(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray,
                  residual: np.ndarray | None = None) -> np.ndarray:
    """y = x . dequant(W)^T (+ residual), fp64, for the prologue's fp16 x."""
    y = _qlinear(ggml_type, W, N, K, x_f16)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float32).astype(np.float64).reshape(y.shape)
    return y


def tolerance_fused(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray,
                    residual: np.ndarray | None = None) -> np.ndarray:
    """The layer's bound for the contraction, 2e-3 * sum_k |x_k w_k|, widened by the one fp16
    ulp by which a prologue computed in fp32 and then rounded to fp16 may land on the other
    side of a rounding boundary than the fp64 value: an fp16 ulp is at most 2^-10 |x_k| for
    normal values and 2^-24 below 2^-14, so the contraction moves by at most
    sum_k (2^-10 |x_k| + 2^-24) |w_k|. With a residual, its fp32 addition adds at most
    2^-24 (|y| + |r|); the |y| part is inside the first term, 2^-23 |r| is added."""
    from . import dequant as _dequant
    x = np.abs(np.asarray(x_f16, dtype=np.float16).astype(np.float64).reshape(-1, K))
    aw = np.abs(_dequant(ggml_type, W, N, K))
    tol = _tolerance(ggml_type, W, N, K, x_f16) + 2.0 ** -10 * (x @ aw.T) + 2.0 ** -24 * aw.sum(axis=1)[None, :]
    if residual is not None:
        tol = tol + 2.0 ** -23 * np.abs(np.asarray(residual, dtype=np.float32).astype(np.float64).reshape(tol.shape))
    return tol
