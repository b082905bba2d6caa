"""fp64 oracle of the model-edge operations on GGUF weights: the embedding gather and the
output head's greedy token choice.

TEST INFRASTRUCTURE (as the rest of oracle/): only tests/ use it; it shares no code with the
CUDA path.

The pages dequantise one embedding row per token for a Q4_K token-embedding table and pick
the next token straight from a Q6_K output head without materialising the logits, checking
the fused choice against np.argmax of the materialised logits
(test/unit/test_llm_quant_cpu.py, test_q6_argmax_matches_materialized_logits).
"""
from __future__ import annotations

import numpy as np

from . import dequant as _dequant
from . import qlinear as _qlinear


def embed_rows(ggml_type: int, W: np.ndarray, N: int, K: int, ids: np.ndarray) -> np.ndarray:
    """Row ids[m] of dequant(W) for every m: (M, K) float64, the exact weights."""
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    if np.any(ids < 0) or np.any(ids >= N):
        raise ValueError("id out of range")
    bb = _block_bytes(ggml_type)
    nsb = K // 256
    W = np.asarray(W, dtype=np.uint8).reshape(-1)
    out = np.empty((len(ids), K), np.float64)
    for m, r in enumerate(ids):   # decode only the requested rows
        out[m] = _dequant(ggml_type, W[r * nsb * bb:(r + 1) * nsb * bb], 1, K)[0]
    return out


def argmax(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """For every token m: the first n with the largest y[m, n] of x . dequant(W)^T (fp64),
    and that largest value."""
    y = _qlinear(ggml_type, W, N, K, x_f16)
    idx = np.argmax(y, axis=1)   # first maximum on ties
    return idx, y[np.arange(y.shape[0]), idx]


def _block_bytes(ggml_type: int) -> int:
    from . import block_bytes
    return block_bytes(ggml_type)
