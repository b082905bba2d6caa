"""Seeded synthetic inputs for the quantized linear layer: packed weight blocks and fp16
activations. Shared by the tests, the smoke check and the benchmark, and by both the oracle
side and the CUDA side of the parity tests.

This module holds none of the layer's arithmetic: it writes uniformly random bytes and
places fp16 scale values at their byte offsets. Uniform random bytes are the stated
distributions because the packed fields are bijections of the values they hold:
  - the 12-byte K-quant scale field is exactly 16 six-bit values (sc[8], m[8]);
  - IQ4_XS scales_h (16 bits) + scales_l (32 bits) are exactly 8 six-bit values;
  - qs / qh / ql bytes are nibbles / bit fields with every pattern allowed.
The only non-uniform fields are the fp16 d / dmin (uniform in [2^-10, 2^-6], rounded to
nearest fp16) and the Q6_K int8 sub-block scales (uniform integers in [-32, 31]).
"""
from __future__ import annotations

import numpy as np

# ggml type id -> bytes per 256-weight superblock (tinygrad/llm/gguf.py, _GGML_QUANT).
BLOCK_BYTES = {12: 144, 13: 176, 14: 210, 23: 136}
TYPE_NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K", 23: "IQ4_XS"}
TYPE_IDS = {v: k for k, v in TYPE_NAMES.items()}

# Byte offsets of the fp16 super-scales inside a block (test/unit/test_llm_quant_cpu.py,
# random_packed: d at 0..1, dmin at 2..3 for Q4_K/Q5_K, d in the last two bytes of Q6_K).
_D_OFFSETS = {12: (0, 2), 13: (0, 2), 14: (208,), 23: (0,)}
_Q6K_SCALES = (192, 208)

D_LO, D_HI = 2.0 ** -10, 2.0 ** -6


def blocks(ggml_type: int, n_blocks: int, seed) -> np.ndarray:
    """(n_blocks, block_bytes) uint8 drawn from the stated distributions.

    Draw order (all vectorised over blocks): every byte uniform, then each fp16
    super-scale in offset order, then (Q6_K) the int8 sub-block scales."""
    bb = BLOCK_BYTES[ggml_type]
    rng = np.random.default_rng(seed)
    out = rng.integers(0, 256, size=(n_blocks, bb), dtype=np.uint8)
    for off in _D_OFFSETS[ggml_type]:
        d = rng.uniform(D_LO, D_HI, size=n_blocks).astype(np.float16)
        out[:, off:off + 2] = d.view(np.uint8).reshape(n_blocks, 2)
    if ggml_type == 14:
        lo, hi = _Q6K_SCALES
        out[:, lo:hi] = rng.integers(-32, 32, size=(n_blocks, hi - lo)).astype(np.int8).view(np.uint8)
    return out


def weights(ggml_type: int, N: int, K: int, seed) -> np.ndarray:
    """Packed N x K matrix as a flat uint8 array: row n, superblock b at byte (n*K/256 + b)*bb."""
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    return blocks(ggml_type, N * (K // 256), seed).reshape(-1)


def activations(M: int, K: int, seed) -> np.ndarray:
    """x[M, K] float16 = fp16(N(0, 1)), round to nearest even."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((M, K)).astype(np.float16)


# Layer shapes of the workloads (K, N); see the design notes for their origin.
DECODE_8B_SHAPES = [(4096, 4096), (4096, 1024), (4096, 12288), (12288, 4096)]   # Q4_K, M = 1 and 4
DECODE_27B_SHAPES = [(5120, 5120), (5120, 17408), (17408, 5120)]               # IQ4_XS, M = 1
PREFILL_SHAPE = (4096, 12288)                                                    # Q4_K, M in 32/128/512
KQUANT_SWEEP_SHAPE = (5120, 17408)                                              # Q5_K / Q6_K, M in 1/256


def workload_seed(cfg: int, shape_idx: int) -> list[int]:
    return [cfg, shape_idx]


def activation_seed(cfg: int, shape_idx: int, M: int) -> list[int]:
    return [cfg, shape_idx, M, 1]
