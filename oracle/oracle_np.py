"""Vectorised numpy decoder of the four GGUF superblock formats (fp64), written apart from
the C oracle in qlinear_oracle.c so that the two can be checked against each other.

TEST INFRASTRUCTURE: only tests/, the smoke check and the benchmark's CPU-baseline leg use
this module. The CUDA path never imports it.

Where the C oracle walks one weight at a time, this module reads every bit field through
`np.unpackbits` (little-endian bit order): a field "bits a..b of byte B" is the slice
bits[..., 8*B + a : 8*B + b + 1] read back as an unsigned integer. Field placement:
  - block byte sizes (144/176/210/136): tinygrad/llm/gguf.py, the _GGML_QUANT table;
  - Q4_K = Q5_K without the 32-byte high-bit array, qs at word 4 (byte 16): commit log of
    explicit-dev, commit "custom kernels: Q4_K support (ggml type 12)";
  - d / dmin offsets: test/unit/test_llm_quant_cpu.py, random_packed();
  - IQ4_XS codebook and [low nibbles, high nibbles] order of a 16-byte group:
    test/unit/test_llm_quant_cpu.py, test_unpack_lut_dot_uop;
  - the rest of the bit placement is the GGUF on-disk layout (not printed on the pages).
"""
from __future__ import annotations

import numpy as np

BLOCK_BYTES = {12: 144, 13: 176, 14: 210, 23: 136}
IQ4_CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113],
                        dtype=np.float64)


def _bits(b: np.ndarray) -> np.ndarray:
    """(nb, nbytes) uint8 -> (nb, 8*nbytes) bits, bit i of byte B at column 8*B + i."""
    return np.unpackbits(b, axis=1, bitorder="little").astype(np.int64)


def _field(bits: np.ndarray, start: int, width: int) -> np.ndarray:
    """Unsigned integer made of `width` consecutive bits starting at bit column `start`."""
    weights = 1 << np.arange(width, dtype=np.int64)
    return bits[:, start:start + width] @ weights


def _f16(blocks: np.ndarray, off: int) -> np.ndarray:
    return np.ascontiguousarray(blocks[:, off:off + 2]).view(np.float16).reshape(-1).astype(np.float64)


def _kquant_scales(S: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """12-byte field -> (scale, min) arrays of shape (nb, 8)."""
    bits = _bits(S)
    sc = np.empty((S.shape[0], 8), np.int64)
    mn = np.empty((S.shape[0], 8), np.int64)
    for j in range(4):
        sc[:, j] = _field(bits, 8 * j, 6)
        mn[:, j] = _field(bits, 8 * (j + 4), 6)
        # sub-block j+4: low 4 bits from byte j+8 (low / high nibble), high 2 bits from the
        # top two bits of byte j (scale) or byte j+4 (min)
        sc[:, j + 4] = _field(bits, 8 * (j + 8), 4) + (_field(bits, 8 * j + 6, 2) << 4)
        mn[:, j + 4] = _field(bits, 8 * (j + 8) + 4, 4) + (_field(bits, 8 * (j + 4) + 6, 2) << 4)
    return sc, mn


def _nibbles_grouped(qs: np.ndarray, group: int) -> np.ndarray:
    """qs (nb, 128) -> (nb, 256) values: each run of `group` bytes yields its `group` low
    nibbles followed by its `group` high nibbles."""
    nb = qs.shape[0]
    g = qs.reshape(nb, -1, group)
    return np.concatenate([g & 15, g >> 4], axis=2).reshape(nb, 256).astype(np.int64)


def dequant_blocks(ggml_type: int, blocks: np.ndarray) -> np.ndarray:
    """(nb, block_bytes) uint8 -> (nb, 256) float64 exact weights."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    nb = blocks.shape[0]
    if ggml_type in (12, 13):
        d, dmin = _f16(blocks, 0), _f16(blocks, 2)
        sc, mn = _kquant_scales(blocks[:, 4:16])
        qs = blocks[:, 16:144] if ggml_type == 12 else blocks[:, 48:176]
        q = _nibbles_grouped(qs, 32)                          # 64 weights per 32 bytes
        if ggml_type == 13:
            hb = _bits(blocks[:, 16:48]).reshape(nb, 32, 8)   # [l, bit] for byte qh[l]
            q = q + 16 * hb.transpose(0, 2, 1).reshape(nb, 256)   # weight 32*j + l <- bit j of qh[l]
        sub_sc = np.repeat(sc, 32, axis=1)
        sub_mn = np.repeat(mn, 32, axis=1)
        return d[:, None] * sub_sc * q - dmin[:, None] * sub_mn
    if ggml_type == 14:
        d = _f16(blocks, 208)
        sc = blocks[:, 192:208].view(np.int8).astype(np.int64)
        ql = blocks[:, 0:128].reshape(nb, 2, 64)              # two halves of 128 weights
        qh = _bits(blocks[:, 128:192]).reshape(nb, 2, 32, 8)  # [half, l, bit]
        q = np.empty((nb, 2, 4, 32), np.int64)                # [half, quarter t, l]
        for t in range(4):
            lbytes = ql[:, :, 32 * (t % 2):32 * (t % 2) + 32].astype(np.int64)
            low4 = (lbytes & 15) if t < 2 else (lbytes >> 4)
            high2 = qh[:, :, :, 2 * t] + 2 * qh[:, :, :, 2 * t + 1]
            q[:, :, t, :] = low4 + 16 * high2
        q = q.reshape(nb, 256)
        return d[:, None] * np.repeat(sc, 16, axis=1) * (q - 32)
    if ggml_type == 23:
        d = _f16(blocks, 0)
        hbits = _bits(blocks[:, 2:4])                         # scales_h, 16 bits
        lbits = _bits(blocks[:, 4:8])                         # scales_l, 32 bits
        ls = np.stack([_field(lbits, 4 * j, 4) + (_field(hbits, 2 * j, 2) << 4) for j in range(8)], axis=1)
        nib = _nibbles_grouped(blocks[:, 8:136], 16)
        return d[:, None] * np.repeat(ls - 32, 32, axis=1) * IQ4_CODEBOOK[nib]
    raise ValueError(f"unsupported ggml type {ggml_type}")


def dequant(ggml_type: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Packed matrix (N rows x K/256 superblocks, contiguous) -> (N, K) float64."""
    bb = BLOCK_BYTES[ggml_type]
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    blocks = np.asarray(W, dtype=np.uint8).reshape(-1)[: N * (K // 256) * bb].reshape(-1, bb)
    return dequant_blocks(ggml_type, blocks).reshape(N, K)


def qlinear_f64(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray) -> np.ndarray:
    """y[M, N] = x[M, K] . dequant(W)^T in fp64 (library matmul for the contraction)."""
    x = np.asarray(x_f16, dtype=np.float16).astype(np.float64).reshape(-1, K)
    return x @ dequant(ggml_type, W, N, K).T
