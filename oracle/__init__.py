"""fp64 oracle of the GGUF weight-only quantized linear layer.

TEST INFRASTRUCTURE. Only tests/, `__graft_entry__.smoke()` and the CPU-baseline leg of
bench.py import this package; the product path (gguf_weight_only_gb300) never does, and the
two share no code. Two independent decoders live here:
  - qlinear_oracle.c: plain C, one weight at a time, fp64, rows split over POSIX threads;
  - oracle_np.py: numpy, every field read through unpackbits.
Both compute y[m, n] = sum_k x[m, k] * w[n, k] with w the exact dequantised weight.
Built on them: fused.py (the SiLU-gated and RMSNorm activations and the residual add, fp64)
and head.py (the embedding gather and the greedy output-head choice).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import oracle_np  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "qlinear_oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/_lib/liboracle.so (portable flags only)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        l.oracle_block_bytes.argtypes = [ctypes.c_int]
        l.oracle_block_bytes.restype = ctypes.c_int
        l.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        l.oracle_half_to_double.restype = ctypes.c_double
        l.oracle_dequant_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        l.oracle_dequant_f64.restype = ctypes.c_int
        l.oracle_qlinear_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        l.oracle_qlinear_f64.restype = ctypes.c_int
        _lib = l
    return _lib


def block_bytes(ggml_type: int) -> int:
    return lib().oracle_block_bytes(int(ggml_type))


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(int(bits))


def dequant(ggml_type: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """C oracle: packed (N x K/256 superblocks) -> (N, K) float64."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    need = N * (K // 256) * max(block_bytes(ggml_type), 0)
    if W.size < need:
        raise ValueError("packed buffer too small")
    out = np.empty((N, K), np.float64)
    rc = lib().oracle_dequant_f64(int(ggml_type), W.ctypes.data, N, K, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_dequant_f64 failed: {rc}")
    return out


def qlinear(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray, n_threads: int | None = None) -> np.ndarray:
    """C oracle: y[M, N] (float64) = x[M, K] . dequant(W)^T, x given as float16."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(np.asarray(x_f16, dtype=np.float16).reshape(-1, K))
    M = x.shape[0]
    need = N * (K // 256) * max(block_bytes(ggml_type), 0)
    if W.size < need:
        raise ValueError("packed buffer too small")
    y = np.empty((M, N), np.float64)
    if n_threads is None:
        n_threads = len(os.sched_getaffinity(0))
    rc = lib().oracle_qlinear_f64(int(ggml_type), W.ctypes.data, N, K, x.view(np.uint16).ctypes.data, M,
                                  y.ctypes.data, int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_qlinear_f64 failed: {rc}")
    return y


def qlinear_rows(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """y[:, rows] only (for sampled checks at full size): decodes just the requested rows."""
    bb = block_bytes(ggml_type)
    nsb = K // 256
    W = np.asarray(W, dtype=np.uint8).reshape(-1)
    rows = np.asarray(rows, dtype=np.int64)
    sub = np.concatenate([W[r * nsb * bb:(r + 1) * nsb * bb] for r in rows]) if len(rows) else np.zeros(0, np.uint8)
    return qlinear(ggml_type, sub, len(rows), K, x_f16)


def tolerance(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound 2e-3 * sum_k |x[m,k] * w[n,k]| (the stated tolerance)."""
    x = np.abs(np.asarray(x_f16, dtype=np.float16).astype(np.float64).reshape(-1, K))
    return 2e-3 * (x @ np.abs(dequant(ggml_type, W, N, K)).T)


def tolerance_rows(ggml_type: int, W: np.ndarray, N: int, K: int, x_f16: np.ndarray, rows: np.ndarray) -> np.ndarray:
    bb = block_bytes(ggml_type)
    nsb = K // 256
    W = np.asarray(W, dtype=np.uint8).reshape(-1)
    rows = np.asarray(rows, dtype=np.int64)
    sub = np.concatenate([W[r * nsb * bb:(r + 1) * nsb * bb] for r in rows]) if len(rows) else np.zeros(0, np.uint8)
    return tolerance(ggml_type, sub, len(rows), K, x_f16)
