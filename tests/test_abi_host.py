"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every
function include/qlinear.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import gguf_weight_only_gb300 as ql
from gguf_weight_only_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlinear.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return ql.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(?:int|const char\s*\*|void)\s*\*?\s*(qlinear\w*)\s*\(", text)
    return sorted(set(names))


def test_header_lists_match_binding():
    assert declared_functions() == sorted(ql.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", qbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_block_bytes_and_metadata(lib):
    assert [ql.block_bytes(t) for t in (12, 13, 14, 23, 270)] == [144, 176, 210, 136, 224]
    assert ql.block_bytes(2) == -1
    assert ql.gemv_max_m() == 8
    for s in range(-10, 1):
        assert isinstance(ql.strerror(s), str) and ql.strerror(s) != "unknown status"
    assert ql.strerror(-99) == "unknown status"
    assert lib.qlinear_last_cuda_error() == 0


def test_launch_count(lib):
    assert ql.launch_count(12, 4096, 4096, 1) == 1
    assert ql.launch_count(12, 4096, 4096, 8) == 1
    assert ql.launch_count(12, 12288, 4096, 512) == 1
    assert ql.launch_count(12, 4096, 100, 1) == -2
    assert ql.launch_count(99, 4096, 4096, 1) == -1


BAD = [
    # (type, W, N, K, x, M, y, expected)
    (7, 16, 8, 256, 16, 1, 16, -1),          # unsupported type
    (12, 16, 8, 300, 16, 1, 16, -2),         # K not a multiple of 256
    (12, 16, 0, 256, 16, 1, 16, -2),         # N < 1
    (12, 16, 8, 256, 16, 0, 16, -2),         # M < 1
    (12, 16, 8, 0, 16, 1, 16, -2),           # K = 0
    (12, 0, 8, 256, 16, 1, 16, -3),          # null W
    (12, 16, 8, 256, 0, 1, 16, -3),          # null x
    (12, 16, 8, 256, 16, 1, 0, -3),          # null y
    (12, 24, 8, 256, 16, 1, 16, -4),         # misaligned W
    (12, 16, 8, 256, 40, 1, 16, -4),         # misaligned x
    (12, 16, 8, 256, 16, 1, 20, -4),         # misaligned y
    (12, 16, 8, 256, 16, 65535 * 32 + 1, 16, -2),   # more tokens than the prefill grid's token tiles
]


@pytest.mark.parametrize("fn", ["qlinear", "qlinear_gemv", "qlinear_gemm"])
@pytest.mark.parametrize("case", BAD)
def test_bad_arguments_rejected_before_launch(lib, fn, case):
    t, W, N, K, x, M, y, expect = case
    f = getattr(lib, fn)
    assert f(t, ctypes.c_void_p(W or None), N, K, ctypes.c_void_p(x or None), M, ctypes.c_void_p(y or None), None) == expect


def test_python_wrapper_raises_without_cuda_tensors(lib):
    import torch
    with pytest.raises(TypeError):
        ql.qlinear(torch.zeros(144, dtype=torch.uint8), 12, 1, 256, torch.zeros(1, 256, dtype=torch.float16))


def test_every_wrapper_rejects_host_tensors(lib):
    """Host (CPU) tensors are refused before anything reaches the library or a device."""
    import torch
    W = torch.zeros(144, dtype=torch.uint8)
    x = torch.zeros(1, 256, dtype=torch.float16)
    f32 = torch.zeros(1, 256, dtype=torch.float32)
    calls = [
        lambda: ql.qlinear_multi([W, W], 12, [1, 1], 256, x),
        lambda: ql.qlinear_silu_mul(W, 12, 1, 256, x, f32),
        lambda: ql.qlinear_rmsnorm(W, 12, 1, 256, f32, torch.zeros(256, dtype=torch.float32), 1e-6),
        lambda: ql.qlinear_argmax(W, 12, 1, 256, x),
        lambda: ql.qlinear_embed(W, 12, 1, 256, torch.zeros(1, dtype=torch.int32)),
        lambda: ql.repack(torch.zeros(210, dtype=torch.uint8), 14, 1, 256),
    ]
    for call in calls:
        with pytest.raises(TypeError):
            call()
    with pytest.raises(ValueError):   # checked before any tensor
        ql.qlinear_multi([W, W], 12, [1], 256, x)


# ------------------------------------------------------------------ qlinear_multi (projections sharing x)

def _multi(lib, t, W, N, K, x, M, y, n):
    k = max(len(W or N or y), 1)
    Wa = (ctypes.c_void_p * k)(*[w or None for w in W]) if W is not None else None
    Na = (ctypes.c_int64 * k)(*N) if N is not None else None
    Ya = (ctypes.c_void_p * k)(*[v or None for v in y]) if y is not None else None
    return lib.qlinear_multi(t, n, Wa, Na, K, ctypes.c_void_p(x or None), M, Ya, None)


def test_max_projections(lib):
    assert ql.max_projections() == 4


MULTI_BAD = [
    # (type, [W], [N], K, x, M, [y], n_proj override, expected)
    (12, None, [8, 8], 256, 16, 1, [16, 32], 2, -3),              # NULL W array
    (12, [16, 32], None, 256, 16, 1, [16, 32], 2, -3),            # NULL N array
    (12, [16, 32], [8, 8], 256, 16, 1, None, 2, -3),              # NULL y array
    (12, [16], [8], 256, 16, 1, [16], 0, -2),                     # no projection
    (12, [16] * 5, [8] * 5, 256, 16, 1, [16] * 5, 5, -2),         # more than 4
    (7, [16, 32], [8, 8], 256, 16, 1, [16, 32], 2, -1),           # unsupported type
    (12, [16, 32], [8, 8], 300, 16, 1, [16, 32], 2, -2),          # K not a multiple of 256
    (12, [16, 32], [8, 0], 256, 16, 1, [16, 32], 2, -2),          # second projection N < 1
    (12, [16, 32], [8, 8], 256, 16, 0, [16, 32], 2, -2),          # M < 1
    (12, [16, 0], [8, 8], 256, 16, 1, [16, 32], 2, -3),           # second W NULL
    (12, [16, 32], [8, 8], 256, 0, 1, [16, 32], 2, -3),           # x NULL
    (12, [16, 32], [8, 8], 256, 16, 1, [16, 0], 2, -3),           # second y NULL
    (12, [16, 40], [8, 8], 256, 16, 1, [16, 32], 2, -4),          # second W misaligned
    (12, [16, 32], [8, 8], 256, 24, 1, [16, 32], 2, -4),          # x misaligned
    (12, [16, 32, 48], [8, 8, 8], 256, 16, 1, [16, 32, 52], 3, -4),  # third y misaligned
]


@pytest.mark.parametrize("case", MULTI_BAD)
def test_multi_bad_arguments_rejected_before_launch(lib, case):
    t, W, N, K, x, M, y, n, expect = case
    assert _multi(lib, t, W, N, K, x, M, y, n) == expect


# ------------------------------------------------------------------ fused prologues

FUSED_BAD = [
    # (fn, type, W, N, K, a, b, M, residual, y, extra(eps, xnorm), expected)
    ("silu", 7, 16, 8, 256, 16, 32, 1, 0, 48, None, -1),
    ("silu", 12, 16, 8, 300, 16, 32, 1, 0, 48, None, -2),
    ("silu", 12, 16, 8, 256, 16, 32, 0, 0, 48, None, -2),
    ("silu", 12, 0, 8, 256, 16, 32, 1, 0, 48, None, -3),
    ("silu", 12, 16, 8, 256, 0, 32, 1, 0, 48, None, -3),
    ("silu", 12, 16, 8, 256, 16, 0, 1, 0, 48, None, -3),
    ("silu", 12, 16, 8, 256, 16, 32, 1, 0, 0, None, -3),
    ("silu", 12, 16, 8, 256, 24, 32, 1, 0, 48, None, -4),
    ("silu", 12, 16, 8, 256, 16, 40, 1, 0, 48, None, -4),
    ("silu", 12, 16, 8, 256, 16, 32, 1, 72, 48, None, -4),
    ("silu", 12, 16, 8, 256, 16, 32, 9, 0, 48, None, -7),
    ("rms", 12, 16, 8, 256, 16, 32, 1, 0, 48, (-1.0, 0), -2),
    ("rms", 12, 16, 8, 256, 16, 32, 1, 0, 48, (float("nan"), 0), -2),
    ("rms", 12, 16, 8, 256, 16, 0, 1, 0, 48, (1e-6, 0), -3),
    ("rms", 12, 16, 8, 256, 16, 32, 1, 0, 48, (1e-6, 88), -4),
    ("rms", 12, 16, 8, 256, 16, 32, 9, 0, 48, (1e-6, 0), -7),
]


@pytest.mark.parametrize("case", FUSED_BAD)
def test_fused_bad_arguments_rejected_before_launch(lib, case):
    fn, t, W, N, K, a, b, M, r, y, extra, expect = case
    v = lambda p: ctypes.c_void_p(p or None)
    if fn == "silu":
        rc = lib.qlinear_silu_mul(t, v(W), N, K, v(a), v(b), M, v(r), v(y), None)
    else:
        eps, xn = extra
        rc = lib.qlinear_rmsnorm(t, v(W), N, K, v(a), v(b), eps, M, v(r), v(y), v(xn), None)
    assert rc == expect


# ------------------------------------------------------------------ greedy head and embedding gather

HEAD_BAD = [
    # (type, W, N, K, x, M, index_out, value_out, expected)
    (7, 16, 8, 256, 16, 1, 32, 48, -1),
    (12, 16, 8, 300, 16, 1, 32, 48, -2),
    (12, 16, 0, 256, 16, 1, 32, 48, -2),
    (12, 0, 8, 256, 16, 1, 32, 48, -3),
    (12, 16, 8, 256, 0, 1, 32, 48, -3),
    (12, 16, 8, 256, 16, 1, 0, 48, -3),
    (12, 24, 8, 256, 16, 1, 32, 48, -4),
    (12, 16, 8, 256, 16, 1, 40, 48, -4),
    (12, 16, 8, 256, 16, 1, 32, 52, -4),
    (12, 16, 8, 256, 16, 9, 32, 48, -7),
]


@pytest.mark.parametrize("case", HEAD_BAD)
def test_argmax_bad_arguments_rejected_before_launch(lib, case):
    t, W, N, K, x, M, io, vo, expect = case
    v = lambda p: ctypes.c_void_p(p or None)
    assert lib.qlinear_argmax(t, v(W), N, K, v(x), M, v(io), v(vo), None) == expect


EMBED_BAD = [
    # (type, W, N, K, ids, M, out, fp16, expected)
    (7, 16, 8, 256, 32, 1, 48, 0, -1),
    (12, 16, 8, 300, 32, 1, 48, 0, -2),
    (12, 16, 0, 256, 32, 1, 48, 0, -2),
    (12, 16, 8, 256, 32, 0, 48, 1, -2),
    (12, 0, 8, 256, 32, 1, 48, 0, -3),
    (12, 16, 8, 256, 0, 1, 48, 0, -3),
    (12, 16, 8, 256, 32, 1, 0, 1, -3),
    (12, 24, 8, 256, 32, 1, 48, 0, -4),
    (12, 16, 8, 256, 34, 1, 48, 0, -4),
    (12, 16, 8, 256, 32, 1, 56, 1, -4),
]


@pytest.mark.parametrize("case", EMBED_BAD)
def test_embed_bad_arguments_rejected_before_launch(lib, case):
    t, W, N, K, ids, M, out, fp16, expect = case
    v = lambda p: ctypes.c_void_p(p or None)
    assert lib.qlinear_embed(t, v(W), N, K, v(ids), M, v(out), fp16, None) == expect


REPACK_BAD = [
    # (type, W_src, N, K, W_dst, expected)
    (12, 16, 8, 256, 32, -1),     # only Q6_K is repacked
    (270, 16, 8, 256, 32, -1),
    (14, 16, 8, 300, 32, -2),
    (14, 16, 0, 256, 32, -2),
    (14, 0, 8, 256, 32, -3),
    (14, 16, 8, 256, 0, -3),
    (14, 24, 8, 256, 32, -4),
    (14, 16, 8, 256, 40, -4),
]


@pytest.mark.parametrize("case", REPACK_BAD)
def test_repack_bad_arguments_rejected_before_launch(lib, case):
    t, src, N, K, dst, expect = case
    v = lambda p: ctypes.c_void_p(p or None)
    assert lib.qlinear_repack(t, v(src), N, K, v(dst), None) == expect


# ------------------------------------------------------------------ qlinear_copy

def test_copy_bad_arguments_rejected_before_launch(lib):
    assert lib.qlinear_copy(ctypes.c_void_p(16), ctypes.c_void_p(16), -1, None) == -2    # bytes < 0
    assert lib.qlinear_copy(ctypes.c_void_p(None), ctypes.c_void_p(16), 8, None) == -3  # null dst
    assert lib.qlinear_copy(ctypes.c_void_p(16), ctypes.c_void_p(None), 8, None) == -3  # null src
    assert lib.qlinear_copy(ctypes.c_void_p(None), ctypes.c_void_p(None), 0, None) == 0  # nothing to do


def test_copy_wrapper_checks_its_tensors(lib):
    import torch
    a = torch.zeros(8, dtype=torch.float32)
    with pytest.raises(ValueError):   # plain (pageable) host memory
        ql.copy(a, torch.zeros(8, dtype=torch.float32))
    with pytest.raises(ValueError):   # not contiguous
        ql.copy(torch.zeros(4, 4)[:, 1], torch.zeros(4))
