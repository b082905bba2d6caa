"""GB300 (sm_103a) GGUF weight-only quantized linear layer: Python binding.

Thin ctypes marshalling over the C ABI in include/qlinear.h (library
gguf_weight_only_gb300/_lib/libqlinear.so, built by `gguf_weight_only_gb300.build`). Every
step of the computation runs in the library's CUDA kernels; PyTorch only provides device
memory and the current stream. There is no CPU fallback: if the library is missing, every
call raises.

    y = qlinear(W_u8_cuda, ggml_type, N, K, x_f16_cuda)      # -> (M, N) float32 cuda
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# QL_DEBUG=1 in the environment loads the bounds-checking build (build.build(debug=True)).
DEBUG = os.environ.get("QL_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "_lib_debug" if DEBUG else "_lib", "libqlinear.so")

Q4_K, Q5_K, Q6_K, IQ4_XS = 12, 13, 14, 23
STATUS = {0: "QL_OK", -1: "QL_ERR_TYPE", -2: "QL_ERR_SHAPE", -3: "QL_ERR_NULL", -4: "QL_ERR_ALIGN",
          -5: "QL_ERR_CUDA", -6: "QL_ERR_TIMEOUT", -7: "QL_ERR_UNSUPPORTED", -8: "QL_ERR_DEVICE",
          -9: "QL_ERR_INDEX", -10: "QL_ERR_BOUNDS"}
# Every function include/qlinear.h declares (the symbol-export test checks this list
# against the header).
EXPORTS = ("qlinear", "qlinear_gemv", "qlinear_gemm", "qlinear_block_bytes", "qlinear_gemv_max_m",
           "qlinear_strerror", "qlinear_last_cuda_error", "qlinear_device_status", "qlinear_launch_count",
           "qlinear_selftest_wait_timeout", "qlinear_multi", "qlinear_max_projections", "qlinear_silu_mul",
           "qlinear_rmsnorm", "qlinear_argmax", "qlinear_embed", "qlinear_repack", "qlinear_copy", "qlinear_gemm_plan")
Q6_K_A16 = 270   # Q6_K in 224-byte aligned blocks (qlinear_repack)

_lib = None


class QLinearError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run gguf_weight_only_gb300.build.build())")
        l = ctypes.CDLL(LIB_PATH)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        for name in ("qlinear", "qlinear_gemv", "qlinear_gemm"):
            f = getattr(l, name)
            f.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
            f.restype = ctypes.c_int
        l.qlinear_block_bytes.argtypes = [ctypes.c_int]
        l.qlinear_block_bytes.restype = ctypes.c_int
        l.qlinear_gemv_max_m.argtypes = []
        l.qlinear_gemv_max_m.restype = ctypes.c_int
        l.qlinear_strerror.argtypes = [ctypes.c_int]
        l.qlinear_strerror.restype = ctypes.c_char_p
        l.qlinear_last_cuda_error.argtypes = []
        l.qlinear_last_cuda_error.restype = ctypes.c_int
        l.qlinear_device_status.argtypes = [vp]
        l.qlinear_device_status.restype = ctypes.c_int
        l.qlinear_launch_count.argtypes = [ctypes.c_int, i64, i64, i64]
        l.qlinear_launch_count.restype = ctypes.c_int
        l.qlinear_selftest_wait_timeout.argtypes = [vp]
        l.qlinear_selftest_wait_timeout.restype = ctypes.c_int
        l.qlinear_multi.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(i64), i64, vp, i64,
                                    ctypes.POINTER(vp), vp]
        l.qlinear_multi.restype = ctypes.c_int
        l.qlinear_max_projections.argtypes = []
        l.qlinear_max_projections.restype = ctypes.c_int
        l.qlinear_silu_mul.argtypes = [ctypes.c_int, vp, i64, i64, vp, vp, i64, vp, vp, vp]
        l.qlinear_silu_mul.restype = ctypes.c_int
        l.qlinear_rmsnorm.argtypes = [ctypes.c_int, vp, i64, i64, vp, vp, ctypes.c_float, i64, vp, vp, vp, vp]
        l.qlinear_rmsnorm.restype = ctypes.c_int
        l.qlinear_argmax.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp, vp]
        l.qlinear_argmax.restype = ctypes.c_int
        l.qlinear_embed.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, ctypes.c_int, vp]
        l.qlinear_embed.restype = ctypes.c_int
        l.qlinear_repack.argtypes = [ctypes.c_int, vp, i64, i64, vp, vp]
        l.qlinear_repack.restype = ctypes.c_int
        l.qlinear_copy.argtypes = [vp, vp, i64, vp]
        l.qlinear_copy.restype = ctypes.c_int
        l.qlinear_gemm_plan.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(i64)]
        l.qlinear_gemm_plan.restype = ctypes.c_int
        _lib = l
    return _lib


def strerror(status: int) -> str:
    return lib().qlinear_strerror(int(status)).decode()


def _check(status: int, what) -> None:
    if status != 0:
        what = what() if callable(what) else what
        extra = ""
        if status == -5:
            extra = f" (cudaError {lib().qlinear_last_cuda_error()})"
        raise QLinearError(status, f"{what}: {STATUS.get(status, status)}: {strerror(status)}{extra}")


_block_bytes_cache: dict = {}


def block_bytes(ggml_type: int) -> int:
    t = int(ggml_type)
    b = _block_bytes_cache.get(t)
    if b is None:
        b = _block_bytes_cache[t] = lib().qlinear_block_bytes(t)
    return b


def gemv_max_m() -> int:
    return lib().qlinear_gemv_max_m()


def launch_count(ggml_type: int, N: int, K: int, M: int) -> int:
    return lib().qlinear_launch_count(int(ggml_type), int(N), int(K), int(M))


def selftest_wait_timeout(stream=None) -> None:
    """Enqueue the diagnostic kernel whose bounded wait runs out (about 2 s); the next
    device_status() then reports QL_ERR_TIMEOUT. Exercises the failure path without a fault."""
    rc = lib().qlinear_selftest_wait_timeout(_stream_handle(stream))
    if rc != 0:
        raise QLinearError(rc, f"qlinear_selftest_wait_timeout: {strerror(rc)}")


def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _device_of(*tensors):
    """torch.cuda.device context of the one CUDA device all tensor arguments live on: the library
    launches on the current device, so a call runs with its tensors' device current (and on that
    device's current stream unless a stream is given, which must belong to it)."""
    import torch
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"tensor arguments must all be on one CUDA device, got {sorted(map(str, devs))}")
    return torch.cuda.device(devs.pop())


def _check_stream(stream, tensor) -> None:
    if stream is not None and stream.device != tensor.device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {tensor.device}")


def qlinear_raw(path: str, ggml_type: int, W_ptr: int, N: int, K: int, x_ptr: int, M: int, y_ptr: int,
                stream_handle: int) -> None:
    """Direct C-ABI call on raw device pointers (no checks beyond the library's own)."""
    l = lib()
    fn = l.qlinear if path == "auto" else l.qlinear_gemv if path == "gemv" else l.qlinear_gemm if path == "gemm" else None
    if fn is None:
        raise ValueError(f"unknown path {path!r}")
    _check(fn(int(ggml_type), W_ptr, int(N), int(K), x_ptr, int(M), y_ptr, stream_handle), lambda: f"qlinear[{path}]")


def qlinear(W, ggml_type: int, N: int, K: int, x, out=None, path: str = "auto", stream=None):
    """y[M, N] float32 = x[M, K] (fp16) . dequant(W)^T on the current CUDA stream.

    W: uint8 CUDA tensor holding N*K/256 packed superblocks (contiguous, 16-byte aligned).
    x: float16 CUDA tensor of shape (M, K) or (K,). path: "auto" | "gemv" | "gemm".
    """
    import torch
    if not (isinstance(W, torch.Tensor) and W.is_cuda and W.dtype == torch.uint8):
        raise TypeError("W must be a uint8 CUDA tensor")
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float16):
        raise TypeError("x must be a float16 CUDA tensor")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError(f"x must have shape (M, {K})")
    if not (W.is_contiguous() and x.is_contiguous()):
        raise ValueError("W and x must be contiguous")
    bb = block_bytes(ggml_type)
    if bb > 0 and W.numel() < N * (K // 256) * bb:
        raise ValueError("W holds fewer bytes than N*K/256 superblocks")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    elif not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() >= M * N):
        raise ValueError("out must be a contiguous float32 CUDA tensor with M*N elements")
    _check_stream(stream, x)
    with _device_of(W, x, out):
        qlinear_raw(path, ggml_type, W.data_ptr(), N, K, x.data_ptr(), M, out.data_ptr(), _stream_handle(stream))
    return out


def max_projections() -> int:
    return lib().qlinear_max_projections()


def qlinear_multi(Ws, ggml_type: int, Ns, K: int, x, outs=None, stream=None):
    """[y_j] = [x . dequant(W_j)^T] for projections sharing x and K, in one decode launch
    when M <= 8 (each W_j a uint8 CUDA tensor of Ns[j] rows; x float16 (M, K) or (K,))."""
    import torch
    Ws, Ns = list(Ws), [int(n) for n in Ns]
    if len(Ws) != len(Ns):
        raise ValueError("Ws and Ns differ in length")
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float16):
        raise TypeError("x must be a float16 CUDA tensor")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dim() != 2 or x.shape[1] != K or not x.is_contiguous():
        raise ValueError(f"x must be a contiguous (M, {K}) tensor")
    M = x.shape[0]
    bb = block_bytes(ggml_type)
    for W, N in zip(Ws, Ns):
        if not (isinstance(W, torch.Tensor) and W.is_cuda and W.dtype == torch.uint8 and W.is_contiguous()):
            raise TypeError("each W must be a contiguous uint8 CUDA tensor")
        if bb > 0 and W.numel() < N * (K // 256) * bb:
            raise ValueError("a W holds fewer bytes than N*K/256 superblocks")
    if outs is None:
        outs = [torch.empty((M, N), dtype=torch.float32, device=x.device) for N in Ns]
    elif len(outs) != len(Ns) or not all(o.is_cuda and o.dtype == torch.float32 and o.is_contiguous()
                                         and o.numel() >= M * N for o, N in zip(outs, Ns)):
        raise ValueError("outs must be contiguous float32 CUDA tensors of M*N[j] elements")
    n = len(Ws)
    w_arr = (ctypes.c_void_p * max(n, 1))(*[W.data_ptr() for W in Ws])
    n_arr = (ctypes.c_int64 * max(n, 1))(*Ns)
    y_arr = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in outs])
    _check_stream(stream, x)
    with _device_of(x, *Ws, *outs):
        _check(lib().qlinear_multi(int(ggml_type), n, w_arr, n_arr, int(K), x.data_ptr(), M, y_arr,
                                   _stream_handle(stream)), "qlinear_multi")
    return outs


def _mk(x, dtype, shape, what):
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == dtype and x.is_contiguous()):
        raise TypeError(f"{what} must be a contiguous {dtype} CUDA tensor")
    n = 1
    for d in shape:
        n *= int(d)
    if x.numel() != n:
        raise ValueError(f"{what} must have {n} elements (shape {tuple(shape)})")
    return x


def _fused_common(W, ggml_type, N, K, M, residual, out, dev):
    import torch
    if not (isinstance(W, torch.Tensor) and W.is_cuda and W.dtype == torch.uint8 and W.is_contiguous()):
        raise TypeError("W must be a contiguous uint8 CUDA tensor")
    bb = block_bytes(ggml_type)
    if bb > 0 and W.numel() < N * (K // 256) * bb:
        raise ValueError("W holds fewer bytes than N*K/256 superblocks")
    if residual is not None:
        _mk(residual, torch.float32, (M, N), "residual")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    else:
        _mk(out, torch.float32, (M, N), "out")
    return out


def qlinear_silu_mul(W, ggml_type: int, N: int, K: int, gate, up, residual=None, out=None, stream=None):
    """y = fp16(silu(gate) * up) . dequant(W)^T (+ residual), one decode launch (M <= 8).
    gate: float16 (M, K); up: float32 (M, K); residual: float32 (M, N) or None (may be out)."""
    import torch
    M = gate.shape[0] if gate.dim() == 2 else 1
    _mk(gate, torch.float16, (M, K), "gate")
    _mk(up, torch.float32, (M, K), "up")
    out = _fused_common(W, ggml_type, N, K, M, residual, out, gate.device)
    _check_stream(stream, gate)
    with _device_of(W, gate, up, residual, out):
        _check(lib().qlinear_silu_mul(int(ggml_type), W.data_ptr(), int(N), int(K), gate.data_ptr(), up.data_ptr(), M,
                                      residual.data_ptr() if residual is not None else None, out.data_ptr(),
                                      _stream_handle(stream)), "qlinear_silu_mul")
    return out


def qlinear_rmsnorm(W, ggml_type: int, N: int, K: int, h, norm_w, eps: float, residual=None, out=None, xnorm=None,
                    stream=None):
    """y = fp16(h * rsqrt(mean(h^2) + eps) * norm_w) . dequant(W)^T (+ residual), one decode
    launch (M <= 8). h: float32 (M, K); norm_w: float32 (K,); xnorm: optional float16 (M, K)
    that receives the normalised fp16 activations."""
    import torch
    M = h.shape[0] if h.dim() == 2 else 1
    _mk(h, torch.float32, (M, K), "h")
    _mk(norm_w, torch.float32, (K,), "norm_w")
    if xnorm is not None:
        _mk(xnorm, torch.float16, (M, K), "xnorm")
    out = _fused_common(W, ggml_type, N, K, M, residual, out, h.device)
    _check_stream(stream, h)
    with _device_of(W, h, norm_w, residual, out, xnorm):
        _check(lib().qlinear_rmsnorm(int(ggml_type), W.data_ptr(), int(N), int(K), h.data_ptr(), norm_w.data_ptr(),
                                     float(eps), M, residual.data_ptr() if residual is not None else None,
                                     out.data_ptr(), xnorm.data_ptr() if xnorm is not None else None,
                                     _stream_handle(stream)), "qlinear_rmsnorm")
    return out


def _weights(W, ggml_type, N, K):
    import torch
    if not (isinstance(W, torch.Tensor) and W.is_cuda and W.dtype == torch.uint8 and W.is_contiguous()):
        raise TypeError("W must be a contiguous uint8 CUDA tensor")
    bb = block_bytes(ggml_type)
    if bb > 0 and W.numel() < N * (K // 256) * bb:
        raise ValueError("W holds fewer bytes than N*K/256 superblocks")


def qlinear_argmax(W, ggml_type: int, N: int, K: int, x, stream=None):
    """Greedy output head for M <= 8 tokens: (index int64 [M], value float32 [M]) of the first
    largest y[m, :] of x . dequant(W)^T, without materialising y."""
    import torch
    M = x.shape[0] if x.dim() == 2 else 1
    _mk(x, torch.float16, (M, K), "x")
    _weights(W, ggml_type, N, K)
    idx = torch.empty(M, dtype=torch.int64, device=x.device)
    val = torch.empty(M, dtype=torch.float32, device=x.device)
    _check_stream(stream, x)
    with _device_of(W, x):
        _check(lib().qlinear_argmax(int(ggml_type), W.data_ptr(), int(N), int(K), x.data_ptr(), M, idx.data_ptr(),
                                    val.data_ptr(), _stream_handle(stream)), "qlinear_argmax")
    return idx, val


def qlinear_embed(W, ggml_type: int, N: int, K: int, ids, fp16: bool = False, out=None, stream=None):
    """Embedding gather: out[m, :] = dequant(W)[ids[m], :] (ids: int32 CUDA tensor), each weight
    rounded once to fp32 (or fp16)."""
    import torch
    if not (isinstance(ids, torch.Tensor) and ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous()):
        raise TypeError("ids must be a contiguous int32 CUDA tensor")
    M = ids.numel()
    _weights(W, ggml_type, N, K)
    dt = torch.float16 if fp16 else torch.float32
    if out is None:
        out = torch.empty((M, K), dtype=dt, device=ids.device)
    else:
        _mk(out, dt, (M, K), "out")
    _check_stream(stream, ids)
    with _device_of(W, ids, out):
        _check(lib().qlinear_embed(int(ggml_type), W.data_ptr(), int(N), int(K), ids.data_ptr(), M, out.data_ptr(),
                                   1 if fp16 else 0, _stream_handle(stream)), "qlinear_embed")
    return out


def repack(W, ggml_type: int, N: int, K: int, out=None, stream=None):
    """Q6_K weights (uint8 CUDA tensor, 210-byte blocks) rewritten into the aligned layout
    Q6_K_A16 (224-byte blocks); use the result with ggml_type = Q6_K_A16."""
    import torch
    _weights(W, ggml_type, N, K)
    n = N * (K // 256) * 224
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=W.device)
    else:
        _mk(out, torch.uint8, (n,), "out")
    _check_stream(stream, W)
    with _device_of(W, out):
        _check(lib().qlinear_repack(int(ggml_type), W.data_ptr(), int(N), int(K), out.data_ptr(),
                                    _stream_handle(stream)), "qlinear_repack")
    return out


def copy(dst, src, stream=None):
    """dst[:] = src (same number of bytes, both contiguous) by the library's copy kernel, for
    moving a step's inputs in and outputs out around its layer calls. Each tensor is on the one
    CUDA device involved or in page-locked host memory (`pin_memory()`), which the kernel reads
    or writes directly. Asynchronous on the device's current stream (or `stream`). The copy
    kernel lets the next kernel start at once, so it is not for weights a layer call reads right
    after it (the layer kernels fetch W before waiting for the kernels ahead of them)."""
    import torch
    for name, t in (("dst", dst), ("src", src)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or page-locked host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError(f"dst has {nbytes} bytes, src {src.numel() * src.element_size()}")
    cuda = [t for t in (dst, src) if t.is_cuda]
    dev_ctx = _device_of(*cuda) if cuda else torch.cuda.device(torch.cuda.current_device())
    with dev_ctx:
        if stream is not None and cuda:
            _check_stream(stream, cuda[0])
        _check(lib().qlinear_copy(dst.data_ptr(), src.data_ptr(), int(nbytes), _stream_handle(stream)), "qlinear_copy")
    return dst


GEMM_PLAN_FIELDS = ("n_tile", "k", "L", "tail", "S", "xk", "a_col", "a_slots", "recv_off", "bar_off", "grid_x",
                    "grid_y", "cluster", "smem")


def gemm_plan(ggml_type: int, N: int, K: int, M: int, num_sms: int, cluster_capacity=None) -> dict:
    """The prefill GEMM's launch plan for this shape, computed on the host (no device needed):
    num_sms SMs and cluster_capacity[i] resident clusters of i + 2 CTAs (None: no clusters)."""
    caps = None
    if cluster_capacity is not None:
        vals = list(cluster_capacity)[:7] + [0] * (7 - len(list(cluster_capacity)[:7]))
        caps = (ctypes.c_int * 7)(*vals)
    out = (ctypes.c_int64 * 14)()
    _check(lib().qlinear_gemm_plan(int(ggml_type), int(N), int(K), int(M), int(num_sms), caps, out), "qlinear_gemm_plan")
    return dict(zip(GEMM_PLAN_FIELDS, (int(v) for v in out)))


def device_status(stream=None) -> int:
    """Take (read and clear atomically, after the stream's work) the device status recorded since
    the last call, synchronising the stream: 0, or QL_ERR_BOUNDS (a QL_DEBUG bounds check failed),
    QL_ERR_TIMEOUT (a bounded wait ran out), QL_ERR_INDEX (an embedding id out of range) or
    QL_ERR_CUDA. The status is one word per device, shared by all streams."""
    return lib().qlinear_device_status(_stream_handle(stream))
