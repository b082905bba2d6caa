"""GPU tests of the library's checking and failure machinery, none of which faults the GPU:

* the QL_DEBUG build (every kernel checks the shared- and global-memory ranges its pipelines
  touch and records a failed check as QL_ERR_BOUNDS) runs one small case of each kernel path and
  must stay silent and match the oracle;
* QL_TEST_FAIL=launch makes every call return QL_ERR_CUDA with the launch error recorded, and
  nothing is launched;
* a pointer that is not device memory of the current device is refused with QL_ERR_DEVICE;
* qlinear_repack followed at once by layer calls on the same stream (the layer kernels read W
  before their dependency wait, so the repack must fence the stream) gives the oracle's result.

The debug build and the launch hook are selected per process (environment read at load / first
use), so those cases run in a child interpreter."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_weight_only_gb300 import build
    build.build()
    import gguf_weight_only_gb300 as q
    q.lib()
    return q


def child(code: str, **env) -> dict:
    """Run `code` in a fresh interpreter at the repo root with extra environment; it prints one
    JSON object last."""
    e = dict(os.environ, **env)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=e, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


# one small case per kernel path: (entry, type, N, K, M)
DEBUG_CASES = [
    ("qlinear", 12, 300, 5120, 1),     # decode, 2-D tensor copies
    ("qlinear", 13, 129, 2560, 1),     # decode, Q5_K
    ("qlinear", 23, 300, 5120, 1),     # decode, tokens-on-n path (IQ4_XS)
    ("qlinear", 14, 129, 2560, 3),     # decode, per-row bulk copies (Q6_K)
    ("qlinear", 12, 64, 4096, 8),      # eight tokens
    ("qlinear", 12, 8000, 4096, 1),    # persistent decode kernel, single-token K-quant path
    ("qlinear", 23, 9728, 8192, 1),    # persistent decode kernel, single-token IQ4_XS path (codebook table)
    ("multi", 12, 64, 1024, 2),        # persistent decode kernel (projection set)
    ("silu", 12, 96, 1024, 1),         # persistent decode kernel, fused prologue
    ("qlinear", 12, 256, 2048, 100),   # tcgen05 prefill GEMM
    ("qlinear", 14, 200, 768, 64),     # prefill GEMM, per-row bulk copies
    ("qlinear", 12, 640, 4096, 32),    # prefill GEMM, superblocks split over a cluster
    ("qlinear", 14, 300, 5120, 9),     # split GEMM, per-row bulk copies
    ("qlinear", 12, 10240, 2048, 16),  # split GEMM, two heads per tail
]

DEBUG_CHILD = r'''
import json, numpy as np, torch
import oracle
from oracle import fused
from gguf_weight_only_gb300 import synth
import gguf_weight_only_gb300 as ql
assert ql.DEBUG and ql.LIB_PATH.endswith("_lib_debug/libqlinear.so")
out = {}
for entry, t, N, K, M in CASES:
    W = synth.weights(t, N, K, [970, t, N, K])
    x = synth.activations(M, K, [971, t, M, K])
    Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
    if entry == "qlinear":
        y = ql.qlinear(Wd, t, N, K, xd)
        ref, tol = oracle.qlinear(t, W, N, K, x), oracle.tolerance(t, W, N, K, x)
    elif entry == "multi":
        W2 = synth.weights(t, N // 2, K, [972, t, N, K])
        ys = ql.qlinear_multi([Wd, torch.from_numpy(W2).cuda()], t, [N, N // 2], K, xd)
        y = torch.cat([ys[0], ys[1]], dim=1)
        Wc = np.concatenate([W, W2])
        ref, tol = oracle.qlinear(t, Wc, N + N // 2, K, x), oracle.tolerance(t, Wc, N + N // 2, K, x)
    else:
        up = synth.activations(M, K, [973, t, M, K]).astype(np.float32)
        y = ql.qlinear_silu_mul(Wd, t, N, K, xd, torch.from_numpy(up).cuda())
        xs = fused.silu_mul_x(x, up)
        ref, tol = fused.qlinear_fused(t, W, N, K, xs), fused.tolerance_fused(t, W, N, K, xs)
    torch.cuda.synchronize()
    st = ql.device_status()
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    out[f"{entry}/{t}/{N}/{K}/{M}"] = [int(st), bool(np.all(err <= tol)), bool(np.all(np.isfinite(err)))]
print(json.dumps(out))
'''


def test_debug_build_is_silent_and_correct(ql):
    from gguf_weight_only_gb300 import build
    build.build(debug=True)
    res = child(f"CASES = {DEBUG_CASES!r}\n" + DEBUG_CHILD, QL_DEBUG="1")
    assert len(res) == len(DEBUG_CASES)
    for key, (status, within, finite) in res.items():
        assert status == 0, f"{key}: device status {status} (QL_ERR_BOUNDS = -10)"
        assert finite and within, key


LAUNCH_CHILD = r'''
import json, numpy as np, torch
import gguf_weight_only_gb300 as ql
from gguf_weight_only_gb300 import synth
W = torch.from_numpy(synth.weights(12, 16, 256, [980])).cuda()
x = torch.from_numpy(synth.activations(1, 256, [981])).cuda()
y = torch.full((1, 16), 7.0, device="cuda")
torch.cuda.synchronize()
res = {}
for M, path in ((1, "auto"), (1, "gemv"), (1, "gemm")):
    try:
        ql.qlinear(W, 12, 16, 256, x, out=y, path=path)
        res[path] = None
    except ql.QLinearError as e:
        res[path] = [e.status, ql.lib().qlinear_last_cuda_error()]
torch.cuda.synchronize()
res["untouched"] = bool(torch.all(y == 7.0).item())
res["status"] = ql.device_status()
print(json.dumps(res))
'''


def test_launch_failure_hook_returns_the_cuda_error_and_launches_nothing(ql):
    res = child(LAUNCH_CHILD, QL_TEST_FAIL="launch")
    for path in ("auto", "gemv", "gemm"):
        assert res[path] == [-5, 701], (path, res[path])   # QL_ERR_CUDA, cudaErrorLaunchOutOfResources
    assert res["untouched"] and res["status"] == 0


def test_host_memory_is_refused_before_any_launch(ql):
    N, K = 16, 256
    W = torch.from_numpy(synth.weights(12, N, K, [990])).cuda()
    x = torch.from_numpy(synth.activations(1, K, [991])).cuda()
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    host = torch.zeros(N * K, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    f = ql.lib().qlinear
    assert f(12, host.data_ptr(), N, K, x.data_ptr(), 1, y.data_ptr(), stream) == -8      # QL_ERR_DEVICE
    plain = np.zeros(64, dtype=np.float32)
    assert f(12, W.data_ptr(), N, K, x.data_ptr(), 1, plain.ctypes.data, stream) == -8
    assert f(12, W.data_ptr(), N, K, x.data_ptr(), 1, y.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert ql.device_status() == 0


@pytest.mark.parametrize("M", [1, 64])
def test_repack_then_layer_on_the_same_stream(ql, M):
    N, K = 1024, 4096
    W = synth.weights(14, N, K, [995, M])
    x = synth.activations(M, K, [996, M])
    Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
    out = torch.empty(N * (K // 256) * 224, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):   # the layer call is enqueued right behind the repack each time
        out.fill_(0xFF)
        ql.repack(Wd, 14, N, K, out=out)
        y = ql.qlinear(out, 270, N, K, xd)
        torch.cuda.synchronize()
        assert ql.device_status() == 0
        err = np.abs(y.cpu().numpy().astype(np.float64) - oracle.qlinear(14, W, N, K, x))
        assert np.all(err <= oracle.tolerance(14, W, N, K, x))
