"""GPU tests of qlinear_copy: host<->device and device<->device copies by the library's kernel,
exact for every size and alignment (the 16-byte path and the byte tail), refusal of pageable host
memory, and a graph of copy -> layer call -> copy (programmatic dependent launches throughout)
that gives the oracle's result in host memory."""
import numpy as np
import pytest

import oracle
from gguf_weight_only_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gguf_weight_only_gb300 import build
    build.build()
    import gguf_weight_only_gb300 as q
    q.lib()
    return q


@pytest.mark.parametrize("nbytes,offset", [(1, 0), (15, 0), (16, 0), (4096, 0), (49152, 0), (1 << 20, 7), (1000003, 3),
                                            (65536, 1)])
def test_copies_are_exact(ql, nbytes, offset):
    rng = np.random.default_rng([1200, nbytes, offset])
    data = rng.integers(0, 256, nbytes + 32, dtype=np.uint8)
    host_src = torch.from_numpy(data).pin_memory()
    dev = torch.empty(nbytes + 32, dtype=torch.uint8, device="cuda")
    dev2 = torch.zeros(nbytes + 32, dtype=torch.uint8, device="cuda")
    host_dst = torch.zeros(nbytes + 32, dtype=torch.uint8).pin_memory()
    ql.copy(dev[offset:offset + nbytes], host_src[:nbytes])                      # host -> device
    ql.copy(dev2[:nbytes], dev[offset:offset + nbytes])                           # device -> device
    ql.copy(host_dst[offset:offset + nbytes], dev2[:nbytes])                      # device -> host
    torch.cuda.synchronize()
    out = host_dst.numpy()
    assert np.array_equal(out[offset:offset + nbytes], data[:nbytes])
    assert not out[:offset].any() and not out[offset + nbytes:].any()            # nothing outside
    assert ql.device_status() == 0


def test_pageable_host_memory_is_refused(ql):
    plain = np.zeros(64, dtype=np.uint8)
    d = torch.empty(64, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert ql.lib().qlinear_copy(d.data_ptr(), plain.ctypes.data, 64, stream) == -8          # QL_ERR_DEVICE
    assert ql.lib().qlinear_copy(plain.ctypes.data, d.data_ptr(), 64, stream) == -8
    torch.cuda.synchronize()


def test_step_graph_copy_layer_copy(ql):
    """A decode step as an engine runs it: x copied in, the layer, y copied out, all captured
    in one graph and replayed; y in host memory equals the oracle's."""
    t, N, K, M = 12, 4096, 4096, 1
    W = synth.weights(t, N, K, [1210])
    Wd = torch.from_numpy(W).cuda()
    xs = [synth.activations(M, K, [1211, i]) for i in range(3)]
    x_host = torch.from_numpy(xs[0]).pin_memory()
    y_host = torch.zeros(M, N, dtype=torch.float32).pin_memory()
    xd = torch.empty(M, K, dtype=torch.float16, device="cuda")
    yd = torch.empty(M, N, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ql.copy(xd, x_host)
        ql.qlinear(Wd, t, N, K, xd, out=yd)
        ql.copy(y_host, yd)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ql.copy(xd, x_host)
        ql.qlinear(Wd, t, N, K, xd, out=yd)
        ql.copy(y_host, yd)
    for x in xs:
        x_host.copy_(torch.from_numpy(x))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        err = np.abs(y_host.numpy().astype(np.float64) - oracle.qlinear(t, W, N, K, x))
        assert np.all(err <= oracle.tolerance(t, W, N, K, x))
    assert ql.device_status() == 0
