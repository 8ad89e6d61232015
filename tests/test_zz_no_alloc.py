"""crisp_route_static: routing with no device allocation, for callers that cannot call
cudaMalloc (for example a plug-in inside an engine that owns all device memory, or a
latency-critical loop that cannot afford an allocation's implicit synchronisation).

Its routes and C_struct must match what the allocating path (crisp_select) produces on
the same inputs, on two calls in a row that share the library's static scratch.  This
file is collected last so that a failure here does not hide the other tests' results.
"""
import ctypes

import numpy as np
import pytest

from tests.parity import to_device
from workloads import get
from workloads.planted import generate

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dsp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dynamic_sparse_prefill_gb300 as d
    return d


def _route_static(dsp, dims, q, k, cfg):
    H = dims.batch * dims.hq
    route = torch.full((H,), 255, dtype=torch.uint8, device="cuda")
    cs = torch.full((H,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = dsp.lib().crisp_route_static(ctypes.byref(dims), ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(k.data_ptr()), ctypes.byref(cfg),
                                      ctypes.c_void_p(route.data_ptr()),
                                      ctypes.c_void_p(cs.data_ptr()),
                                      ctypes.c_void_p(status.data_ptr()), stream)
    assert st == 0
    torch.cuda.synchronize()
    return route.cpu().numpy(), cs.cpu().numpy(), int(status.item())


def _route_alloc(dsp, dims, q, k, cfg):
    ctx = dsp.Context(dims)
    ctx.select(dims, q, k, cfg)
    assert ctx.sync_status() == 0
    sel = ctx.selection_get(dims, with_csr=False)
    ctx.close()
    return sel["route_vs"], sel["c_struct"]


def test_route_static_matches_allocating_path_twice(dsp):
    cases = []
    for name in ("tiny_n4k", "llama8b_n32k"):   # 2*32 and 32*256 = 8192 tiles (the limit)
        w = get(name)
        g = generate(w)
        dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
        cfg = dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy)
        q, k = to_device(g["q"]), to_device(g["k"])
        cases.append((dims, q, k, cfg))
    for dims, q, k, cfg in cases + cases:        # two rounds: the scratch is reused
        r_alloc, c_alloc = _route_alloc(dsp, dims, q, k, cfg)
        r_static, c_static, status = _route_static(dsp, dims, q, k, cfg)
        assert status == 0
        assert np.array_equal(r_static, r_alloc)
        np.testing.assert_allclose(c_static, c_alloc, rtol=1e-4, atol=1e-6)


def test_route_static_rejects_sizes_beyond_its_scratch(dsp):
    w = get("tiny_n4k")
    g = generate(w)
    q, k = to_device(g["q"]), to_device(g["k"])
    cfg = dsp.default_cfg()
    out = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cs = torch.zeros(256, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for dims in (dsp.make_dims(1, 64 * 1024, 64, 64),   # 64 heads x 512 tiles > 8192
                 dsp.make_dims(1, 1024, 130, 130)):      # more than 128 heads
        st = dsp.lib().crisp_route_static(ctypes.byref(dims), ctypes.c_void_p(q.data_ptr()),
                                          ctypes.c_void_p(k.data_ptr()), ctypes.byref(cfg),
                                          ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(cs.data_ptr()),
                                          ctypes.c_void_p(status.data_ptr()), None)
        assert st == 2  # CRISP_ERR_UNSUPPORTED, before any work is queued
    # parameters crisp_select refuses are refused here too (CRISP_ERR_INVALID_ARG)
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    for bad in (dsp.default_cfg(gamma=0.0), dsp.default_cfg(gamma=1.5),
                dsp.default_cfg(flags=dsp.FLAG_MEDIAN_FLOOR | dsp.FLAG_VS_GAMMA_CUMSUM)):
        st = dsp.lib().crisp_route_static(ctypes.byref(dims), ctypes.c_void_p(q.data_ptr()),
                                          ctypes.c_void_p(k.data_ptr()), ctypes.byref(bad),
                                          ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(cs.data_ptr()),
                                          ctypes.c_void_p(status.data_ptr()), None)
        assert st == 1
