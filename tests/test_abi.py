"""CPU checks of the C ABI: the library loads, exports every function include/crisp.h
declares, and validates arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from dynamic_sparse_prefill_gb300 import _lib
    return _lib


def declared_functions():
    text = open(os.path.join(ROOT, "include", "crisp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(crisp_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    lib = L.lib()
    decl = declared_functions()
    assert decl == sorted(L.EXPORTED)
    for name in decl:
        assert hasattr(lib, name), name


def test_prefill_launch_plan(L):
    """Launches per crisp_prefill on 152 SMs.  Selection: PatSearch and the route (2 for
    N_b <= 256, where the route kernel merges the row statistics itself, else 4), PE block
    means 1, pooled softmax 1, the gamma cut (1 kernel for N_b <= 256, else 12: radix init,
    four histogram and digit passes, tie counts and scan, masks), CSR 2 for at most 32768
    rows (else 3).  Then the work order (1
    kernel for at most 16384 rows, else 3), the attention launches (KV heads per launch:
    >= 8 rows per SM, or as many as fit 48 MB of L2) and the rescue pass."""
    lib = L.lib()
    cases = [((1, 524288, 32, 8), 21 + 3 + 8 + 1),    # one KV head per launch
             ((1, 131072, 32, 8), 20 + 3 + 8 + 1),    # 32768 rows: CSR in 2 launches
             ((1, 131200, 32, 8), 21 + 3 + 8 + 1),    # 32800 rows: CSR in 3
             ((1, 32768, 32, 8), 7 + 1 + 3 + 1),      # N_b = 256: the short-sequence kernels
             ((1, 32896, 32, 8), 20 + 1 + 4 + 1),     # N_b = 257 (2 KV heads per launch)
             ((1, 8192, 32, 8), 7 + 1 + 1 + 1),       # everything in one attention launch
             ((1, 4096, 2, 2), 7 + 1 + 1 + 1),
             ((2, 16384, 32, 8), 7 + 1 + 3 + 1)]     # 16 KV heads, 6 per launch (8 MiB each)
    for (b, n, hq, hkv), want in cases:
        d = L.make_dims(b, n, hq, hkv)
        assert lib.crisp_prefill_launches(ctypes.byref(d), 152) == want, (b, n, hq, hkv)
    assert lib.crisp_prefill_launches(ctypes.byref(L.make_dims(1, 100, 2, 2)), 152) == 0
    assert lib.crisp_prefill_launches(ctypes.byref(L.make_dims(1, 4096, 2, 2)), 0) == 0


def test_default_cfg_is_the_pages_defaults(L):
    c = L.lib().crisp_cfg_default()
    assert (c.B, c.b, c.w_sink, c.w_local, c.k_min_tokens) == (128, 128, 128, 128, 1024)
    assert abs(c.tau_proxy - 0.2) < 1e-7 and c.alpha == 1.0 and abs(c.gamma - 0.95) < 1e-7
    assert c.flags == 0


def test_status_strings(L):
    lib = L.lib()
    for s in range(8):
        assert lib.crisp_status_string(s)
    assert lib.crisp_status_string(5) == b"device wait timed out"


@pytest.mark.parametrize("dims,status", [
    ((1, 4096, 2, 2, 64), 2),     # d != 128
    ((1, 4000, 2, 2, 128), 2),    # n not a multiple of 128
    ((1, 0, 2, 2, 128), 1),
    ((1, 4096, 3, 2, 128), 1),    # hq % hkv != 0
    ((0, 4096, 2, 2, 128), 1),
    ((1, 1 << 21, 2, 2, 128), 2),  # beyond the supported length
])
def test_create_rejects_bad_dims_on_host(L, dims, status):
    lib = L.lib()
    h = ctypes.c_void_p()
    d = L.Dims(*dims)
    assert lib.crisp_create(ctypes.byref(d), ctypes.byref(h)) == status
    assert not h.value


def test_null_arguments(L):
    lib = L.lib()
    assert lib.crisp_create(None, None) == 1
    d = L.Dims(1, 4096, 2, 2, 128)
    assert lib.crisp_select(None, ctypes.byref(d), None, None, None, None) == 1
    assert lib.crisp_sync_status(None, None) == 1
    lib.crisp_destroy(None)
    assert lib.crisp_last_error(None) == b""
