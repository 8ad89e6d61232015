"""ctypes binding of libcrisp.so (include/crisp.h).

Argument marshalling only: tensors are passed as raw device pointers
(``tensor.data_ptr()``) with the current torch CUDA stream; every step of the CRISP
path runs in the library's CUDA kernels.  There is no fallback: if the library is not
built, importing the binding raises.
"""
import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcrisp.so")

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "NO_MEMORY", 4: "CUDA",
                5: "TIMEOUT", 6: "DEVICE_ASSERT", 7: "NO_SELECTION"}
FLAG_FORCE_VS = 0x1
FLAG_FORCE_PE = 0x2
FLAG_MEDIAN_FLOOR = 0x4
FLAG_VS_GAMMA_CUMSUM = 0x8
FLAG_GRAPH_REPLAY = 0x10
DEBUG_DROP_ARRIVE = 0x1

# Every entry point include/crisp.h declares.
EXPORTED = ["crisp_cfg_default", "crisp_create", "crisp_destroy", "crisp_select", "crisp_attend",
            "crisp_prefill", "crisp_dense", "crisp_selection_get", "crisp_selection_set",
            "crisp_selection_stats", "crisp_sync_status", "crisp_set_debug",
            "crisp_status_string", "crisp_last_error", "crisp_route_static", "crisp_jsd",
            "crisp_attend_info", "crisp_prefill_host", "crisp_prefill_launches"]


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n", ctypes.c_int32), ("hq", ctypes.c_int32),
                ("hkv", ctypes.c_int32), ("d", ctypes.c_int32)]


class Cfg(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("b", ctypes.c_int32), ("w_sink", ctypes.c_int32),
                ("w_local", ctypes.c_int32), ("k_min_tokens", ctypes.c_int32),
                ("tau_proxy", ctypes.c_float), ("alpha", ctypes.c_float),
                ("gamma", ctypes.c_float), ("flags", ctypes.c_uint32)]


class SelectionHost(ctypes.Structure):
    _fields_ = [("route_vs", ctypes.c_void_p), ("c_struct", ctypes.c_void_p),
                ("mu", ctypes.c_void_p), ("counts", ctypes.c_void_p), ("p_v", ctypes.c_void_p),
                ("p_s", ctypes.c_void_p), ("sel_v", ctypes.c_void_p), ("sel_s", ctypes.c_void_p),
                ("row_ptr", ctypes.c_void_p), ("col", ctypes.c_void_p),
                ("col_capacity", ctypes.c_int64), ("nnz", ctypes.c_int64)]


class Stats(ctypes.Structure):
    _fields_ = [("nnz", ctypes.c_int64), ("rows", ctypes.c_int64), ("max_row", ctypes.c_int64),
                ("pe_rescued", ctypes.c_int64), ("n_vs", ctypes.c_int32),
                ("n_pe", ctypes.c_int32), ("near_routes", ctypes.c_int32),
                ("near_vs_blocks", ctypes.c_int64), ("near_pe_pairs", ctypes.c_int64)]


class CrispError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: crisp status {STATUS_NAMES.get(status, status)}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"CUDA library {path} is not built (run __graft_entry__.build() or "
                          f"python -m dynamic_sparse_prefill_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    DP, CP = ctypes.POINTER(Dims), ctypes.POINTER(Cfg)
    sig = {
        "crisp_cfg_default": (Cfg, []),
        "crisp_create": (ctypes.c_int, [DP, ctypes.POINTER(P)]),
        "crisp_destroy": (None, [P]),
        "crisp_select": (ctypes.c_int, [P, DP, P, P, CP, P]),
        "crisp_attend": (ctypes.c_int, [P, DP, P, P, P, P, P]),
        "crisp_prefill": (ctypes.c_int, [P, DP, P, P, P, CP, P, P]),
        "crisp_dense": (ctypes.c_int, [P, DP, P, P, P, P, P]),
        "crisp_selection_get": (ctypes.c_int, [P, DP, P, ctypes.POINTER(SelectionHost)]),
        "crisp_selection_set": (ctypes.c_int, [P, DP, P, P, P, ctypes.c_int64]),
        "crisp_selection_stats": (ctypes.c_int, [P, DP, P, ctypes.POINTER(Stats)]),
        "crisp_attend_info": (ctypes.c_int, [P, P, ctypes.POINTER(ctypes.c_int64)]),
        "crisp_prefill_host": (ctypes.c_int, [P, DP, P, P, P, CP, P, P, P, P, P, P]),
        "crisp_sync_status": (ctypes.c_int, [P, P]),
        "crisp_set_debug": (ctypes.c_int, [P, ctypes.c_uint32, ctypes.c_uint64]),
        "crisp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "crisp_last_error": (ctypes.c_char_p, [P]),
        "crisp_route_static": (ctypes.c_int, [DP, P, P, CP, P, P, P, P]),
        "crisp_jsd": (ctypes.c_int, [P, DP, P, P, ctypes.c_float, P, P, P]),
        "crisp_prefill_launches": (ctypes.c_int32, [DP, ctypes.c_int32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def default_cfg(**kw) -> Cfg:
    c = lib().crisp_cfg_default()
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def make_dims(batch, n, hq, hkv, d=128) -> Dims:
    return Dims(batch, n, hq, hkv, d)


def prefill_launches(dims: Dims, num_sms: int) -> int:
    """Kernel launches of one crisp_prefill on a GPU with num_sms SMs (host arithmetic)."""
    return int(lib().crisp_prefill_launches(ctypes.byref(dims), num_sms))


class Context:
    """Owns a crisp_ctx (device workspace for problems up to `max_dims`)."""

    def __init__(self, max_dims: Dims):
        self._lib = lib()
        self._h = ctypes.c_void_p()
        st = self._lib.crisp_create(ctypes.byref(max_dims), ctypes.byref(self._h))
        if st != OK:
            raise CrispError(st, "crisp_create")
        self.max_dims = max_dims

    def close(self):
        if self._h:
            self._lib.crisp_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st, what):
        if st != OK:
            detail = self._lib.crisp_last_error(self._h) or b""
            raise CrispError(st, f"{what} {detail.decode(errors='replace')}")

    def select(self, dims, q, k, cfg, stream=None):
        self._check(self._lib.crisp_select(self._h, ctypes.byref(dims), _ptr(q), _ptr(k),
                                           ctypes.byref(cfg), _stream(stream)), "crisp_select")

    def attend(self, dims, q, k, v, o, stream=None):
        self._check(self._lib.crisp_attend(self._h, ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(o), _stream(stream)), "crisp_attend")

    def prefill(self, dims, q, k, v, cfg, o, stream=None):
        self._check(self._lib.crisp_prefill(self._h, ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                            ctypes.byref(cfg), _ptr(o), _stream(stream)),
                    "crisp_prefill")

    def prefill_host(self, dims, qh, kh, vh, cfg, oh, q, k, v, o, stream=None):
        """crisp_prefill from (page-locked) host tensors qh, kh, vh into oh, staged through
        the device tensors q, k, v, o with the copies overlapping the work."""
        self._check(self._lib.crisp_prefill_host(self._h, ctypes.byref(dims), _ptr(qh), _ptr(kh),
                                                 _ptr(vh), ctypes.byref(cfg), _ptr(oh), _ptr(q),
                                                 _ptr(k), _ptr(v), _ptr(o), _stream(stream)),
                    "crisp_prefill_host")

    def dense(self, dims, q, k, v, o, stream=None):
        self._check(self._lib.crisp_dense(self._h, ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                          _ptr(o), _stream(stream)), "crisp_dense")

    def jsd(self, dims, q, k, tau_jsd, d_js, route_vs, stream=None):
        """FlexPrefill's JSD routing signal for the current selection (device outputs)."""
        self._check(self._lib.crisp_jsd(self._h, ctypes.byref(dims), _ptr(q), _ptr(k),
                                        ctypes.c_float(tau_jsd), _ptr(d_js), _ptr(route_vs),
                                        _stream(stream)), "crisp_jsd")

    def attend_info(self, stream=None) -> int:
        """Query-block rows the last attend/dense recomputed in the rescue pass."""
        rows = ctypes.c_int64(0)
        self._check(self._lib.crisp_attend_info(self._h, _stream(stream), ctypes.byref(rows)),
                    "crisp_attend_info")
        return rows.value

    def sync_status(self, stream=None) -> int:
        return self._lib.crisp_sync_status(self._h, _stream(stream))

    def set_debug(self, flags: int, timeout_ns: int = 0):
        self._check(self._lib.crisp_set_debug(self._h, flags, timeout_ns), "crisp_set_debug")

    def stats(self, dims, stream=None) -> dict:
        s = Stats()
        self._check(self._lib.crisp_selection_stats(self._h, ctypes.byref(dims), _stream(stream),
                                                    ctypes.byref(s)), "crisp_selection_stats")
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def selection_get(self, dims, stream=None, with_csr=True) -> dict:
        H = dims.batch * dims.hq
        nb = dims.n // 128
        out = {
            "route_vs": np.zeros(H, np.uint8), "c_struct": np.zeros(H, np.float32),
            "mu": np.zeros((H, 2), np.float32), "counts": np.zeros((H, 4), np.int32),
            "p_v": np.zeros((H, nb), np.float32), "p_s": np.zeros((H, nb), np.float32),
            "sel_v": np.zeros((H, nb), np.uint8), "sel_s": np.zeros((H, nb), np.uint8),
            "row_ptr": np.zeros(H * nb + 1, np.int64),
        }
        sh = SelectionHost()
        for key in ["route_vs", "c_struct", "mu", "counts", "p_v", "p_s", "sel_v", "sel_s",
                    "row_ptr"]:
            setattr(sh, key, out[key].ctypes.data)
        sh.col = None
        sh.col_capacity = 0
        self._check(self._lib.crisp_selection_get(self._h, ctypes.byref(dims), _stream(stream),
                                                  ctypes.byref(sh)), "crisp_selection_get")
        out["nnz"] = int(sh.nnz)
        if with_csr:
            col = np.zeros(max(int(sh.nnz), 1), np.int32)
            sh.col = col.ctypes.data
            sh.col_capacity = col.size
            self._check(self._lib.crisp_selection_get(self._h, ctypes.byref(dims),
                                                      _stream(stream), ctypes.byref(sh)),
                        "crisp_selection_get")
            out["col"] = col[: int(sh.nnz)]
        return out

    def selection_set(self, dims, row_ptr: np.ndarray, col: np.ndarray, stream=None):
        rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
        cl = np.ascontiguousarray(col, dtype=np.int32)
        self._check(self._lib.crisp_selection_set(self._h, ctypes.byref(dims), _stream(stream),
                                                  ctypes.c_void_p(rp.ctypes.data),
                                                  ctypes.c_void_p(cl.ctypes.data),
                                                  ctypes.c_int64(int(rp[-1]))),
                    "crisp_selection_set")
